"""Seeded Gaussian-mixture K/V/q generator shaped like the long-context decode
workloads described for RetroInfer ("RetroInfer: A Vector Storage Engine for
Scalable Long-Context LLM Inference", technical summary §4: Llama-3.1 class
models, 120K to 1M tokens of context).

Recipe, per sequence b (own PCG64 stream) and per KV head g, in this draw order:

1. four outlier channels, drawn without replacement from the d channels;
2. planted means mu_p ~ N(0, I_d): ``planted_per_seg`` of them for every
   ``seg_len``-token segment of absolute positions;
3. for every segment in position order: each token picks one of its segment's
   planted means uniformly; key = mean + 0.3 * N(0, I); value ~ N(0, I);
4. keys only: the outlier channels are multiplied by 8, then the first four
   tokens (attention sinks) are scaled to 4x their norm;
5. for each query head of the group: two distinct planted means a, b of this
   KV head, q = (mu_a + mu_b) / 2 + 0.5 * N(0, I) (no outlier scaling, so the
   query is out of distribution relative to the keys, as RetrievalAttention's
   abstract describes).

Everything is then rounded to bf16 (round to nearest even).  Arrays are
returned as raw bf16 bit patterns (uint16) so that every consumer sees the
same bits.  None of the wave-index arithmetic is here.
"""

from __future__ import annotations

import dataclasses
import math
from typing import Dict, List, Optional

import numpy as np

SINK_TOKENS_SCALED = 4
KEY_NOISE_SIGMA = 0.3
QUERY_NOISE_SIGMA = 0.5
OUTLIER_CHANNELS = 4
OUTLIER_FACTOR = 8.0
SINK_NORM_FACTOR = 4.0


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    Hq: int
    Hkv: int
    N: int
    d: int
    sink: int
    window: int
    seg_len: int
    k_per_seg: int
    iters: int
    planted_per_seg: int
    seeds: tuple
    retrieval_frac: Optional[float] = None  # r = ceil(frac * C)
    r_fixed: Optional[int] = None  # explicit r (tiny case)
    description: str = ""

    @property
    def n_seg(self) -> int:
        return -(-self.N // self.seg_len)

    @property
    def n_clusters(self) -> int:
        return self.n_seg * self.k_per_seg

    @property
    def r(self) -> int:
        return retrieval_budget(self)

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


def retrieval_budget(w: Workload, frac: Optional[float] = None) -> int:
    """Clusters retrieved per query head: an explicit r, else ceil(frac * C)."""
    if frac is None:
        if w.r_fixed is not None:
            return w.r_fixed
        frac = w.retrieval_frac
    return int(math.ceil(round(frac * w.n_clusters, 9)))


def _seeds(base, count):
    return tuple(base + i for i in range(count))


WORKLOADS: Dict[str, Workload] = {
    w.name: w
    for w in [
        Workload(
            name="tiny_4k_1h",
            B=1, Hq=1, Hkv=1, N=4096, d=128, sink=4, window=64,
            seg_len=4096, k_per_seg=64, iters=10, planted_per_seg=64,
            seeds=(0,), r_fixed=8,
            description="single head, 4096-token context, 64 clusters, top-8",
        ),
        Workload(
            name="llama3_8b_128k_b1",
            B=1, Hq=32, Hkv=8, N=131072, d=128, sink=4, window=512,
            seg_len=8192, k_per_seg=512, iters=10, planted_per_seg=512,
            seeds=(1,), retrieval_frac=0.018,
            description="Llama-3-8B attention shape (32 q / 8 kv heads, d=128), "
                        "131072-token context, batch 1, 8192 clusters/head, 1.8% budget",
        ),
        Workload(
            name="llama3_8b_128k_b16",
            B=16, Hq=32, Hkv=8, N=131072, d=128, sink=4, window=512,
            seg_len=8192, k_per_seg=512, iters=10, planted_per_seg=512,
            seeds=_seeds(100, 16), retrieval_frac=0.02,
            description="as llama3_8b_128k_b1 at batch 16 (one seed and index per "
                        "sequence); budgets 1/2/3% of tokens",
        ),
        Workload(
            name="llama3_8b_1m_b1",
            B=1, Hq=32, Hkv=8, N=1048576, d=128, sink=4, window=1024,
            seg_len=8192, k_per_seg=512, iters=10, planted_per_seg=512,
            seeds=(2,), retrieval_frac=0.01,
            description="1048576-token context, 65536 clusters/head, 1% budget",
        ),
        Workload(
            name="build_128k_8h",
            B=1, Hq=32, Hkv=8, N=131072, d=128, sink=4, window=512,
            seg_len=8192, k_per_seg=512, iters=10, planted_per_seg=512,
            seeds=(3,), retrieval_frac=0.018,
            description="index build: 131072 tokens x 8 KV heads, 16 segments x 512 "
                        "centroids, 10 iterations",
        ),
    ]
}


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit pattern, round to nearest even (finite inputs)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return u.astype(np.uint16)


def bf16_bits_to_float32(b: np.ndarray) -> np.ndarray:
    b = np.ascontiguousarray(b, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32)


def _gen_sequence(w: Workload, seed: int, N: int, want_q: bool):
    rng = np.random.Generator(np.random.PCG64(seed))
    d = w.d
    L = w.seg_len
    n_seg = -(-N // L)
    group = w.Hq // w.Hkv
    K = np.empty((w.Hkv, N, d), np.uint16)
    V = np.empty((w.Hkv, N, d), np.uint16)
    labels = np.empty((w.Hkv, N), np.int32)
    q = np.empty((w.Hq, d), np.uint16) if want_q else None
    for g in range(w.Hkv):
        outl = rng.choice(d, OUTLIER_CHANNELS, replace=False)
        means = rng.standard_normal((n_seg, w.planted_per_seg, d), dtype=np.float32)
        for s in range(n_seg):
            lo, hi = s * L, min((s + 1) * L, N)
            pick = rng.integers(0, w.planted_per_seg, size=hi - lo)
            keys = means[s][pick] + np.float32(KEY_NOISE_SIGMA) * rng.standard_normal(
                (hi - lo, d), dtype=np.float32)
            vals = rng.standard_normal((hi - lo, d), dtype=np.float32)
            keys[:, outl] *= np.float32(OUTLIER_FACTOR)
            if lo < SINK_TOKENS_SCALED:
                keys[: SINK_TOKENS_SCALED - lo] *= np.float32(SINK_NORM_FACTOR)
            K[g, lo:hi] = bf16_bits(keys)
            V[g, lo:hi] = bf16_bits(vals)
            labels[g, lo:hi] = s * w.planted_per_seg + pick
        if want_q:
            flat = means.reshape(-1, d)
            for j in range(group):
                a, b = rng.choice(flat.shape[0], 2, replace=False)
                qv = (flat[a] + flat[b]) * np.float32(0.5) + np.float32(
                    QUERY_NOISE_SIGMA) * rng.standard_normal(d, dtype=np.float32)
                q[g * group + j] = bf16_bits(qv)
    return K, V, q, labels


def generate(w: Workload, N: Optional[int] = None, batches: Optional[List[int]] = None,
             want_q: bool = True) -> Dict[str, np.ndarray]:
    """Draw the workload's K, V (bf16 bits, [B, Hkv, N, d]), q ([B, Hq, d]) and
    planted labels ([B, Hkv, N]).  ``N`` overrides the context length (same
    recipe, shorter sequence); ``batches`` selects a subset of sequences."""
    N = w.N if N is None else N
    batches = list(range(w.B)) if batches is None else list(batches)
    Ks, Vs, qs, ls = [], [], [], []
    for b in batches:
        K, V, q, lab = _gen_sequence(w, w.seeds[b], N, want_q)
        Ks.append(K)
        Vs.append(V)
        qs.append(q)
        ls.append(lab)
    out = {
        "K": np.stack(Ks),
        "V": np.stack(Vs),
        "labels": np.stack(ls),
    }
    if want_q:
        out["q"] = np.stack(qs)
    return out
