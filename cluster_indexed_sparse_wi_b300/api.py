"""PyTorch-facing binding of libwi: allocates device tensors with torch and
passes their pointers to the C ABI.  Every step of the index build and of the
decode runs in libwi's CUDA kernels; this module only marshals arguments.

Method: "RetroInfer: A Vector Storage Engine for Scalable Long-Context LLM
Inference" -- wave index (technical summary §2.A), segmented clustering (§3).
"""

from __future__ import annotations

import ctypes
import dataclasses
import math
from typing import Dict, Optional, Tuple

import torch

from . import _lib as L


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _need(t: torch.Tensor, name: str, dtype, shape, device=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError("%s must be a torch.Tensor" % name)
    if t.dtype != dtype:
        raise TypeError("%s must be %s, got %s" % (name, dtype, t.dtype))
    if tuple(t.shape) != tuple(shape):
        raise ValueError("%s must have shape %s, got %s" % (name, tuple(shape), tuple(t.shape)))
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    if device is not None and t.device != device:
        raise ValueError("%s must live on %s" % (name, device))


@dataclasses.dataclass
class IndexConfig:
    B: int
    Hkv: int
    N: int
    sink: int
    window: int
    seg_len: int
    k_per_seg: int
    iters: int
    d: int = 128

    @property
    def n_seg(self) -> int:
        return -(-self.N // self.seg_len)

    @property
    def n_clusters(self) -> int:
        return self.n_seg * self.k_per_seg

    @property
    def n_idx(self) -> int:
        return self.N - self.sink - self.window

    def params(self) -> L.BuildParams:
        return L.BuildParams(self.B, self.Hkv, self.N, self.d, self.sink, self.window,
                             self.seg_len, self.k_per_seg, self.iters)


_FIELD_DTYPES = {
    "centroid_key": torch.float32, "unit_centroid": torch.bfloat16, "value_sum": torch.float32,
    "size": torch.int32, "offset": torch.int32, "perm": torch.int32, "assign": torch.int32,
    "k_sorted": torch.bfloat16, "v_sorted": torch.bfloat16,
}


def index_sizes(cfg: IndexConfig) -> Dict[str, int]:
    """Bytes of every index array (wi_index_sizes); no device work."""
    out = (ctypes.c_size_t * len(L.FIELDS))()
    L.check(L.lib().wi_index_sizes(ctypes.byref(cfg.params()), out), "wi_index_sizes")
    return {name: int(out[i]) for i, name in enumerate(L.FIELDS)}


def build_workspace_bytes(cfg: IndexConfig) -> int:
    n = L.lib().wi_build_workspace_bytes(ctypes.byref(cfg.params()))
    if n == 0:
        raise L.WIError(L.WI_ERR_INVALID_ARG, "wi_build_workspace_bytes")
    return int(n)


class WaveIndex:
    """The caller-owned device arrays of a wave index and the wi_index struct
    that points at them."""

    def __init__(self, cfg: IndexConfig, device):
        self.cfg = cfg
        dev = torch.device(device)
        if dev.type == "cuda" and dev.index is None:
            dev = torch.device("cuda", torch.cuda.current_device())
        self.device = dev
        B, H, N, C, d, n = cfg.B, cfg.Hkv, cfg.N, cfg.n_clusters, cfg.d, cfg.n_idx
        shapes = {
            "centroid_key": (B, H, C, d), "unit_centroid": (B, H, C, d),
            "value_sum": (B, H, C, d), "size": (B, H, C), "offset": (B, H, C + 1),
            "perm": (B, H, n), "assign": (B, H, N), "k_sorted": (B, H, n, d),
            "v_sorted": (B, H, n, d),
        }
        sizes = index_sizes(cfg)
        self.tensors: Dict[str, torch.Tensor] = {}
        for name in L.FIELDS:
            t = torch.empty(shapes[name], dtype=_FIELD_DTYPES[name], device=self.device)
            assert t.numel() * t.element_size() == sizes[name], name
            self.tensors[name] = t
        self.struct = L.IndexStruct(*[t.data_ptr() for t in (self.tensors[f] for f in L.FIELDS)])
        self.workspace = torch.zeros(build_workspace_bytes(cfg), dtype=torch.uint8,
                                     device=self.device)

    def __getattr__(self, name):
        tensors = self.__dict__.get("tensors")
        if tensors is not None and name in tensors:
            return tensors[name]
        raise AttributeError(name)

    @property
    def n_clusters(self) -> int:
        return self.cfg.n_clusters

    def _kv(self, K, V=None):
        c = self.cfg
        _need(K, "K", torch.bfloat16, (c.B, c.Hkv, c.N, c.d), self.device)
        if V is not None:
            _need(V, "V", torch.bfloat16, (c.B, c.Hkv, c.N, c.d), self.device)

    # individual build steps ---------------------------------------------
    def init(self, K, stream=None):
        self._kv(K)
        L.check(L.lib().wi_build_init(ctypes.byref(self.cfg.params()), _ptr(K),
                                      ctypes.byref(self.struct), _ptr(self.workspace),
                                      self.workspace.numel(), _stream(stream)), "wi_build_init")

    def assign_step(self, K, stream=None):
        self._kv(K)
        L.check(L.lib().wi_kmeans_assign(ctypes.byref(self.cfg.params()), _ptr(K),
                                         ctypes.byref(self.struct), _ptr(self.workspace),
                                         self.workspace.numel(), _stream(stream)),
                "wi_kmeans_assign")

    def update_step(self, K, stream=None):
        self._kv(K)
        L.check(L.lib().wi_kmeans_update(ctypes.byref(self.cfg.params()), _ptr(K),
                                         ctypes.byref(self.struct), _ptr(self.workspace),
                                         self.workspace.numel(), _stream(stream)),
                "wi_kmeans_update")

    def finalize(self, K, V, stream=None):
        self._kv(K, V)
        L.check(L.lib().wi_build_finalize(ctypes.byref(self.cfg.params()), _ptr(K), _ptr(V),
                                          ctypes.byref(self.struct), _ptr(self.workspace),
                                          self.workspace.numel(), _stream(stream)),
                "wi_build_finalize")

    def build(self, K, V, stream=None):
        self._kv(K, V)
        L.check(L.lib().wi_build_index(ctypes.byref(self.cfg.params()), _ptr(K), _ptr(V),
                                       ctypes.byref(self.struct), _ptr(self.workspace),
                                       self.workspace.numel(), _stream(stream)),
                "wi_build_index")
        return self

    def status(self, stream=None) -> int:
        return sync_status(self.workspace, stream)

    def extended(self, K, V, stream=None) -> "WaveIndex":
        """The index of the grown context K, V [B, Hkv, N', d] (N' >= N):
        positions that left the local window join their segment's nearest
        unit centroid, earlier positions keep their clusters
        (wi_index_extend).  Returns a new WaveIndex; this one is unchanged."""
        c = self.cfg
        N1 = K.shape[2]
        cfg = dataclasses.replace(c, N=N1)
        new = WaveIndex(cfg, self.device)
        new._kv(K, V)
        L.check(L.lib().wi_index_extend(ctypes.byref(cfg.params()), _ptr(K), _ptr(V),
                                        ctypes.byref(self.struct), ctypes.byref(new.struct),
                                        _ptr(new.workspace), new.workspace.numel(),
                                        _stream(stream)), "wi_index_extend")
        return new

    def round_bf16(self, stream=None) -> Tuple[torch.Tensor, torch.Tensor]:
        """bf16 copies (round to nearest even) of the mean keys and value
        sums: the leaner index a Decoder with index_dtype="bf16" streams."""
        c = self.cfg
        shape = (c.B, c.Hkv, c.n_clusters, c.d)
        ck = torch.empty(shape, dtype=torch.bfloat16, device=self.device)
        vs = torch.empty(shape, dtype=torch.bfloat16, device=self.device)
        L.check(L.lib().wi_index_round_bf16(ctypes.byref(self.struct), _ptr(ck), _ptr(vs),
                                            _stream(stream)), "wi_index_round_bf16")
        return ck, vs


def build_index(K: torch.Tensor, V: torch.Tensor, sink: int, window: int, seg_len: int,
                k_per_seg: int, iters: int, stream=None) -> WaveIndex:
    """Build the wave index of K, V (bf16 [B, Hkv, N, 128], on the GPU)."""
    B, H, N, d = K.shape
    cfg = IndexConfig(B, H, N, sink, window, seg_len, k_per_seg, iters, d)
    return WaveIndex(cfg, K.device).build(K, V, stream)


def sync_status(workspace: torch.Tensor, stream=None) -> int:
    """Synchronise the stream and read-and-clear the device status word."""
    st = ctypes.c_int(0)
    L.check(L.lib().wi_sync_status(_ptr(workspace), _stream(stream), ctypes.byref(st)),
            "wi_sync_status")
    return st.value


class Decoder:
    """Decode attention against one WaveIndex with fixed (Hq, r, scale); owns
    its workspace and output buffers.

    rank: "score" (the r largest cluster scores) or "mass" (the r largest
    estimated attention masses n_c e^{s_c}).  share: "head" (every query head
    selects its own set) or "group" (one set per KV group, on the group's
    summed ranking keys).  index_dtype: "f32" streams the index's float32
    mean keys and value sums; "bf16" streams bf16 copies of them (made once,
    here, by WaveIndex.round_bf16), half the index bytes.  A call given prev_q and
    prev_topk (the previous step's queries and returned ids; prev_topk may be
    this decoder's own topk buffer) reuses the previous sets of every KV group
    whose queries all keep a cosine >= tau with their previous query."""

    def __init__(self, index: WaveIndex, Hq: int, r: int, scale: Optional[float] = None,
                 rank: str = "score", share: str = "head", index_dtype: str = "f32"):
        c = index.cfg
        if rank not in L.RANKS:
            raise ValueError("rank must be one of %s" % sorted(L.RANKS))
        if share not in L.SHARES:
            raise ValueError("share must be one of %s" % sorted(L.SHARES))
        self.share = share
        if index_dtype not in ("f32", "bf16"):
            raise ValueError("index_dtype must be 'f32' or 'bf16'")
        self.index_dtype = index_dtype
        self.index16 = index.round_bf16() if index_dtype == "bf16" else None
        self.index = index
        self.Hq = Hq
        self.r = r
        self.rank = rank
        self.scale = 1.0 / math.sqrt(c.d) if scale is None else float(scale)
        self.params = L.DecodeParams(c.B, Hq, c.Hkv, c.N, c.d, c.sink, c.window, r, self.scale)
        lay = L.DecodeLayout()
        L.check(L.lib().wi_decode_workspace_layout(ctypes.byref(self.params), c.n_clusters,
                                                   ctypes.byref(lay)), "wi_decode_workspace_layout")
        self.layout = lay
        dev = index.device
        self.workspace = torch.zeros(lay.total, dtype=torch.uint8, device=dev)
        # out and lse share one buffer, so one copy moves both to the host
        n_out = c.B * Hq * c.d
        self.results = torch.empty(n_out + c.B * Hq, dtype=torch.float32, device=dev)
        self.out = self.results[:n_out].view(c.B, Hq, c.d)
        self.lse = self.results[n_out:].view(c.B, Hq)
        self.topk = torch.empty((c.B, Hq, max(r, 1)), dtype=torch.int32, device=dev)
        self.reused = torch.zeros((c.B, Hq), dtype=torch.int32, device=dev)

    def _q(self, q):
        c = self.index.cfg
        _need(q, "q", torch.bfloat16, (c.B, self.Hq, c.d), self.index.device)

    def capture(self, q, K, V, with_topk: bool = False) -> "torch.cuda.CUDAGraph":
        """The fused decode call on device buffers, captured as a CUDA graph."""
        return capture_graph(lambda: self(q, K, V, with_topk=with_topk), self.index.device)

    def __call__(self, q, K, V, stream=None, with_topk: bool = True, prev_q=None,
                 prev_topk=None, tau: float = 1.0):
        """out [B,Hq,128] f32, lse [B,Hq] f32, topk ids [B,Hq,r] i32."""
        self._q(q)
        self.index._kv(K, V)
        topk = self.topk if (with_topk and self.r > 0) else None
        if (self.rank == "score" and self.share == "head" and self.index16 is None
                and prev_q is None):
            L.check(L.lib().wi_decode_attention(
                ctypes.byref(self.params), _ptr(q), _ptr(K), _ptr(V),
                ctypes.byref(self.index.struct), _ptr(self.out), _ptr(self.lse), _ptr(topk),
                _ptr(self.workspace), self.workspace.numel(), _stream(stream)),
                "wi_decode_attention")
        else:
            c = self.index.cfg
            opt = L.DecodeOptions(L.RANKS[self.rank], float(tau), None, None, _ptr(self.reused),
                                  L.SHARES[self.share])
            if self.index16 is not None:
                opt.centroid_key_bf16, opt.value_sum_bf16 = (_ptr(self.index16[0]),
                                                             _ptr(self.index16[1]))
            if prev_q is not None:
                _need(prev_q, "prev_q", torch.bfloat16, (c.B, self.Hq, c.d), self.index.device)
                if prev_topk is None:
                    raise ValueError("prev_topk is required with prev_q")
                _need(prev_topk, "prev_topk", torch.int32, (c.B, self.Hq, self.r),
                      self.index.device)
                opt.prev_q, opt.prev_topk = _ptr(prev_q), _ptr(prev_topk)
            L.check(L.lib().wi_decode_attention_ex(
                ctypes.byref(self.params), ctypes.byref(opt), _ptr(q), _ptr(K), _ptr(V),
                ctypes.byref(self.index.struct), _ptr(self.out), _ptr(self.lse), _ptr(topk),
                _ptr(self.workspace), self.workspace.numel(), _stream(stream)),
                "wi_decode_attention_ex")
        return self.out, self.lse, (self.topk[..., :self.r] if topk is not None else None)

    # stages -------------------------------------------------------------
    def score(self, q, stream=None):
        self._q(q)
        L.check(L.lib().wi_decode_score(ctypes.byref(self.params), _ptr(q),
                                        ctypes.byref(self.index.struct), _ptr(self.workspace),
                                        self.workspace.numel(), _stream(stream)),
                "wi_decode_score")

    def select(self, stream=None, with_topk: bool = False):
        topk = self.topk if (with_topk and self.r > 0) else None
        L.check(L.lib().wi_decode_select(ctypes.byref(self.params), ctypes.byref(self.index.struct),
                                         _ptr(topk), _ptr(self.workspace), self.workspace.numel(),
                                         _stream(stream)), "wi_decode_select")

    def attend(self, q, K, V, stream=None):
        """Exact attention, retrieved-estimate subtraction and merge into
        self.out / self.lse."""
        self._q(q)
        self.index._kv(K, V)
        L.check(L.lib().wi_decode_attend(ctypes.byref(self.params), _ptr(q), _ptr(K), _ptr(V),
                                         ctypes.byref(self.index.struct), _ptr(self.out),
                                         _ptr(self.lse), _ptr(self.workspace),
                                         self.workspace.numel(), _stream(stream)),
                "wi_decode_attend")
        return self.out, self.lse

    # workspace views ------------------------------------------------------
    def _view(self, off: int, count: int, dtype, shape):
        nbytes = count * torch.tensor([], dtype=dtype).element_size()
        return self.workspace[off:off + nbytes].view(dtype).view(shape)

    def scores(self) -> torch.Tensor:
        c = self.index.cfg
        return self._view(self.layout.scores, c.B * self.Hq * c.n_clusters, torch.float32,
                          (c.B, self.Hq, c.n_clusters))

    def head_max(self) -> torch.Tensor:
        c = self.index.cfg
        return self._view(self.layout.head_max, c.B * self.Hq, torch.float32, (c.B, self.Hq))

    def selected(self) -> Tuple[torch.Tensor, torch.Tensor, torch.Tensor]:
        """Retrieved ids (ascending, -1 padding), their first sorted rows and
        their sizes, each [B, Hq, r]."""
        c = self.index.cfg
        rs = max(self.r, 1)
        shape = (c.B, self.Hq, rs)
        n = c.B * self.Hq * rs
        ids = self._view(self.layout.selected, n, torch.int32, shape)
        rows = self._view(self.layout.sel_rows, n, torch.int32, shape)
        cnts = self._view(self.layout.sel_counts, n, torch.int32, shape)
        return ids[..., :self.r], rows[..., :self.r], cnts[..., :self.r]

    def status(self, stream=None) -> int:
        return sync_status(self.workspace, stream)


def capture_graph(fn, device) -> "torch.cuda.CUDAGraph":
    """Run `fn` once on a side stream (first-call set-up), then capture it into
    a CUDA graph; replaying the graph re-issues the same kernel launches with
    one host call."""
    side = torch.cuda.Stream(device=device)
    side.wait_stream(torch.cuda.current_stream(device))
    with torch.cuda.stream(side):
        fn()
    side.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=side):
        fn()
    return g


class DecodeStep:
    """One decode step as a CUDA graph over host buffers: q is copied from
    pinned host memory, the decode kernel runs, and out / lse are copied
    back into pinned host memory.  `step(q_host)` replays the graph and waits
    for the results."""

    def __init__(self, dec: "Decoder", K, V):
        c = dec.index.cfg
        dev = dec.index.device
        self.dec = dec
        self.q_host = torch.zeros((c.B, dec.Hq, c.d), dtype=torch.bfloat16, pin_memory=True)
        self.results_host = torch.empty(dec.results.numel(), dtype=torch.float32, pin_memory=True)
        n_out = dec.out.numel()
        self.out_host = self.results_host[:n_out].view(tuple(dec.out.shape))
        self.lse_host = self.results_host[n_out:].view(tuple(dec.lse.shape))
        self.q_dev = torch.zeros((c.B, dec.Hq, c.d), dtype=torch.bfloat16, device=dev)
        self.h2d_bytes = self.q_host.numel() * 2
        self.d2h_bytes = self.out_host.numel() * 4 + self.lse_host.numel() * 4

        def body():
            self.q_dev.copy_(self.q_host, non_blocking=True)
            dec(self.q_dev, K, V, with_topk=False)
            self.results_host.copy_(dec.results, non_blocking=True)

        self.graph = capture_graph(body, dev)

    def __call__(self, q_host: Optional[torch.Tensor] = None):
        if q_host is not None:
            self.q_host.copy_(q_host)
        self.graph.replay()
        torch.cuda.current_stream().synchronize()
        return self.out_host, self.lse_host


def decode_attention(q, K, V, index: WaveIndex, r: int, scale: Optional[float] = None,
                     stream=None):
    """One tripartite decode step: returns (out, lse, topk_ids)."""
    dec = Decoder(index, q.shape[1], r, scale)
    return dec(q, K, V, stream)
