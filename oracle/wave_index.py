"""Plain fp64 NumPy oracle of the wave index (build + tripartite decode).

TEST INFRASTRUCTURE ONLY (see the package docstring): no product code imports
this module.

Sources.  The method is described only in prose, on these pages:

* "RetroInfer: A Vector Storage Engine for Scalable Long-Context LLM
  Inference", technical summary (es), §2.A "Wave Index": the tripartite
  approximation -- §2.A.1 steady zone (sink tokens + local window, exact),
  §2.A.2 retrieval zone (spherical-k-means clustering index, the clusters most
  similar to the query are attended exactly), §2.A.3 estimation zone (cluster
  centroids estimate the remaining tokens' contribution); §3 "segmented
  clustering" (k-means on short segments of the sequence).
* the same paper's technical summary (ar), §2.a "Wave Index": the estimation
  zone uses cluster centroids and the sum of value vectors (Sigma V); the
  retrieval zone is a cluster-based vector index; §2.b "Execution Buffer":
  retrieved KV laid out contiguously for FlashAttention-class kernels.

No page prints a formula, so each step below is the plainest reading of that
prose (the readings are listed with the function that takes them).  The zone
merge is a log-sum-exp combine of the zones' softmax terms.

Parity pins (tests/test_oracle_pins.py), none of which re-types this code:

* decode with a budget covering every non-empty cluster == full softmax
  attention computed by torch's scaled_dot_product_attention in float64;
* clusters whose members share one key (singletons included) make the
  estimation exact: output == full attention for every budget;
* q = 0 gives the plain mean of all values and lse = ln N (closed form);
* steady + retrieved token weights plus estimated cluster masses sum to 1;
* brute-force Python loops on tiny inputs (attention, argmax assignment,
  stable (cluster, position) sort, init indices);
* the update's unrounded centroid maximises sum of cosines (Cauchy-Schwarz)
  and bf16 rounding matches torch's round-to-nearest-even cast;
* planted, well-separated clusters are recovered exactly by the build.

"Parity unpinned": the approximation error of the estimation zone relative
to full attention.  The pages call the estimate accuracy-bounded but print no
bound, so it is reported, never gated.
"""

from __future__ import annotations

import math
from typing import Dict, List, Optional

import numpy as np

__all__ = [
    "bf16_round",
    "bf16_bits_to_f64",
    "steady_positions",
    "segment_positions",
    "kmeans_init",
    "kmeans_assign",
    "kmeans_update",
    "kmeans_segment",
    "index_statistics",
    "build_index_head",
    "build_index",
    "extend_index_head",
    "cluster_scores",
    "select_clusters",
    "ranking_keys",
    "reuse_groups",
    "round_index_bf16",
    "group_selection",
    "decode_head",
    "decode",
]


# --------------------------------------------------------------------------
# number formats
# --------------------------------------------------------------------------

def bf16_round(x) -> np.ndarray:
    """Round float64 values directly to the nearest bf16 value (8 significand
    bits, ties to even) and return them as float64.  Finite, normal-range
    inputs; bf16 is the tensor-core operand type of the centroids."""
    x = np.asarray(x, dtype=np.float64)
    m, e = np.frexp(x)  # x = m * 2**e, 0.5 <= |m| < 1
    return np.ldexp(np.rint(m * 256.0), e - 8)  # np.rint: half to even


def bf16_bits_to_f64(bits) -> np.ndarray:
    """Exact upcast of bf16 bit patterns (uint16) to float64."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


# --------------------------------------------------------------------------
# zones
# --------------------------------------------------------------------------

def steady_positions(N: int, sink: int, window: int) -> np.ndarray:
    """Steady zone: the first ``sink`` positions and the last ``window``
    positions (RetroInfer summary §2.A.1: sink tokens and the local window,
    always attended exactly).  Requires sink + window <= N, so the two spans
    never overlap."""
    return np.concatenate([np.arange(0, sink), np.arange(N - window, N)]).astype(np.int64)


def segment_positions(N: int, sink: int, window: int, seg_len: int) -> List[np.ndarray]:
    """Indexable positions of each segment.

    Reading (RetroInfer summary §3, segmented clustering): the sequence is cut
    into segments of ``seg_len`` consecutive absolute positions,
    [s*seg_len, (s+1)*seg_len); the steady zone is excluded from the index, so
    segment s holds the positions of that span inside [sink, N - window).
    There are ceil(N / seg_len) segments; a segment may hold fewer tokens than
    seg_len, or none."""
    n_seg = -(-N // seg_len)
    lo_idx, hi_idx = sink, N - window
    out = []
    for s in range(n_seg):
        lo = max(s * seg_len, lo_idx)
        hi = min((s + 1) * seg_len, N, hi_idx)
        out.append(np.arange(lo, max(lo, hi), dtype=np.int64))
    return out


# --------------------------------------------------------------------------
# segmented spherical k-means (one segment)
# --------------------------------------------------------------------------

def _normalize_rows(x: np.ndarray) -> np.ndarray:
    n = np.sqrt(np.sum(x * x, axis=1, keepdims=True))
    return np.divide(x, n, out=np.zeros_like(x), where=n > 0)


def kmeans_init(keys: np.ndarray, k: int) -> np.ndarray:
    """Initial unit centroids of one segment.

    Reading (the pages do not state the initialisation): deterministic strided
    seeding.  With the segment's m keys in position order, centroid j is key
    number floor(j * m / k), scaled to unit length and rounded to bf16.  A
    segment with no keys gets zero centroids (they are never assigned)."""
    m, d = keys.shape
    if m == 0:
        return np.zeros((k, d))
    pick = (np.arange(k, dtype=np.int64) * m) // k
    return bf16_round(_normalize_rows(keys[pick]))


def kmeans_assign(keys: np.ndarray, mu: np.ndarray):
    """Assignment step of spherical k-means: a(i) = argmax_j k_i . mu_j, the
    lowest j among exact maxima (argmax of k_i . mu_j equals argmax of the
    cosine, since ||k_i|| is a positive per-row constant).

    Returns (a, cos) where cos[i, j] = k_i . mu_j / ||k_i|| (0 for a zero key),
    the bounded score that tie tolerances are stated on."""
    dots = keys @ mu.T
    a = np.argmax(dots, axis=1).astype(np.int64)  # first maximum = lowest j
    norms = np.sqrt(np.sum(keys * keys, axis=1))
    cos = np.divide(dots, norms[:, None], out=np.zeros_like(dots), where=norms[:, None] > 0)
    return a, cos


def kmeans_update(keys: np.ndarray, a: np.ndarray, mu_prev: np.ndarray):
    """Update step of spherical k-means (Dhillon-Modha): for every non-empty
    cluster j, mu_j = normalize(sum over members of k_i / ||k_i||), rounded to
    bf16.  An empty cluster, or one whose member directions sum to zero, keeps
    its previous centroid.

    Returns (mu_bf16, mu_exact) -- the second is the unrounded unit vector (or
    the previous centroid where it was kept), exposed for the optimality pin."""
    k, d = mu_prev.shape
    unit = _normalize_rows(keys)
    sums = np.zeros((k, d))
    np.add.at(sums, a, unit)
    counts = np.bincount(a, minlength=k)
    norm = np.sqrt(np.sum(sums * sums, axis=1))
    keep = (counts == 0) | (norm == 0)
    mu_exact = np.where(keep[:, None], mu_prev, sums / np.where(norm > 0, norm, 1.0)[:, None])
    mu = np.where(keep[:, None], mu_prev, bf16_round(mu_exact))
    return mu, mu_exact


def kmeans_segment(keys: np.ndarray, k: int, iters: int, trace: bool = False):
    """``iters`` rounds of (assign, update) from the strided init.  Returns the
    assignment of the last round and the centroids after its update; with
    ``trace`` also every round's (mu_in, a, mu_out)."""
    if iters < 1:
        raise ValueError("iters must be >= 1")
    mu = kmeans_init(keys, k)
    hist = []
    a = np.zeros(keys.shape[0], dtype=np.int64)
    for _ in range(iters):
        if keys.shape[0] == 0:
            break
        a, _ = kmeans_assign(keys, mu)
        mu_new, _ = kmeans_update(keys, a, mu)
        if trace:
            hist.append((mu, a, mu_new))
        mu = mu_new
    return (a, mu, hist) if trace else (a, mu)


# --------------------------------------------------------------------------
# index of one (sequence, KV head)
# --------------------------------------------------------------------------

def index_statistics(K: np.ndarray, V: np.ndarray, pos: np.ndarray, c: np.ndarray,
                     n_clusters: int) -> Dict[str, np.ndarray]:
    """Per-cluster statistics from an assignment (position pos[i] -> cluster
    c[i]):

    * n_c (cluster size) -- the estimation zone's softmax mass needs it, and the
      pages' "centroid and Sigma V" estimate implies it;
    * centroid key k_bar_c = sum k_i / n_c (mean raw key; 0 when empty), stored
      as float32 -- reading: the zone scores and estimates with the mean key,
      since a unit centroid carries no key magnitude;
    * value sum vsum_c = Sigma v_i (technical summary (ar) §2.a), float32;
    * perm: positions sorted stably by (cluster, position), with offsets --
      the cluster-contiguous layout of the execution buffer (§2.b);
    * K_sorted / V_sorted = K[perm], V[perm]."""
    d = K.shape[1]
    order = np.lexsort((pos, c))  # primary key c, then position
    perm = pos[order]
    cs = c[order]
    n = np.bincount(c, minlength=n_clusters).astype(np.int64)
    offset = np.zeros(n_clusters + 1, dtype=np.int64)
    offset[1:] = np.cumsum(n)
    ksum = np.zeros((n_clusters, d))
    vsum = np.zeros((n_clusters, d))
    np.add.at(ksum, cs, K[perm])
    np.add.at(vsum, cs, V[perm])
    kbar = np.divide(ksum, n[:, None], out=np.zeros_like(ksum), where=n[:, None] > 0)
    return {
        "size": n,
        "offset": offset,
        "perm": perm,
        "centroid_key": kbar.astype(np.float32).astype(np.float64),
        "value_sum": vsum.astype(np.float32).astype(np.float64),
        "k_sorted": K[perm],
        "v_sorted": V[perm],
    }


def build_index_head(K: np.ndarray, V: np.ndarray, sink: int, window: int, seg_len: int,
                     k_per_seg: int, iters: int) -> Dict[str, np.ndarray]:
    """Segmented spherical k-means index over one head's keys K [N, d] (fp64
    values of bf16 inputs), with values V [N, d].  Cluster j of segment s has
    the global id s * k_per_seg + j.  ``assign`` maps every position to its
    cluster, -1 for the steady zone."""
    N, d = K.shape
    segs = segment_positions(N, sink, window, seg_len)
    C = len(segs) * k_per_seg
    assign = np.full(N, -1, dtype=np.int64)
    mu = np.zeros((C, d))
    for s, pos in enumerate(segs):
        a, m = kmeans_segment(K[pos], k_per_seg, iters)
        mu[s * k_per_seg:(s + 1) * k_per_seg] = m
        assign[pos] = s * k_per_seg + a
    idx = np.arange(sink, N - window, dtype=np.int64)
    st = index_statistics(K, V, idx, assign[idx], C)
    st["unit_centroid"] = mu
    st["assign"] = assign
    st["n_clusters"] = C
    return st


def extend_index_head(K: np.ndarray, V: np.ndarray, old: Dict[str, np.ndarray], N_old: int,
                      sink: int, window: int, seg_len: int,
                      k_per_seg: int) -> Dict[str, np.ndarray]:
    """Index maintenance during decode (RetroInfer summary §2.A.1: the local
    window slides, so its oldest tokens leave the steady zone).  The context
    grew from N_old to N = K.shape[0] positions; the positions
    [N_old - window, N - window) leave the window and join the index without
    re-clustering.

    Readings (the pages are silent on maintenance):
    * every earlier position keeps its cluster, and the unit centroids are
      kept (clusters of segments that appear only now start empty, with zero
      centroids, as an empty segment's do at build time);
    * a joining position p goes to the nearest unit centroid,
      argmax_j k_p . mu_j with the lowest j among equal maxima, of its own
      segment p // seg_len, which must have held indexable positions before
      (ValueError otherwise: a segment without centroids is opened by
      re-clustering, i.e. a rebuild);
    * sizes, mean keys, value sums and the sorted copies are then those of
      the new assignment (``index_statistics``)."""
    N, d = K.shape
    segs_old = segment_positions(N_old, sink, window, seg_len)
    clustered = [s for s, pos in enumerate(segs_old) if pos.size > 0]
    if not clustered:
        raise ValueError("the earlier index holds no clustered segment")
    last = clustered[-1]
    if N - window > (last + 1) * seg_len:
        raise ValueError("joining positions reach a segment without centroids")
    C = -(-N // seg_len) * k_per_seg
    mu = np.zeros((C, d))
    C_old = old["unit_centroid"].shape[0]
    mu[:C_old] = old["unit_centroid"]
    assign = np.full(N, -1, dtype=np.int64)
    lo, hi_old, hi = sink, N_old - window, N - window
    assign[lo:hi_old] = old["assign"][lo:hi_old]
    for p in range(max(hi_old, lo), hi):
        s = p // seg_len
        a, _ = kmeans_assign(K[p:p + 1], mu[s * k_per_seg:(s + 1) * k_per_seg])
        assign[p] = s * k_per_seg + a[0]
    idx = np.arange(sink, hi, dtype=np.int64)
    st = index_statistics(K, V, idx, assign[idx], C)
    st["unit_centroid"] = mu
    st["assign"] = assign
    st["n_clusters"] = C
    return st


def build_index(K: np.ndarray, V: np.ndarray, sink: int, window: int, seg_len: int,
                k_per_seg: int, iters: int) -> Dict[str, np.ndarray]:
    """Index for K, V [B, Hkv, N, d]: every (sequence, KV head) independently.
    Arrays gain leading [B, Hkv] axes."""
    B, H = K.shape[:2]
    heads = [[build_index_head(K[b, h], V[b, h], sink, window, seg_len, k_per_seg, iters)
              for h in range(H)] for b in range(B)]
    out = {}
    for key in heads[0][0]:
        if key == "n_clusters":
            out[key] = heads[0][0][key]
        else:
            out[key] = np.stack([np.stack([heads[b][h][key] for h in range(H)]) for b in range(B)])
    return out


# --------------------------------------------------------------------------
# decode: tripartite attention for one query head
# --------------------------------------------------------------------------

def cluster_scores(q: np.ndarray, centroid_key: np.ndarray, size: np.ndarray,
                   scale: float) -> np.ndarray:
    """s_c = scale * q . k_bar_c for non-empty clusters, -inf for empty ones
    (RetroInfer summary §2.A.2: the clusters most similar to the query)."""
    s = scale * (centroid_key @ q)
    return np.where(size > 0, s, -np.inf)


def ranking_keys(s: np.ndarray, size: np.ndarray, rank: str = "score") -> np.ndarray:
    """The key clusters are ranked by for the retrieval zone.

    * ``"score"``: s_c, the cluster's logit (RetroInfer summary §2.A.2: the
      clusters most similar to the query);
    * ``"mass"``: the estimated attention mass n_c e^{s_c} of the cluster,
      compared in log space as s_c + ln n_c.  Reading: the "attention-aware"
      index of the technical summary (ar) §2.a ranks by the share of the
      softmax a cluster would take, which is what its estimate weighs; an
      empty cluster has no mass (-inf)."""
    if rank == "score":
        return s
    if rank != "mass":
        raise ValueError(rank)
    n = np.asarray(size, dtype=np.float64)
    with np.errstate(divide="ignore"):
        return np.where((n > 0) & np.isfinite(s), s + np.log(np.where(n > 0, n, 1.0)), -np.inf)


def select_clusters(s: np.ndarray, r: int) -> np.ndarray:
    """Retrieval zone: the r clusters with the largest key s (a score or a
    ranking key), ordered by (key descending, cluster id ascending); clusters
    whose key is -inf (empty) are never taken, so fewer when fewer are
    non-empty.  Returned sorted by id."""
    ids = np.arange(s.shape[0])
    finite = np.isfinite(s)
    order = np.lexsort((ids[finite], -s[finite]))
    return np.sort(ids[finite][order][:r])


def round_index_bf16(index: Dict[str, np.ndarray]) -> Dict[str, np.ndarray]:
    """The leaner index of the GQA-shared variant: centroid keys and value
    sums held as bf16 (round to nearest, ties to even), which halves the
    bytes decode streams from the index.  Reading: the pages fix no storage
    type; the rounding is applied to the float32 index the build stores, so
    the quantisation is decided in the precision the stored values have.
    Sizes, offsets, perm and the sorted copies are unchanged."""
    out = dict(index)
    for key in ("centroid_key", "value_sum"):
        out[key] = bf16_round(np.asarray(index[key], dtype=np.float32).astype(np.float64))
    return out


def group_selection(q_group: np.ndarray, centroid_key: np.ndarray, size: np.ndarray,
                    scale: float, r: int, rank: str = "score") -> np.ndarray:
    """GQA-shared retrieval zone: one set for all query heads of a KV head,
    the r largest summed ranking keys sum_h key_h(c) over the group's queries
    q_group [G, d] (ties to the lower id).  Reading: the pages leave the
    selection granularity open; summing the heads' keys is the plainest group
    score (for scores it is the score of the summed query)."""
    keys = np.zeros(centroid_key.shape[0])
    for qh in q_group:
        keys = keys + ranking_keys(cluster_scores(qh, centroid_key, size, scale), size, rank)
    return select_clusters(keys, r)


def reuse_groups(q: np.ndarray, q_prev: np.ndarray, group: int, tau: float) -> np.ndarray:
    """Speculative reuse with fine-grained correction (FreeKV technical
    summary §2.A.1-2): the retrieval set of the previous decoding step is
    reused while the query has not moved, and re-selected for the KV heads
    whose queries did.  Reading: the similarity of a KV head is the smallest
    cosine cos(q_t, q_{t-1}) over its query heads; it reuses iff that is at
    least tau.

    q, q_prev: [Hq, d] (one sequence).  Returns a bool per KV head."""
    qn = np.linalg.norm(q, axis=1)
    pn = np.linalg.norm(q_prev, axis=1)
    dot = np.sum(q * q_prev, axis=1)
    cos = np.divide(dot, qn * pn, out=np.zeros_like(dot), where=(qn > 0) & (pn > 0))
    return cos.reshape(-1, group).min(axis=1) >= tau


def decode_head(q: np.ndarray, K: np.ndarray, V: np.ndarray, index: Dict[str, np.ndarray],
                sink: int, window: int, r: int, scale: float,
                selected: Optional[np.ndarray] = None,
                rank: str = "score") -> Dict[str, np.ndarray]:
    """Tripartite attention of one query q [d] over one KV head (K, V [N, d]).

    Steps (RetroInfer summary §2.A; technical summary (ar) §2.a):

    1. scores s_c of every cluster against the query;
    2. retrieval zone T = the top-r clusters by the ranking key (the score,
       or the attention mass with ``rank="mass"``), or ``selected`` if given
       (empty clusters in it attend nothing);
    3. exact token set S = steady zone + members of T, logits l_i = scale q.k_i;
    4. estimation zone E = non-empty clusters outside T: each member's logit is
       taken as its cluster's score, so cluster c contributes n_c e^{s_c} to
       the softmax mass and e^{s_c} * vsum_c to the weighted value sum;
    5. log-sum-exp merge: M = max over S logits and E scores,
       L = sum_S e^{l_i - M} + sum_E n_c e^{s_c - M},
       out = (sum_S e^{l_i - M} v_i + sum_E e^{s_c - M} vsum_c) / L,
       lse = M + ln L.

    Returns out, lse, the selected ids, the scores, and the weights
    (w_i for i in S, omega_c for c in E) that sum to 1."""
    N = K.shape[0]
    size = index["size"]
    s = cluster_scores(q, index["centroid_key"], size, scale)
    if selected is None:
        T = select_clusters(ranking_keys(s, size, rank), r)
    else:
        T = np.unique(np.asarray(selected, np.int64))
    members = [index["perm"][index["offset"][c]:index["offset"][c + 1]] for c in T]
    S = np.concatenate([steady_positions(N, sink, window)] + members).astype(np.int64)
    logits = scale * (K[S] @ q)
    inT = np.zeros(s.shape[0], dtype=bool)
    inT[T] = True
    E = np.nonzero((~inT) & (size > 0))[0]
    sE = s[E]
    M = max(logits.max(initial=-np.inf), sE.max(initial=-np.inf))
    if not np.isfinite(M):
        return {"out": np.zeros(K.shape[1]), "lse": -np.inf, "selected": T, "scores": s,
                "token_pos": S, "token_w": np.zeros(len(S)), "est_ids": E,
                "est_w": np.zeros(len(E))}
    eS = np.exp(logits - M)
    eE = np.exp(sE - M)
    L = eS.sum() + (size[E] * eE).sum()
    num = eS @ V[S] + eE @ index["value_sum"][E]
    return {
        "out": num / L,
        "lse": M + math.log(L),
        "selected": T,
        "scores": s,
        "token_pos": S,
        "token_w": eS / L,
        "est_ids": E,
        "est_w": size[E] * eE / L,
    }


def decode(q: np.ndarray, K: np.ndarray, V: np.ndarray, index: Dict[str, np.ndarray],
           sink: int, window: int, r: int, scale: Optional[float] = None,
           heads: Optional[List[tuple]] = None, rank: str = "score",
           prev_q: Optional[np.ndarray] = None, prev_selected: Optional[dict] = None,
           tau: float = 1.0, share: str = "head",
           index_dtype: str = "f32") -> Dict[str, np.ndarray]:
    """Decode attention for q [B, Hq, d] against K, V [B, Hkv, N, d] and a
    per-(b, kv head) index with leading [B, Hkv] axes.  Query head h reads KV
    head h // (Hq / Hkv) (grouped-query attention).  ``heads`` restricts the
    work to a list of (b, h) pairs; the other rows of the result stay NaN.

    ``rank`` picks the ranking key of the retrieval zone (``ranking_keys``).
    With ``prev_q`` [B, Hq, d] and ``prev_selected`` ({(b, h): ids}) the
    previous step's selection is reused by every KV head that
    ``reuse_groups`` keeps at threshold ``tau``; the others select afresh.
    ``reused`` [B, Hkv] reports the decision.

    ``share="group"`` gives every query head of a KV head the group's shared
    set (``group_selection``) instead of its own; ``index_dtype="bf16"``
    decodes against ``round_index_bf16(index)``."""
    if share not in ("head", "group") or index_dtype not in ("f32", "bf16"):
        raise ValueError((share, index_dtype))
    if index_dtype == "bf16":
        index = round_index_bf16(index)
    B, Hq, d = q.shape
    Hkv = K.shape[1]
    group = Hq // Hkv
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    out = np.full((B, Hq, d), np.nan)
    lse = np.full((B, Hq), np.nan)
    sel = {}
    reused = np.zeros((B, Hkv), dtype=bool)
    if prev_q is not None:
        for b in range(B):
            reused[b] = reuse_groups(q[b], prev_q[b], group, tau)
    todo = heads if heads is not None else [(b, h) for b in range(B) for h in range(Hq)]
    for b, h in todo:
        g = h // group
        ih = {key: index[key][b, g] for key in ("size", "centroid_key", "value_sum", "perm",
                                                 "offset")}
        given = prev_selected[(b, h)] if reused[b, g] else None
        if given is None and share == "group":
            given = group_selection(q[b, g * group:(g + 1) * group], ih["centroid_key"],
                                    ih["size"], scale, r, rank)
        res = decode_head(q[b, h], K[b, g], V[b, g], ih, sink, window, r, scale,
                          selected=given, rank=rank)
        out[b, h] = res["out"]
        lse[b, h] = res["lse"]
        sel[(b, h)] = res["selected"]
    return {"out": out, "lse": lse, "selected": sel, "reused": reused}
