"""GPU parity of the decode options against the CPU oracle: the attention-mass
ranking of the retrieval zone, speculative reuse of the previous step's
retrieval sets with the per-KV-head cosine correction, the GQA-shared
retrieval zone and the bf16 index.

Tolerances as in the plain decode parity: ranking keys within 1e-4 of the
boundary may swap (the mass key adds ln n_c, computed in f32 on the GPU);
outputs max relative error <= 1e-2 per head; lse within 1e-3.  Reuse
decisions compare an f32 cosine with tau, so every case keeps each group's
cosine (oracle, f64) at least 1e-3 away from tau.
"""

import numpy as np
import pytest
import torch

from oracle import wave_index as wi
from tests._util import bf16_bits, bf16_tensor, f64, head_index, rel_err, sets_match_mod_ties
from tests.test_gpu_decode import gpu_index, random_case

pytestmark = pytest.mark.gpu

OUT_TOL = 1e-2
LSE_TOL = 1e-3
KEY_TOL = 1e-4
COS_MARGIN = 1e-3


def lib():
    import cluster_indexed_sparse_wi_b300 as wl
    return wl


def compare(dec, g, oidx, r, rank="score", given=None, qbits=None, share="head"):
    """Check every head of the decoder's last call against the oracle: heads in
    `given` must have attended over exactly that set; the others over the
    oracle's selection by `rank` (up to ties).  Returns the heads whose GPU
    set differs from the oracle's own selection."""
    torch.cuda.synchronize()
    qbits = g["q"] if qbits is None else qbits
    out, lse = dec.out.cpu().numpy(), dec.lse.cpu().numpy()
    topk = dec.topk[..., :r].cpu().numpy()
    Kf, Vf, qf = f64(g["K"]), f64(g["V"]), f64(qbits)
    B, Hq, _ = qf.shape
    group = Hq // Kf.shape[1]
    cfg = dec.index.cfg
    for b in range(B):
        for h in range(Hq):
            gg = h // group
            hi = head_index(oidx, b, gg)
            sel = topk[b, h][topk[b, h] >= 0]
            assert np.all(np.diff(sel) > 0)
            assert np.all(topk[b, h][len(sel):] == -1)
            if given is not None and (b, h) in given:
                want = np.asarray(given[(b, h)])
                assert sel.tolist() == want.tolist(), (b, h)
                ref = wi.decode_head(qf[b, h], Kf[b, gg], Vf[b, gg], hi, cfg.sink, cfg.window, r,
                                     dec.scale, selected=want)
            elif share == "group":
                qg = qf[b, gg * group:(gg + 1) * group]
                want = wi.group_selection(qg, hi["centroid_key"], hi["size"], dec.scale, r, rank)
                keys = sum(wi.ranking_keys(wi.cluster_scores(x, hi["centroid_key"], hi["size"],
                                                             dec.scale), hi["size"], rank)
                           for x in qg)
                assert len(sel) == len(want)
                assert sets_match_mod_ties(sel, want, keys, KEY_TOL * group), (b, h)
                ref = wi.decode_head(qf[b, h], Kf[b, gg], Vf[b, gg], hi, cfg.sink, cfg.window, r,
                                     dec.scale, selected=sel)
            else:
                ref = wi.decode_head(qf[b, h], Kf[b, gg], Vf[b, gg], hi, cfg.sink, cfg.window, r,
                                     dec.scale, rank=rank)
                keys = wi.ranking_keys(ref["scores"], hi["size"], rank)
                assert len(sel) == len(ref["selected"])
                assert sets_match_mod_ties(sel, ref["selected"], keys, KEY_TOL), (b, h)
                if set(sel.tolist()) != set(ref["selected"].tolist()):
                    ref = wi.decode_head(qf[b, h], Kf[b, gg], Vf[b, gg], hi, cfg.sink,
                                         cfg.window, r, dec.scale, selected=sel)
            e = rel_err(out[b, h], ref["out"])
            assert e <= OUT_TOL, (b, h, e)
            assert abs(lse[b, h] - ref["lse"]) <= LSE_TOL, (b, h, lse[b, h], ref["lse"])


# ---------------------------------------------------------------- mass ranking

@pytest.mark.parametrize("G,k,assign_mode", [(1, 32, "random"), (4, 32, "random"),
                                            (2, 33, "random"), (4, 64, "kmeans")])
def test_mass_ranking_parity(G, k, assign_mode):
    # skewed cluster sizes (random mode) make the mass order differ from the
    # score order; k = 33 gives rows that are not 16-byte aligned
    Hkv = 2
    g, oidx = random_case(50 + G + k, B=2, Hq=Hkv * G, Hkv=Hkv, N=6000, sink=4, window=100,
                          seg_len=1024, k=k, assign_mode=assign_mode)
    ix = gpu_index(g, oidx, 4, 100, 1024, k)
    wl = lib()
    K, V, q = (bf16_tensor(g[n], "cuda") for n in ("K", "V", "q"))
    r = 12
    dec = wl.Decoder(ix, Hkv * G, r, rank="mass")
    dec(q, K, V)
    assert dec.status() == 0
    compare(dec, g, oidx, r, rank="mass")
    if assign_mode == "random":
        plain = wl.Decoder(ix, Hkv * G, r)
        plain(q, K, V)
        torch.cuda.synchronize()
        assert not torch.equal(plain.topk, dec.topk)  # the two rankings differ somewhere


def test_mass_ranking_many_clusters():
    # C = 40448 > 8192: keys beyond the first 8192 are recomputed from the
    # scores and sizes at every pass
    g, oidx = random_case(57, B=1, Hq=2, Hkv=1, N=40000, sink=4, window=64, seg_len=512, k=512,
                          assign_mode="random")
    ix = gpu_index(g, oidx, 4, 64, 512, 512)
    wl = lib()
    K, V, q = (bf16_tensor(g[n], "cuda") for n in ("K", "V", "q"))
    r = 700
    dec = wl.Decoder(ix, 2, r, rank="mass")
    dec(q, K, V)
    assert dec.status() == 0
    compare(dec, g, oidx, r, rank="mass")


# ---------------------------------------------------------------- speculative reuse

def _perturbed(qbits, eps_per_group, group, seed):
    """Previous queries: q + eps_g * noise per KV group g, cast to bf16."""
    rng = np.random.default_rng(seed)
    qf = f64(qbits)
    B, Hq, d = qf.shape
    eps = np.repeat(np.asarray(eps_per_group, np.float64), group)[None, :, None]
    prev = qf + eps * rng.standard_normal((B, Hq, d))
    return bf16_bits(torch.from_numpy(prev.astype(np.float32)).to(torch.bfloat16))


def _oracle_reuse(qbits, prevbits, group, tau):
    q, p = f64(qbits), f64(prevbits)
    flags = np.stack([wi.reuse_groups(q[b], p[b], group, tau) for b in range(q.shape[0])])
    # every group's cosine must sit clear of tau
    for b in range(q.shape[0]):
        for t in (tau - COS_MARGIN, tau + COS_MARGIN):
            assert np.array_equal(wi.reuse_groups(q[b], p[b], group, t), flags[b])
    return flags


def test_reuse_decisions_and_parity():
    Hkv, G = 4, 4
    g, oidx = random_case(60, B=2, Hq=Hkv * G, Hkv=Hkv, N=7000, sink=4, window=128,
                          seg_len=2048, k=64)
    ix = gpu_index(g, oidx, 4, 128, 2048, 64)
    wl = lib()
    K, V = (bf16_tensor(g[n], "cuda") for n in ("K", "V"))
    r = 9
    # step t-1 with the previous queries: groups 0 and 2 barely moved, 1 and 3 did
    prev_bits = _perturbed(g["q"], [0.02, 2.0, 0.05, 3.0], G, seed=61)
    prev_q = bf16_tensor(prev_bits, "cuda")
    dec = wl.Decoder(ix, Hkv * G, r)
    dec(prev_q, K, V)
    compare(dec, g, oidx, r, qbits=prev_bits)
    prev_topk = dec.topk[..., :r].clone()
    tau = 0.9
    flags = _oracle_reuse(g["q"], prev_bits, G, tau)
    assert flags.any() and not flags.all()
    q = bf16_tensor(g["q"], "cuda")
    dec(q, K, V, prev_q=prev_q, prev_topk=prev_topk, tau=tau)
    assert dec.status() == 0
    reused = dec.reused.cpu().numpy()
    assert np.array_equal(reused, np.repeat(flags, G, axis=1).astype(np.int32))
    pk = prev_topk.cpu().numpy()
    given = {(b, h): pk[b, h][pk[b, h] >= 0] for b in range(2) for h in range(Hkv * G)
             if flags[b, h // G]}
    compare(dec, g, oidx, r, given=given)
    # the same call with topk_ids aliasing prev_topk (in place) gives the same result
    ref_out, ref_topk = dec.out.clone(), dec.topk.clone()
    dec.topk[..., :r].copy_(prev_topk)
    dec(q, K, V, prev_q=prev_q, prev_topk=dec.topk[..., :r], tau=tau)
    torch.cuda.synchronize()
    assert torch.equal(dec.topk, ref_topk)
    assert torch.equal(dec.out, ref_out)
    assert dec.status() == 0


def test_reuse_threshold_extremes_and_given_sets():
    Hkv, G = 2, 4
    g, oidx = random_case(62, B=1, Hq=Hkv * G, Hkv=Hkv, N=6000, sink=4, window=64,
                          seg_len=1024, k=32, assign_mode="random")
    ix = gpu_index(g, oidx, 4, 64, 1024, 32)
    wl = lib()
    K, V, q = (bf16_tensor(g[n], "cuda") for n in ("K", "V", "q"))
    r = 10
    C = oidx["n_clusters"]
    rng = np.random.default_rng(63)
    # arbitrary valid previous sets: ascending ids (empty clusters allowed),
    # some rows shorter than r, -1 padding
    prev = np.full((1, Hkv * G, r), -1, np.int32)
    given = {}
    for h in range(Hkv * G):
        n = int(rng.integers(0, r + 1))
        ids = np.sort(rng.choice(C, n, replace=False)).astype(np.int32)
        prev[0, h, :n] = ids
        given[(0, h)] = ids
    prev_topk = torch.from_numpy(prev).cuda()
    prev_q = bf16_tensor(_perturbed(g["q"], [0.5, 0.5], G, seed=64), "cuda")
    plain = wl.Decoder(ix, Hkv * G, r)
    plain(q, K, V)
    dec = wl.Decoder(ix, Hkv * G, r)
    # tau > 1: no cosine reaches it; the result is the plain decode, bit for bit
    dec(q, K, V, prev_q=prev_q, prev_topk=prev_topk, tau=1.5)
    torch.cuda.synchronize()
    assert dec.status() == 0
    assert int(dec.reused.sum()) == 0
    assert torch.equal(dec.out, plain.out) and torch.equal(dec.topk, plain.topk)
    # tau = -2: every head takes its given set
    dec(q, K, V, prev_q=prev_q, prev_topk=prev_topk, tau=-2.0)
    assert dec.status() == 0
    assert int(dec.reused.sum()) == Hkv * G
    compare(dec, g, oidx, r, given=given)


def test_reuse_invalid_rows_select_afresh():
    Hkv, G = 1, 4
    g, oidx = random_case(65, B=1, Hq=Hkv * G, Hkv=Hkv, N=6000, sink=4, window=64,
                          seg_len=1024, k=32, assign_mode="random")
    ix = gpu_index(g, oidx, 4, 64, 1024, 32)
    wl = lib()
    K, V, q = (bf16_tensor(g[n], "cuda") for n in ("K", "V", "q"))
    r = 6
    C = oidx["n_clusters"]
    rows = np.array([[1, 5, 9, -1, -1, -1],      # valid
                     [5, 1, 9, -1, -1, -1],      # not ascending
                     [3, 3, 7, -1, -1, -1],      # repeated id
                     [2, C, -1, -1, -1, -1]],    # out of range
                    dtype=np.int32)[None]
    dec = wl.Decoder(ix, Hkv * G, r)
    dec(q, K, V, prev_q=q, prev_topk=torch.from_numpy(rows).cuda(), tau=0.5)
    assert dec.status() == wl._lib.WI_ERR_INVALID_ARG
    assert dec.reused.cpu().numpy().tolist() == [[1, 0, 0, 0]]
    compare(dec, g, oidx, r, given={(0, 0): np.array([1, 5, 9])})


def test_reuse_gap_rows_and_r_zero():
    # a -1 before a valid id is not a retrieval set either; with r = 0 the
    # options change nothing
    g, oidx = random_case(66, B=1, Hq=2, Hkv=1, N=5000, sink=4, window=64, seg_len=1024, k=32,
                          assign_mode="random")
    ix = gpu_index(g, oidx, 4, 64, 1024, 32)
    wl = lib()
    K, V, q = (bf16_tensor(g[n], "cuda") for n in ("K", "V", "q"))
    dec = wl.Decoder(ix, 2, 4)
    rows = torch.tensor([[[-1, 3, -1, -1], [0, 1, 2, 3]]], dtype=torch.int32, device="cuda")
    dec(q, K, V, prev_q=q, prev_topk=rows, tau=0.0)
    assert dec.status() == wl._lib.WI_ERR_INVALID_ARG
    assert dec.reused.cpu().numpy().tolist() == [[0, 1]]
    compare(dec, g, oidx, 4, given={(0, 1): np.array([0, 1, 2, 3])})
    d0 = wl.Decoder(ix, 2, 0)
    plain = wl.Decoder(ix, 2, 0)
    plain(q, K, V)
    d0(q, K, V, prev_q=q, prev_topk=torch.zeros((1, 2, 0), dtype=torch.int32, device="cuda"),
       tau=0.0)
    torch.cuda.synchronize()
    assert d0.status() == 0 and torch.equal(d0.out, plain.out)


# ---------------------------------------------------------------- GQA-shared selection

@pytest.mark.parametrize("G,rank", [(1, "score"), (2, "score"), (4, "score"), (8, "score"),
                                    (4, "mass")])
def test_shared_selection_parity(G, rank):
    Hkv = 2
    g, oidx = random_case(70 + G, B=2, Hq=Hkv * G, Hkv=Hkv, N=6000, sink=4, window=100,
                          seg_len=1024, k=32, assign_mode="random")
    ix = gpu_index(g, oidx, 4, 100, 1024, 32)
    wl = lib()
    K, V, q = (bf16_tensor(g[n], "cuda") for n in ("K", "V", "q"))
    r = 11
    dec = wl.Decoder(ix, Hkv * G, r, rank=rank, share="group")
    dec(q, K, V)
    assert dec.status() == 0
    compare(dec, g, oidx, r, rank=rank, share="group")
    topk = dec.topk.cpu().numpy()
    for b in range(2):
        for gg in range(Hkv):
            rows = topk[b, gg * G:(gg + 1) * G]
            assert (rows == rows[0]).all()
    # each head's scores and maximum are its own
    sc = dec.scores().cpu().numpy()
    hm = dec.head_max().cpu().numpy()
    fin = np.isfinite(sc)
    np.testing.assert_array_equal(hm, np.where(fin.any(-1), np.where(fin, sc, -np.inf).max(-1),
                                               -np.inf))
    if G > 1:
        per = wl.Decoder(ix, Hkv * G, r, rank=rank)
        per(q, K, V)
        torch.cuda.synchronize()
        assert not torch.equal(per.topk, dec.topk)


def test_shared_selection_with_reuse_and_many_clusters():
    # C = 40448: the group row spans several chunks; then every group reuses
    # the sets of its first head's previous row
    Hkv, G = 1, 4
    g, oidx = random_case(75, B=1, Hq=Hkv * G, Hkv=Hkv, N=40000, sink=4, window=64,
                          seg_len=512, k=512, assign_mode="random")
    ix = gpu_index(g, oidx, 4, 64, 512, 512)
    wl = lib()
    K, V, q = (bf16_tensor(g[n], "cuda") for n in ("K", "V", "q"))
    r = 300
    dec = wl.Decoder(ix, G, r, share="group")
    dec(q, K, V)
    assert dec.status() == 0
    compare(dec, g, oidx, r, share="group")
    prev = dec.topk[..., :r].clone()
    prev[0, 1:] = -1  # only the first head's row is read
    dec(q, K, V, prev_q=q, prev_topk=prev, tau=0.5)
    assert dec.status() == 0
    assert dec.reused.cpu().numpy().tolist() == [[1] * G]
    ids = prev[0, 0].cpu().numpy()
    ids = ids[ids >= 0]
    compare(dec, g, oidx, r, given={(0, h): ids for h in range(G)})


# ---------------------------------------------------------------- bf16 index

@pytest.mark.parametrize("G,k,share", [(1, 32, "head"), (4, 33, "head"), (8, 64, "head"),
                                       (4, 32, "group")])
def test_bf16_index_parity(G, k, share):
    # k = 33: 3 tiles per group, the last ragged, so stages carry a pair and a
    # single tile; the oracle decodes against its own bf16 rounding of the
    # float32 index the GPU holds
    Hkv = 2
    g, oidx = random_case(80 + G + k, B=2, Hq=Hkv * G, Hkv=Hkv, N=7000, sink=4, window=100,
                          seg_len=1024, k=k, assign_mode="random")
    ix = gpu_index(g, oidx, 4, 100, 1024, k)
    wl = lib()
    K, V, q = (bf16_tensor(g[n], "cuda") for n in ("K", "V", "q"))
    r = 10
    dec = wl.Decoder(ix, Hkv * G, r, share=share, index_dtype="bf16")
    ck, vs = dec.index16
    assert torch.equal(ck, ix.centroid_key.to(torch.bfloat16))
    assert torch.equal(vs, ix.value_sum.to(torch.bfloat16))
    dec(q, K, V)
    assert dec.status() == 0
    o16 = dict(oidx)
    for key in ("centroid_key", "value_sum"):
        o16[key] = ix.tensors[key].double().cpu().numpy()
    compare(dec, g, wi.round_index_bf16(o16), r, share=share)
