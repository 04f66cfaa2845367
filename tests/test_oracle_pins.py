"""Pins of the CPU oracle against facts fixed outside it (closed forms, library
routines, brute force, invariants).  CPU only.

The method follows "RetroInfer: A Vector Storage Engine for Scalable
Long-Context LLM Inference" (technical summaries §2.A / §2.a and §3).
"""

import json
import math
import os

import numpy as np
import pytest
import torch

from oracle import wave_index as wi

HERE = os.path.dirname(os.path.abspath(__file__))


# ---------------------------------------------------------------- helpers

def sdpa64(q, K, V, scale):
    """Softmax attention of one query by torch's library routine, float64."""
    qt = torch.from_numpy(np.asarray(q, np.float64)).view(1, 1, 1, -1)
    Kt = torch.from_numpy(np.asarray(K, np.float64)).view(1, 1, K.shape[0], -1)
    Vt = torch.from_numpy(np.asarray(V, np.float64)).view(1, 1, V.shape[0], -1)
    out = torch.nn.functional.scaled_dot_product_attention(qt, Kt, Vt, scale=scale)
    lse = torch.logsumexp(scale * (Kt[0, 0] @ qt[0, 0, 0]), dim=0)
    return out.view(-1).numpy(), float(lse)


def bf16_vals(rng, shape, scale=1.0):
    x = (rng.standard_normal(shape) * scale).astype(np.float32)
    return torch.from_numpy(x).to(torch.bfloat16).double().numpy()


def vsum_atol(idx):
    """Bound on the output error caused by storing value sums in float32: each
    estimated cluster weighs in with e^{s_c-M}/L <= 1/n_c, and the weights'
    masses sum to at most 1."""
    n = np.maximum(idx["size"], 1)[:, None]
    return 2.0 ** -23 * float(np.max(np.abs(idx["value_sum"]) / n, initial=0.0)) + 1e-13


def small_case(seed=0, N=700, d=128, sink=4, window=32, seg_len=256, k=16, iters=3,
               planted=6):
    rng = np.random.default_rng(seed)
    means = rng.standard_normal((planted, d))
    lab = rng.integers(0, planted, N)
    K = bf16_vals(rng, (N, d), 0.4) + torch.from_numpy(means[lab]).to(torch.bfloat16).double().numpy()
    K = torch.from_numpy(K).to(torch.bfloat16).double().numpy()
    V = bf16_vals(rng, (N, d))
    q = bf16_vals(rng, (d,))
    idx = wi.build_index_head(K, V, sink, window, seg_len, k, iters)
    return K, V, q, idx


# ---------------------------------------------------------------- number format

def test_bf16_round_matches_torch_cast():
    rng = np.random.default_rng(1)
    x = np.concatenate([
        rng.standard_normal(20000).astype(np.float32),
        (rng.standard_normal(2000) * 1e-3).astype(np.float32),
        # exact halfway cases between two bf16 neighbours: low 16 bits = 0x8000
        ((rng.integers(0x3F000000, 0x40800000, 4000, dtype=np.uint32) & 0xFFFF0000) | 0x8000)
        .view(np.float32),
    ])
    ref = torch.from_numpy(x).to(torch.bfloat16).double().numpy()
    np.testing.assert_array_equal(wi.bf16_round(x.astype(np.float64)), ref)


def test_bf16_round_fp64_is_nearest_ties_even():
    rng = np.random.default_rng(2)
    x = rng.standard_normal(20000)
    y = wi.bf16_round(x)
    # neighbours: y is a bf16 value; its distance to x is at most half an ulp
    ulp = 2.0 ** (np.floor(np.log2(np.abs(y))) - 7)
    assert np.all(np.abs(x - y) <= ulp / 2 + 1e-300)
    yb = torch.from_numpy(y.astype(np.float32)).to(torch.bfloat16).double().numpy()
    np.testing.assert_array_equal(y, yb)  # y is representable in bf16


# ---------------------------------------------------------------- worked example

def test_worked_example_hand_derived():
    g = json.load(open(os.path.join(HERE, "golden", "worked_example_2d.json")))
    K = np.array(g["K"], np.float64)
    V = np.array(g["V"], np.float64)
    q = np.array(g["q"], np.float64)
    idx = wi.build_index_head(K, V, g["sink"], g["window"], g["seg_len"], g["k_per_seg"],
                              g["iters"])
    for key, val in g["expect_index"].items():
        np.testing.assert_array_equal(idx[key], np.array(val), err_msg=key)
    for r, e in g["expect_decode"].items():
        res = wi.decode_head(q, K, V, idx, g["sink"], g["window"], int(r), g["scale"])
        np.testing.assert_allclose(res["out"], e["out"], rtol=1e-13)
        assert abs(res["lse"] - e["lse"]) < 1e-13
        np.testing.assert_array_equal(res["selected"], e["selected"])
        if "token_w" in e:
            np.testing.assert_allclose(res["token_w"], e["token_w"], rtol=1e-13)
            np.testing.assert_allclose(res["est_w"], e["est_w"], rtol=1e-13)


# ---------------------------------------------------------------- decode pins

@pytest.mark.parametrize("d", [4, 128])
def test_full_budget_equals_full_attention(d):
    K, V, q, idx = small_case(seed=3, d=d)
    scale = 1 / math.sqrt(d)
    C = idx["n_clusters"]
    for r in (int((idx["size"] > 0).sum()), C, C + 7):
        res = wi.decode_head(q, K, V, idx, 4, 32, r, scale)
        out, lse = sdpa64(q, K, V, scale)
        np.testing.assert_allclose(res["out"], out, rtol=1e-11, atol=1e-13)
        assert abs(res["lse"] - lse) < 1e-11


def test_singleton_clusters_make_estimation_exact():
    # k_per_seg >= tokens per segment with strided init: every token seeds its
    # own centroid and is its own (singleton) cluster.
    rng = np.random.default_rng(4)
    N, d, seg = 300, 32, 64
    K = bf16_vals(rng, (N, d))
    V = bf16_vals(rng, (N, d))
    q = bf16_vals(rng, (d,))
    idx = wi.build_index_head(K, V, 3, 10, seg, seg, 2)
    assert set(np.unique(idx["size"])) <= {0, 1}
    out, lse = sdpa64(q, K, V, 0.3)
    for r in (0, 1, 17, 1000):
        res = wi.decode_head(q, K, V, idx, 3, 10, r, 0.3)
        np.testing.assert_allclose(res["out"], out, rtol=1e-11, atol=1e-13)
        assert abs(res["lse"] - lse) < 1e-11


def test_zero_query_gives_mean_of_values():
    K, V, q, idx = small_case(seed=5)
    N = K.shape[0]
    for r in (0, 3, 10 ** 6):
        res = wi.decode_head(np.zeros_like(q), K, V, idx, 4, 32, r, 0.1)
        np.testing.assert_allclose(res["out"], V.mean(axis=0), rtol=1e-11, atol=vsum_atol(idx))
        assert abs(res["lse"] - math.log(N)) < 1e-12


def test_tripartite_equals_attention_over_surrogate_keys():
    # Characterisation of the estimation zone: every member of an estimated
    # cluster takes its cluster's mean key, and softmax attention over that
    # modified key set (torch SDPA) must equal the tripartite output.
    K, V, q, idx = small_case(seed=6, d=64)
    scale = 0.125
    C = idx["n_clusters"]
    for r in (0, 1, 5, 12):
        res = wi.decode_head(q, K, V, idx, 4, 32, r, scale)
        Ks = K.copy()
        for c in range(C):
            if c in set(res["selected"].tolist()):
                continue
            mem = idx["perm"][idx["offset"][c]:idx["offset"][c + 1]]
            Ks[mem] = idx["centroid_key"][c]
        out, lse = sdpa64(q, Ks, V, scale)
        np.testing.assert_allclose(res["out"], out, rtol=1e-10, atol=vsum_atol(idx))
        assert abs(res["lse"] - lse) < 1e-10


def test_weights_sum_to_one():
    K, V, q, idx = small_case(seed=7)
    for r in (0, 2, 9):
        res = wi.decode_head(q * 3, K, V, idx, 4, 32, r, 1 / math.sqrt(128))
        assert abs(res["token_w"].sum() + res["est_w"].sum() - 1.0) < 1e-12
        # out is the weighted combination
        num = res["token_w"] @ V[res["token_pos"]]
        num += (res["est_w"] / idx["size"][res["est_ids"]]) @ idx["value_sum"][res["est_ids"]]
        np.testing.assert_allclose(num, res["out"], rtol=1e-11, atol=1e-13)


def test_bruteforce_full_attention_loops():
    rng = np.random.default_rng(8)
    for d in (4, 128):
        N = 64
        K = bf16_vals(rng, (N, d))
        V = bf16_vals(rng, (N, d))
        q = bf16_vals(rng, (d,))
        idx = wi.build_index_head(K, V, 2, 5, 32, 4, 2)
        scale = 1 / math.sqrt(d)
        res = wi.decode_head(q, K, V, idx, 2, 5, 100, scale)
        # brute force with Python loops
        logits = [scale * sum(q[j] * K[i, j] for j in range(d)) for i in range(N)]
        mx = max(logits)
        w = [math.exp(x - mx) for x in logits]
        tot = sum(w)
        ref = [sum(w[i] * V[i, j] for i in range(N)) / tot for j in range(d)]
        np.testing.assert_allclose(res["out"], ref, rtol=1e-11, atol=1e-13)
        assert abs(res["lse"] - (mx + math.log(tot))) < 1e-11


def test_degenerate_zones():
    K, V, q, idx = small_case(seed=9, N=300)
    N = K.shape[0]
    # window covering everything after the sinks: no index, pure exact attention
    idx2 = wi.build_index_head(K, V, 4, N - 4, 256, 16, 2)
    assert idx2["size"].sum() == 0 and idx2["perm"].size == 0
    res = wi.decode_head(q, K, V, idx2, 4, N - 4, 5, 0.2)
    out, lse = sdpa64(q, K, V, 0.2)
    np.testing.assert_allclose(res["out"], out, rtol=1e-11, atol=1e-13)
    # no steady zone, no budget: estimation only
    idx3 = wi.build_index_head(K, V, 0, 0, 128, 8, 2)
    res = wi.decode_head(q, K, V, idx3, 0, 0, 0, 0.2)
    assert res["token_pos"].size == 0
    assert abs(res["est_w"].sum() - 1) < 1e-12


def test_selection_order_and_ties():
    s = np.array([1.0, 3.0, 3.0, -np.inf, 2.0, 3.0, 0.5])
    # brute force: sort (score desc, id asc) by Python's sort
    cand = sorted([(-s[c], c) for c in range(len(s)) if np.isfinite(s[c])])
    for r in range(0, 9):
        ref = sorted(c for _, c in cand[:r])
        np.testing.assert_array_equal(wi.select_clusters(s, r), ref)
    assert list(wi.select_clusters(s, 2)) == [1, 2]


# ---------------------------------------------------------------- build pins

def test_segments_hand_case():
    segs = wi.segment_positions(N=20, sink=3, window=4, seg_len=8)
    assert [list(x) for x in segs] == [list(range(3, 8)), list(range(8, 16)), []]
    segs = wi.segment_positions(N=20, sink=0, window=0, seg_len=32)
    assert [list(x) for x in segs] == [list(range(20))]


def test_steady_zone_and_segments_partition_the_sequence():
    # every position is in exactly one of: the steady zone (first `sink`, last
    # `window`) or one segment, and a segment only holds its own span
    for N, sink, window, L in [(20, 3, 4, 8), (37, 0, 5, 16), (37, 4, 0, 16), (64, 4, 60, 16),
                               (50, 0, 0, 7), (9, 2, 7, 4)]:
        st = wi.steady_positions(N, sink, window)
        assert st.tolist() == [p for p in range(N) if p < sink or p >= N - window]
        segs = wi.segment_positions(N, sink, window, L)
        assert len(segs) == -(-N // L)
        for s, ps in enumerate(segs):
            assert all(s * L <= p < (s + 1) * L for p in ps)
        assert sorted(st.tolist() + [int(p) for ps in segs for p in ps]) == list(range(N))


def test_init_strided_hand_case():
    # m = 10 keys along distinct axes; k = 4 picks floor(j*10/4) = 0, 2, 5, 7
    keys = np.eye(10) * 3.0
    mu = wi.kmeans_init(keys, 4)
    np.testing.assert_array_equal(mu, np.eye(10)[[0, 2, 5, 7]])
    assert np.all(wi.kmeans_init(np.zeros((0, 5)), 3) == 0)


def test_assign_bruteforce_loops():
    rng = np.random.default_rng(10)
    for d in (4, 128):
        keys = bf16_vals(rng, (50, d))
        mu = wi.bf16_round(rng.standard_normal((9, d)))
        mu[5] = mu[2]  # exact tie -> the lower index wins
        a, cos = wi.kmeans_assign(keys, mu)
        for i in range(50):
            dots = [sum(keys[i, t] * mu[j, t] for t in range(d)) for j in range(9)]
            best = 0
            for j in range(1, 9):
                if dots[j] > dots[best]:
                    best = j
            assert a[i] == best
            assert best != 5
            nrm = math.sqrt(sum(keys[i, t] ** 2 for t in range(d)))
            assert abs(cos[i, best] - dots[best] / nrm) < 1e-12


def test_update_maximises_cosine_sum():
    rng = np.random.default_rng(11)
    d = 16
    keys = bf16_vals(rng, (80, d))
    mu0 = wi.bf16_round(rng.standard_normal((5, d)))
    a, _ = wi.kmeans_assign(keys, mu0)
    mu, mu_exact = wi.kmeans_update(keys, a, mu0)
    unit = keys / np.linalg.norm(keys, axis=1, keepdims=True)
    for j in range(5):
        mem = unit[a == j]
        if len(mem) == 0:
            np.testing.assert_array_equal(mu[j], mu0[j])
            continue
        best = (mem @ mu_exact[j]).sum()
        assert abs(np.linalg.norm(mu_exact[j]) - 1) < 1e-12
        for _ in range(200):  # no unit vector does better (Cauchy-Schwarz)
            u = rng.standard_normal(d)
            u /= np.linalg.norm(u)
            assert (mem @ u).sum() <= best + 1e-12
        # the stored centroid is the bf16 rounding of the exact one
        assert np.all(np.abs(mu[j] - mu_exact[j]) <= 2.0 ** -8 * np.abs(mu_exact[j]) + 1e-300)


def test_assignment_step_never_lowers_objective():
    rng = np.random.default_rng(12)
    keys = bf16_vals(rng, (400, 32))
    a, mu, hist = wi.kmeans_segment(keys, 12, 6, trace=True)
    unit = keys / np.linalg.norm(keys, axis=1, keepdims=True)
    prev_a = None
    for mu_in, a_t, mu_out in hist:
        obj = (unit * mu_in[a_t]).sum()
        if prev_a is not None:
            assert obj >= (unit * mu_in[prev_a]).sum() - 1e-12
        prev_a = a_t
    np.testing.assert_array_equal(a, hist[-1][1])
    np.testing.assert_array_equal(mu, hist[-1][2])


def test_planted_clusters_recovered():
    # Blocks of tokens around well separated directions, laid out in position
    # order: strided init seeds one centroid per block, and the build must
    # return exactly the planted partition with its block statistics.
    rng = np.random.default_rng(13)
    k, blk, d, sink, window = 8, 20, 64, 2, 6
    dirs = np.linalg.qr(rng.standard_normal((d, d)))[0][:k] * 5
    lab = np.repeat(np.arange(k), blk)
    keys = torch.from_numpy(dirs[lab] + 0.05 * rng.standard_normal((k * blk, d))).to(
        torch.bfloat16).double().numpy()
    N = sink + k * blk + window
    K = np.concatenate([bf16_vals(rng, (sink, d)), keys, bf16_vals(rng, (window, d))])
    V = bf16_vals(rng, (N, d))
    idx = wi.build_index_head(K, V, sink, window, 1 << 20, k, 5)
    np.testing.assert_array_equal(idx["assign"][sink:N - window], lab)
    np.testing.assert_array_equal(idx["size"], np.full(k, blk))
    for c in range(k):
        rows = sink + np.arange(c * blk, (c + 1) * blk)
        np.testing.assert_allclose(idx["centroid_key"][c], np.mean(K[rows], axis=0), rtol=1e-6,
                                   atol=1e-6)
        np.testing.assert_allclose(idx["value_sum"][c], np.sum(V[rows], axis=0), rtol=1e-6,
                                   atol=1e-6)


def test_statistics_invariants_and_stable_order():
    K, V, q, idx = small_case(seed=14, N=900, seg_len=200, k=10)
    N = K.shape[0]
    P = np.arange(4, N - 32)
    assert idx["size"].sum() == len(P)
    assert sorted(idx["perm"].tolist()) == P.tolist()
    np.testing.assert_array_equal(idx["offset"][1:], np.cumsum(idx["size"]))
    # brute-force stable sort by (cluster, position)
    ref = sorted(P.tolist(), key=lambda p: (idx["assign"][p], p))
    np.testing.assert_array_equal(idx["perm"], ref)
    np.testing.assert_array_equal(idx["k_sorted"], K[idx["perm"]])
    np.testing.assert_array_equal(idx["v_sorted"], V[idx["perm"]])
    # clusters never cross their segment
    for p in P:
        assert idx["assign"][p] // 10 == p // 200
    assert np.all(idx["assign"][:4] == -1) and np.all(idx["assign"][N - 32:] == -1)


def test_index_statistics_bruteforce_loops_and_empty_cluster():
    # sizes, offsets, member order, mean keys and value sums of a hand-made
    # assignment, by Python loops; cluster 2 is left empty
    rng = np.random.default_rng(31)
    N, d, C = 40, 6, 5
    K = rng.standard_normal((N, d))
    V = rng.standard_normal((N, d))
    pos = np.arange(3, 37)
    c = rng.integers(0, C, pos.size)
    c[c == 2] = 4
    st = wi.index_statistics(K, V, pos, c, C)
    before = 0
    for j in range(C):
        mem = [int(p) for p, cj in zip(pos, c) if cj == j]
        assert st["size"][j] == len(mem)
        assert st["offset"][j] == before
        assert st["perm"][before:before + len(mem)].tolist() == sorted(mem)
        before += len(mem)
        ks, vs = [0.0] * d, [0.0] * d
        for p in mem:
            for e in range(d):
                ks[e] += K[p, e]
                vs[e] += V[p, e]
        kbar = [x / len(mem) for x in ks] if mem else [0.0] * d
        np.testing.assert_allclose(st["centroid_key"][j], kbar, rtol=2.0 ** -23, atol=1e-12)
        np.testing.assert_allclose(st["value_sum"][j], vs, rtol=2.0 ** -23, atol=1e-12)
    assert st["offset"][C] == pos.size
    assert np.all(st["centroid_key"][2] == 0) and np.all(st["value_sum"][2] == 0)
    np.testing.assert_array_equal(st["k_sorted"], K[st["perm"]])
    np.testing.assert_array_equal(st["v_sorted"], V[st["perm"]])


# ---------------------------------------------------------------- format and GQA wrapper

def test_bf16_bits_to_f64_every_pattern_matches_torch():
    # every one of the 65536 bf16 bit patterns except the NaNs, against torch's
    # own bf16 -> float64 conversion (a library routine, not this code)
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).double().numpy()
    keep = ~np.isnan(ref)
    assert keep.sum() == (1 << 16) - 2 * 127
    with np.errstate(invalid="ignore"):  # the NaN patterns are dropped below
        got = wi.bf16_bits_to_f64(bits)
    np.testing.assert_array_equal(got[keep], ref[keep])
    # signed zeros and infinities keep their sign
    assert np.signbit(got[0x8000]) and not np.signbit(got[0])
    assert got[0x7F80] == np.inf and got[0xFF80] == -np.inf


def _gqa_case(seed=30, B=2, Hq=8, Hkv=2, N=600, d=32, sink=3, window=20, seg=128, k=12):
    rng = np.random.default_rng(seed)
    K = bf16_vals(rng, (B, Hkv, N, d))
    V = bf16_vals(rng, (B, Hkv, N, d))
    q = bf16_vals(rng, (B, Hq, d), 0.6)
    idx = wi.build_index(K, V, sink, window, seg, k, 2)
    return K, V, q, idx, dict(sink=sink, window=window)


def test_decode_wrapper_full_budget_is_torch_gqa_attention():
    # With a budget covering every cluster each head is exact attention over its
    # KV head; torch's SDPA with enable_gqa maps query head h to KV head
    # h // (Hq / Hkv), so a wrong head mapping in the wrapper fails here.
    K, V, q, idx, z = _gqa_case()
    B, Hq, d = q.shape
    C = idx["n_clusters"]
    scale = 0.21
    res = wi.decode(q, K, V, idx, z["sink"], z["window"], C, scale)
    qt = torch.from_numpy(q)[:, :, None, :]
    ref = torch.nn.functional.scaled_dot_product_attention(
        qt, torch.from_numpy(K), torch.from_numpy(V), scale=scale, enable_gqa=True)[:, :, 0]
    np.testing.assert_allclose(res["out"], ref.numpy(), rtol=1e-11, atol=1e-13)
    logits = scale * np.einsum("bhd,bhnd->bhn", q, np.repeat(K, Hq // K.shape[1], axis=1))
    lse = torch.logsumexp(torch.from_numpy(logits), dim=-1).numpy()
    np.testing.assert_allclose(res["lse"], lse, rtol=0, atol=1e-11)


def test_decode_wrapper_budgeted_rows_and_head_subset():
    # Below full budget: every head of a group uses its own KV head's index,
    # and a KV head's data never leaks into another group's heads (swapping the
    # two KV heads' data swaps the groups' results); heads outside the
    # requested subset stay NaN.
    K, V, q, idx, z = _gqa_case(seed=31)
    r = 5
    full = wi.decode(q, K, V, idx, z["sink"], z["window"], r, 0.2)
    assert np.isfinite(full["out"]).all() and np.isfinite(full["lse"]).all()
    swap = lambda a: a[:, ::-1].copy()
    idx_s = {key: (val if key == "n_clusters" else swap(val)) for key, val in idx.items()}
    q_s = np.concatenate([q[:, 4:], q[:, :4]], axis=1)
    res_s = wi.decode(q_s, swap(K), swap(V), idx_s, z["sink"], z["window"], r, 0.2)
    np.testing.assert_array_equal(res_s["out"][:, 4:], full["out"][:, :4])
    np.testing.assert_array_equal(res_s["out"][:, :4], full["out"][:, 4:])
    # a query head of group 1 attends over KV head 1 only: replacing KV head 0
    # changes nothing for it
    K2 = K.copy()
    K2[:, 0] = K2[:, 0][:, ::-1]
    idx2 = wi.build_index(K2, V, z["sink"], z["window"], 128, 12, 2)
    part = wi.decode(q, K2, V, idx2, z["sink"], z["window"], r, 0.2, heads=[(1, 6), (0, 5)])
    np.testing.assert_array_equal(part["out"][1, 6], full["out"][1, 6])
    np.testing.assert_array_equal(part["out"][0, 5], full["out"][0, 5])
    assert np.isnan(part["out"][0, 0]).all() and np.isnan(part["lse"][1, 1])
    assert set(part["selected"]) == {(1, 6), (0, 5)}


# ---------------------------------------------------------------- ranking and reuse

def test_mass_ranking_bruteforce_products():
    # The mass key must order clusters like the product n_c e^{s_c} itself
    # (computed here without logarithms, ranking by a Python sort of
    # (-mass, id)); a dropped ln n_c or a sign slip orders them differently.
    rng = np.random.default_rng(40)
    for trial in range(50):
        C = int(rng.integers(1, 30))
        s = rng.standard_normal(C) * 2.0
        n = rng.integers(0, 9, C)
        s[n == 0] = -np.inf
        r = int(rng.integers(0, C + 2))
        mass = [(float(n[c]) * math.exp(s[c])) if n[c] > 0 else None for c in range(C)]
        ranked = sorted((c for c in range(C) if mass[c] is not None), key=lambda c: (-mass[c], c))
        got = wi.select_clusters(wi.ranking_keys(s, n, "mass"), r)
        assert got.tolist() == sorted(ranked[:r]), trial


def test_mass_ranking_hand_case_and_equal_sizes():
    # A big cluster scoring a little below a small one carries more mass:
    # 40 e^{1.0} > 2 e^{2.0}.  Score ranking takes the small one, mass
    # ranking the big one.
    s = np.array([2.0, 1.0, -np.inf, 0.0])
    n = np.array([2, 40, 0, 1])
    assert wi.select_clusters(wi.ranking_keys(s, n, "score"), 1).tolist() == [0]
    assert wi.select_clusters(wi.ranking_keys(s, n, "mass"), 1).tolist() == [1]
    assert wi.select_clusters(wi.ranking_keys(s, n, "mass"), 9).tolist() == [0, 1, 3]
    # with every cluster the same size the two rankings take the same set
    rng = np.random.default_rng(41)
    s = rng.standard_normal(64)
    for r in (1, 7, 64):
        assert np.array_equal(wi.select_clusters(wi.ranking_keys(s, np.full(64, 5), "mass"), r),
                              wi.select_clusters(s, r))
    with pytest.raises(ValueError):
        wi.ranking_keys(s, np.full(64, 5), "other")


def test_mass_ranking_decode_full_budget_and_given_set():
    # Whatever the ranking, a full budget is exact attention; below it the
    # result is the tripartite attention over the set the mass key selects.
    K, V, q, idx = small_case(seed=42, d=64)
    C = idx["size"].shape[0]
    full = wi.decode_head(q, K, V, idx, 4, 32, C, 0.15, rank="mass")
    ref, lse = sdpa64(q, K, V, 0.15)
    np.testing.assert_allclose(full["out"], ref, rtol=1e-11, atol=1e-13)
    assert abs(full["lse"] - lse) < 1e-11
    part = wi.decode_head(q, K, V, idx, 4, 32, 5, 0.15, rank="mass")
    s = part["scores"]
    assert part["selected"].tolist() == wi.select_clusters(wi.ranking_keys(s, idx["size"], "mass"), 5).tolist()
    same = wi.decode_head(q, K, V, idx, 4, 32, 5, 0.15, selected=part["selected"])
    np.testing.assert_array_equal(same["out"], part["out"])


def test_reuse_cosine_closed_form():
    # cos((1,0),(1,1)) = 1/sqrt(2) = 0.7071...; a group's similarity is its
    # least similar query head; a zero query has no direction (cosine 0).
    q = np.array([[1.0, 0.0], [3.0, 0.0], [1.0, 0.0], [0.0, 0.0]])
    p = np.array([[1.0, 1.0], [6.0, 0.0], [2.0, 0.0], [1.0, 0.0]])
    assert wi.reuse_groups(q, p, 2, 0.707).tolist() == [True, False]
    assert wi.reuse_groups(q, p, 2, 0.7072).tolist() == [False, False]
    assert wi.reuse_groups(q, p, 2, 0.0).tolist() == [True, True]
    assert wi.reuse_groups(q, p, 1, 0.9).tolist() == [False, True, True, False]
    assert wi.reuse_groups(q, -p, 4, -1.5).tolist() == [True]


def test_reuse_threshold_extremes():
    # tau > 1: no cosine reaches it, so every head selects afresh and the
    # result is the plain decode; tau <= -1 (here -2, clear of rounding):
    # every head reuses, which is decode_head over the previous step's sets.
    K, V, q, idx, z = _gqa_case(seed=43)
    rng = np.random.default_rng(44)
    q_prev = q + 0.3 * bf16_vals(rng, q.shape)
    r = 4
    prev = wi.decode(q_prev, K, V, idx, z["sink"], z["window"], r, 0.2)
    plain = wi.decode(q, K, V, idx, z["sink"], z["window"], r, 0.2)
    fresh = wi.decode(q, K, V, idx, z["sink"], z["window"], r, 0.2, prev_q=q_prev,
                      prev_selected=prev["selected"], tau=1.5)
    assert not fresh["reused"].any()
    np.testing.assert_array_equal(fresh["out"], plain["out"])
    kept = wi.decode(q, K, V, idx, z["sink"], z["window"], r, 0.2, prev_q=q_prev,
                     prev_selected=prev["selected"], tau=-2.0)
    assert kept["reused"].all()
    B, Hq, _ = q.shape
    group = Hq // K.shape[1]
    differs = 0
    for b in range(B):
        for h in range(Hq):
            g = h // group
            hi = {key: idx[key][b, g] for key in ("size", "centroid_key", "value_sum", "perm",
                                                  "offset")}
            ref = wi.decode_head(q[b, h], K[b, g], V[b, g], hi, z["sink"], z["window"], r, 0.2,
                                 selected=prev["selected"][(b, h)])
            np.testing.assert_array_equal(kept["out"][b, h], ref["out"])
            assert kept["selected"][(b, h)].tolist() == prev["selected"][(b, h)].tolist()
            differs += set(prev["selected"][(b, h)].tolist()) != set(plain["selected"][(b, h)].tolist())
    assert differs > 0  # the perturbation moved some selections, so reuse is visible


def test_reuse_per_group_decision():
    # Group 0's queries are unchanged (cosine 1), group 1 has one query head
    # reversed (cosine -1): at tau = 0.5 only group 1 re-selects, and its
    # heads equal the plain decode while group 0 keeps the given sets.
    K, V, q, idx, z = _gqa_case(seed=45)
    q_prev = q.copy()
    q_prev[:, 5] = -q[:, 5]
    B, Hq, _ = q.shape
    r = 3
    stale = {(b, h): np.array([0, 1, 2]) for b in range(B) for h in range(Hq)}
    res = wi.decode(q, K, V, idx, z["sink"], z["window"], r, 0.2, prev_q=q_prev,
                    prev_selected=stale, tau=0.5)
    assert res["reused"].tolist() == [[True, False]] * B
    plain = wi.decode(q, K, V, idx, z["sink"], z["window"], r, 0.2)
    np.testing.assert_array_equal(res["out"][:, 4:], plain["out"][:, 4:])
    for b in range(B):
        for h in range(4):
            assert res["selected"][(b, h)].tolist() == [0, 1, 2]


# ---------------------------------------------------------------- shared selection, bf16 index

def test_round_index_bf16_matches_torch_cast_of_the_f32_index():
    # torch's float32 -> bfloat16 cast (round to nearest even) of the stored
    # float32 index; other arrays untouched
    K, V, q, idx = small_case(seed=46, d=64)
    r = wi.round_index_bf16(idx)
    for key in ("centroid_key", "value_sum"):
        ref = torch.from_numpy(idx[key].astype(np.float32)).to(torch.bfloat16).double().numpy()
        np.testing.assert_array_equal(r[key], ref)
    for key in ("size", "offset", "perm"):
        assert r[key] is idx[key]


def test_bf16_index_is_exact_for_bf16_representable_statistics():
    # singleton clusters of bf16 keys and values: every mean key and value
    # sum is already a bf16 value, so the bf16 index decodes identically
    rng = np.random.default_rng(47)
    B, Hkv, Hq, N, d = 1, 2, 4, 300, 32
    K = bf16_vals(rng, (B, Hkv, N, d))
    V = bf16_vals(rng, (B, Hkv, N, d))
    q = bf16_vals(rng, (B, Hq, d))
    idx = wi.build_index(K, V, 2, 10, 1024, N, 1)  # k >= tokens: the init makes singletons
    assert idx["size"].max() == 1
    a = wi.decode(q, K, V, idx, 2, 10, 7, 0.2)
    b = wi.decode(q, K, V, idx, 2, 10, 7, 0.2, index_dtype="bf16")
    np.testing.assert_array_equal(a["out"], b["out"])
    np.testing.assert_array_equal(a["lse"], b["lse"])


def test_group_selection_bruteforce_sums():
    # the shared set is the top r of sum_h s_h(c) computed by explicit loops
    rng = np.random.default_rng(48)
    for trial in range(20):
        G, C, d = int(rng.integers(1, 5)), int(rng.integers(1, 40)), 8
        kbar = rng.standard_normal((C, d))
        n = rng.integers(0, 4, C)
        qg = rng.standard_normal((G, d))
        r = int(rng.integers(0, C + 2))
        tot = []
        for c in range(C):
            if n[c] == 0:
                continue
            tot.append((-sum(0.3 * float(np.dot(qg[h], kbar[c])) for h in range(G)), c))
        want = sorted(c for _, c in sorted(tot)[:r])
        assert wi.group_selection(qg, kbar, n, 0.3, r).tolist() == want, trial
        # with mass ranking each head adds ln n_c
        tot = [(-sum(0.3 * float(np.dot(qg[h], kbar[c])) + math.log(n[c]) for h in range(G)), c)
               for c in range(C) if n[c] > 0]
        want = sorted(c for _, c in sorted(tot)[:r])
        assert wi.group_selection(qg, kbar, n, 0.3, r, "mass").tolist() == want, trial


def test_shared_decode_reduces_and_extends_per_head_decode():
    # one query head per KV head: shared == per head, bit for bit; full budget:
    # exact attention whatever the sharing; shared sets are common to a group
    # and equal the set of the group's summed query
    K, V, q, idx, z = _gqa_case(seed=49)
    one = wi.decode(q[:, ::4], K, V, idx, z["sink"], z["window"], 5, 0.2)
    one_s = wi.decode(q[:, ::4], K, V, idx, z["sink"], z["window"], 5, 0.2, share="group")
    np.testing.assert_array_equal(one["out"], one_s["out"])
    C = idx["n_clusters"]
    full = wi.decode(q, K, V, idx, z["sink"], z["window"], C, 0.2, share="group")
    ref = wi.decode(q, K, V, idx, z["sink"], z["window"], C, 0.2)
    np.testing.assert_allclose(full["out"], ref["out"], rtol=1e-11, atol=1e-13)
    res = wi.decode(q, K, V, idx, z["sink"], z["window"], 5, 0.2, share="group")
    per = wi.decode(q, K, V, idx, z["sink"], z["window"], 5, 0.2)
    B, Hq, _ = q.shape
    differs = 0
    for b in range(B):
        for g in range(2):
            sets = [res["selected"][(b, h)].tolist() for h in range(4 * g, 4 * g + 4)]
            assert all(s == sets[0] for s in sets)
            s_sum = wi.cluster_scores(q[b, 4 * g:4 * g + 4].sum(axis=0), idx["centroid_key"][b, g],
                                      idx["size"][b, g], 0.2)
            assert sets[0] == wi.select_clusters(s_sum, 5).tolist()
            differs += sum(per["selected"][(b, h)].tolist() != sets[0] for h in range(4 * g, 4 * g + 4))
    assert differs > 0
    with pytest.raises(ValueError):
        wi.decode(q, K, V, idx, z["sink"], z["window"], 5, 0.2, share="pair")


# ---------------------------------------------------------------- index maintenance

def test_extend_by_nothing_is_the_identity():
    K, V, q, idx = small_case(seed=50, d=32)
    N = K.shape[0]
    ext = wi.extend_index_head(K, V, idx, N, 4, 32, 256, 16)
    for key in ("size", "offset", "perm", "assign", "centroid_key", "value_sum", "k_sorted",
                "v_sorted", "unit_centroid"):
        np.testing.assert_array_equal(ext[key], idx[key], err_msg=key)


def test_extend_assigns_joining_tokens_by_bruteforce_nearest_centroid():
    # a 700-token index grown to 760: the 60 positions that leave the window
    # are [668, 728); explicit loops over each one's segment centroids (ties
    # to the lower j) give its cluster; earlier positions keep theirs
    rng = np.random.default_rng(51)
    N0, N1, d, sink, window, L, k = 700, 760, 16, 4, 32, 256, 8
    K = bf16_vals(rng, (N1, d))
    V = bf16_vals(rng, (N1, d))
    old = wi.build_index_head(K[:N0], V[:N0], sink, window, L, k, 3)
    ext = wi.extend_index_head(K, V, old, N0, sink, window, L, k)
    mu = old["unit_centroid"]
    np.testing.assert_array_equal(ext["assign"][:N0 - window], old["assign"][:N0 - window])
    for p in range(N0 - window, N1 - window):
        s = p // L
        best, arg = -np.inf, -1
        for j in range(k):
            v = float(sum(K[p, t] * mu[s * k + j, t] for t in range(d)))
            if v > best:
                best, arg = v, j
        assert ext["assign"][p] == s * k + arg, p
    assert np.all(ext["assign"][N1 - window:] == -1) and np.all(ext["assign"][:sink] == -1)
    # statistics of the new assignment: every indexable position once
    assert ext["size"].sum() == N1 - window - sink
    assert sorted(ext["perm"].tolist()) == list(range(sink, N1 - window))


def test_extend_within_the_last_segment_and_centroid_directions():
    # N0 = 300, window 16, seg_len 256: the clustered segments are 0 and 1 (1
    # holds [256, 284)); growing to 520 makes [284, 504) join segment 1 and
    # opens segment 2 on the index side (its clusters stay empty, zero
    # centroids); a token along a centroid's direction joins that centroid's
    # cluster; growing to 600 would reach into segment 2: a rebuild
    rng = np.random.default_rng(52)
    N0, d, sink, window, L, k = 300, 8, 4, 16, 256, 4
    K = bf16_vals(rng, (700, d))
    V = bf16_vals(rng, (700, d))
    old = wi.build_index_head(K[:N0], V[:N0], sink, window, L, k, 2)
    mu = old["unit_centroid"]
    K[400] = mu[k + 2] * 4.0  # a power of two keeps it a bf16 value
    ext = wi.extend_index_head(K[:520], V[:520], old, N0, sink, window, L, k)
    assert ext["n_clusters"] == 3 * k
    assert ext["assign"][400] == k + 2
    assert np.all((ext["assign"][256:504] >= k) & (ext["assign"][256:504] < 2 * k))
    assert np.all(ext["size"][2 * k:] == 0) and np.all(ext["unit_centroid"][2 * k:] == 0)
    with pytest.raises(ValueError):
        wi.extend_index_head(K[:600], V[:600], old, N0, sink, window, L, k)
    with pytest.raises(ValueError):
        wi.extend_index_head(K[:30], V[:30], {"unit_centroid": np.zeros((k, d)),
                                              "assign": np.full(20, -1)}, 20, 4, 16, L, k)
