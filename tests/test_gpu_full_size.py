"""GPU parity at the full sizes of the bench workloads.

The check runs the decode launch that bench.py times: one fused decode call
over an index built on the GPU.  Sampled query heads are then compared with
the oracle, which runs on the index the GPU used (downloaded for the head's
KV group).

* 128K context: 8192 clusters per head, r = 148; one round of index tiles,
  selection values held in registers.
* 1M context: 65536 clusters per head, r = 656; four rounds of index tiles,
  selection values re-read per pass.
* 128K context, batch 16: seven rounds of index tiles (value-sum tiles of
  earlier rounds read their scores back), heads of several sequences.
* 128K context with the bf16 index (two index tiles per staging stage).

Tolerances are those of test_gpu_decode:
* cluster scores: relative 1e-5;
* selected sets: exact up to ties;
* outputs: maximum relative error <= 1e-2 per head;
* lse: within 1e-3.
"""

import numpy as np
import pytest
import torch

from oracle import wave_index as wi
from workloads import WORKLOADS, generate
from tests._util import bf16_tensor, rel_err, sets_match_mod_ties

pytestmark = pytest.mark.gpu

OUT_TOL = 1e-2
LSE_TOL = 1e-3
SCORE_TOL = 1e-5


def gpu_head_index(ix, b, g):
    return {"size": ix.size[b, g].cpu().numpy().astype(np.int64),
            "centroid_key": ix.centroid_key[b, g].double().cpu().numpy(),
            "value_sum": ix.value_sum[b, g].double().cpu().numpy(),
            "perm": ix.perm[b, g].cpu().numpy().astype(np.int64),
            "offset": ix.offset[b, g].cpu().numpy().astype(np.int64)}


@pytest.mark.parametrize("name,heads,index_dtype", [
    ("llama3_8b_128k_b1", [(0, 0), (0, 13), (0, 22), (0, 31)], "f32"),
    ("llama3_8b_128k_b1", [(0, 2), (0, 29)], "bf16"),
    ("llama3_8b_1m_b1", [(0, 5), (0, 30)], "f32"),
    ("llama3_8b_128k_b16", [(0, 3), (7, 17), (15, 30)], "f32")])
def test_full_size_sampled_heads(name, heads, index_dtype):
    import cluster_indexed_sparse_wi_b300 as wl
    w = WORKLOADS[name]
    g = generate(w)
    dev = torch.device("cuda", 0)
    K, V, q = (bf16_tensor(g[n], "cuda") for n in ("K", "V", "q"))
    cfg = wl.IndexConfig(w.B, w.Hkv, w.N, w.sink, w.window, w.seg_len, w.k_per_seg, w.iters)
    ix = wl.WaveIndex(cfg, dev)
    ix.build(K, V)
    torch.cuda.synchronize()
    assert ix.status() == 0
    dec = wl.Decoder(ix, w.Hq, w.r, index_dtype=index_dtype)
    out, lse, topk = dec(q, K, V)
    torch.cuda.synchronize()
    assert dec.status() == 0
    out, lse, topk = out.cpu().numpy(), lse.cpu().numpy(), topk.cpu().numpy()
    scores = dec.scores().cpu().numpy()
    G = w.Hq // w.Hkv
    groups = {}
    for b, h in heads:
        gg = h // G
        if (b, gg) not in groups:
            hi = gpu_head_index(ix, b, gg)
            if index_dtype == "bf16":
                hi = wi.round_index_bf16(hi)
            groups[(b, gg)] = (wi.bf16_bits_to_f64(g["K"][b, gg]),
                               wi.bf16_bits_to_f64(g["V"][b, gg]), hi)
        Kf, Vf, hi = groups[(b, gg)]
        qf = wi.bf16_bits_to_f64(g["q"][b, h])
        ref = wi.decode_head(qf, Kf, Vf, hi, w.sink, w.window, w.r, dec.scale)
        s_ref = ref["scores"]
        fin = np.isfinite(s_ref)
        assert np.array_equal(np.isfinite(scores[b, h]), fin)
        np.testing.assert_allclose(scores[b, h][fin], s_ref[fin], rtol=SCORE_TOL, atol=SCORE_TOL)
        sel = topk[b, h][topk[b, h] >= 0]
        assert len(sel) == min(w.r, int(fin.sum()))
        assert np.all(np.diff(sel) > 0)  # ascending ids
        assert sets_match_mod_ties(sel, ref["selected"], s_ref, SCORE_TOL)
        if set(sel.tolist()) != set(ref["selected"].tolist()):
            ref = wi.decode_head(qf, Kf, Vf, hi, w.sink, w.window, w.r, dec.scale, selected=sel)
        e = rel_err(out[b, h], ref["out"])
        assert e <= OUT_TOL, (name, b, h, e)
        assert abs(lse[b, h] - ref["lse"]) <= LSE_TOL, (name, b, h, lse[b, h], ref["lse"])
