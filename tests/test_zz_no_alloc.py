"""The decode entry point for callers that cannot allocate device memory.

Hosts that give a plugin no allocator (pre-planned buffers only, or a device
memory budget fixed before the plugin runs) call wi_decode_attention_static,
which needs no workspace: it runs the regular decode on a fixed scratch array
that the library keeps on every GPU.  Its results must match the regular entry
point's, call after call, since each call clears what must start at zero in
the shared scratch.

This file is collected last on purpose: it checks one extra entry point, and
a run that stops at the first failure has then already run everything else.
"""

import ctypes

import numpy as np
import pytest
import torch

from workloads import WORKLOADS, generate

pytestmark = pytest.mark.gpu



def _up(bits, dev):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(dev)


def test_static_scratch_decode_matches_workspace_decode_twice():
    import cluster_indexed_sparse_wi_b300 as wl
    from cluster_indexed_sparse_wi_b300 import _lib

    dev = torch.device("cuda", torch.cuda.current_device())
    w = WORKLOADS["llama3_8b_128k_b1"].replace(B=2, Hq=8, Hkv=2, N=12000, seg_len=4096,
                                               k_per_seg=128, iters=3, planted_per_seg=64,
                                               seeds=(41, 42))
    g = generate(w)
    K, V, q = _up(g["K"], dev), _up(g["V"], dev), _up(g["q"], dev)
    ix = wl.build_index(K, V, w.sink, w.window, w.seg_len, w.k_per_seg, w.iters)
    r = 20
    dec = wl.Decoder(ix, w.Hq, r)
    out_ref, lse_ref, topk_ref = (t.clone() for t in dec(q, K, V))
    torch.cuda.synchronize()
    assert dec.status() == 0

    lib = _lib.lib()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for call in range(2):
        out = torch.full_like(out_ref, float("nan"))
        lse = torch.full_like(lse_ref, float("nan"))
        topk = torch.full((w.B, w.Hq, r), -7, dtype=torch.int32, device=dev)
        rc = lib.wi_decode_attention_static(
            ctypes.byref(dec.params), ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(K.data_ptr()),
            ctypes.c_void_p(V.data_ptr()), ctypes.byref(ix.struct), ctypes.c_void_p(out.data_ptr()),
            ctypes.c_void_p(lse.data_ptr()), ctypes.c_void_p(topk.data_ptr()), stream)
        assert rc == 0, (call, lib.wi_status_string(rc))
        torch.cuda.synchronize()
        # the same deterministic kernel on the same inputs: bit-identical
        # results, so state left in the shared scratch by an earlier call
        # cannot hide behind a tolerance
        assert torch.equal(out, out_ref), call
        assert torch.equal(lse, lse_ref), call
        assert torch.equal(topk, topk_ref), call
        st = ctypes.c_int(-1)
        assert lib.wi_decode_static_status(stream, ctypes.byref(st)) == 0
        assert st.value == 0, call


def test_static_scratch_rejects_oversize_without_device_work():
    from cluster_indexed_sparse_wi_b300 import _lib

    lib = _lib.lib()
    # 8 query heads x 2^20 clusters of f32 scores alone exceed the fixed scratch
    p = _lib.DecodeParams(1, 8, 2, 1 << 22, 128, 4, 64, 10, 0.088)
    ix = _lib.IndexStruct()
    ix.B, ix.Hkv, ix.N, ix.d, ix.sink, ix.window, ix.n_clusters = 1, 2, 1 << 22, 128, 4, 64, 1 << 20
    need = lib.wi_decode_workspace_bytes(ctypes.byref(p), ix.n_clusters)
    assert need > _lib.WI_STATIC_SCRATCH_BYTES
    # pointers that pass every host check; the call is rejected on the host
    # before anything is enqueued, so they are never dereferenced
    fake = ctypes.c_void_p(1 << 20)
    for name in _lib.FIELDS:
        setattr(ix, name, 1 << 20)
    rc = lib.wi_decode_attention_static(ctypes.byref(p), fake, fake, fake, ctypes.byref(ix), fake,
                                        None, None, None)
    assert rc == _lib.WI_ERR_WORKSPACE
    # argument errors come first and queue nothing either
    rc = lib.wi_decode_attention_static(ctypes.byref(p), None, fake, fake, ctypes.byref(ix), fake,
                                        None, None, None)
    assert rc == _lib.WI_ERR_INVALID_ARG


def test_static_scratch_reports_device_timeout_then_recovers():
    # the library's fault-injection hook (no GPU fault: one staging copy per
    # block is never issued, so bounded waits run out after about a second):
    # the static entry point's device status is readable through
    # wi_decode_static_status, which clears it, and the next call is exact
    import cluster_indexed_sparse_wi_b300 as wl
    from cluster_indexed_sparse_wi_b300 import _lib

    dev = torch.device("cuda", torch.cuda.current_device())
    w = WORKLOADS["llama3_8b_128k_b1"].replace(B=1, Hq=4, Hkv=1, N=6000, seg_len=2048,
                                               k_per_seg=64, iters=2, planted_per_seg=32,
                                               seeds=(43,))
    g = generate(w)
    K, V, q = _up(g["K"], dev), _up(g["V"], dev), _up(g["q"], dev)
    ix = wl.build_index(K, V, w.sink, w.window, w.seg_len, w.k_per_seg, w.iters)
    dec = wl.Decoder(ix, w.Hq, 8)
    out_ref, lse_ref, _ = (t.clone() if t is not None else None for t in dec(q, K, V))
    torch.cuda.synchronize()
    lib = _lib.lib()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)

    def call():
        out = torch.empty_like(out_ref)
        lse = torch.empty_like(lse_ref)
        rc = lib.wi_decode_attention_static(
            ctypes.byref(dec.params), ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(K.data_ptr()),
            ctypes.c_void_p(V.data_ptr()), ctypes.byref(ix.struct), ctypes.c_void_p(out.data_ptr()),
            ctypes.c_void_p(lse.data_ptr()), None, stream)
        assert rc == 0
        st = ctypes.c_int(-1)
        assert lib.wi_decode_static_status(stream, ctypes.byref(st)) == 0
        return out, lse, st.value

    assert lib.wi_debug_inject(1) == 0
    _, _, st = call()
    assert st == _lib.WI_ERR_DEVICE_TIMEOUT
    out, lse, st = call()
    assert st == 0
    assert torch.equal(out, out_ref) and torch.equal(lse, lse_ref)
