"""The C-ABI library loads, exports every symbol include/wi.h declares, and
rejects invalid arguments on the host.  CPU only: no call here reaches the
device (every call below fails validation before any CUDA call)."""

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    from cluster_indexed_sparse_wi_b300 import build_lib
    build_lib.build()
    from cluster_indexed_sparse_wi_b300 import _lib
    return _lib


def header_symbols():
    text = open(os.path.join(ROOT, "include", "wi.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return re.findall(r"^\s*WI_API\s+(?:const\s+)?\w+(?:\s+\w+)?\s*\*?\s*(wi_\w+)\s*\(", text, flags=re.M)


def test_header_declares_the_binding_symbols(L):
    syms = header_symbols()
    assert syms == L.SYMBOLS


def test_library_exports_every_header_symbol(L):
    lib = L.lib()
    for s in header_symbols():
        assert hasattr(lib, s), s
    out = os.popen("nm -D --defined-only %s" % L.LIB_PATH).read()
    exported = set(re.findall(r" T (wi_\w+)", out))
    assert exported == set(header_symbols())


def test_status_strings_and_version(L):
    lib = L.lib()
    assert lib.wi_status_string(0) == b"ok"
    assert lib.wi_status_string(L.WI_ERR_DEVICE_TIMEOUT) == b"device-side wait timed out"
    assert lib.wi_version() == b"0.1.0"


def bp(L, **kw):
    p = dict(B=1, Hkv=2, N=4096, d=128, sink=4, window=64, seg_len=1024, k_per_seg=64, iters=3)
    p.update(kw)
    return L.BuildParams(*[p[k] for k in ("B", "Hkv", "N", "d", "sink", "window", "seg_len",
                                          "k_per_seg", "iters")])


def test_index_sizes(L):
    lib = L.lib()
    out = (ctypes.c_size_t * 9)()
    assert lib.wi_index_sizes(ctypes.byref(bp(L)), out) == 0
    C, n_idx = 4 * 64, 4096 - 68
    assert out[0] == 2 * C * 128 * 4 and out[1] == 2 * C * 128 * 2
    assert out[3] == 2 * C * 4 and out[4] == 2 * (C + 1) * 4
    assert out[5] == 2 * n_idx * 4 and out[6] == 2 * 4096 * 4
    assert out[7] == 2 * n_idx * 256
    assert lib.wi_build_workspace_bytes(ctypes.byref(bp(L))) >= 2 * 4096 * 4


@pytest.mark.parametrize("kw,code", [
    (dict(d=64), 2), (dict(sink=4000, window=100), 1), (dict(iters=0), 1),
    (dict(seg_len=0), 1), (dict(seg_len=1 << 15), 2), (dict(k_per_seg=513), 2),
    (dict(N=0), 1), (dict(window=-1), 1),
])
def test_build_param_validation(L, kw, code):
    lib = L.lib()
    out = (ctypes.c_size_t * 9)()
    assert lib.wi_index_sizes(ctypes.byref(bp(L, **kw)), out) == code
    assert lib.wi_build_workspace_bytes(ctypes.byref(bp(L, **kw))) == 0
    ix = L.IndexStruct()
    fake = ctypes.c_void_p(1 << 20)
    assert lib.wi_build_index(ctypes.byref(bp(L, **kw)), fake, fake, ctypes.byref(ix), fake,
                              1 << 30, None) == code


def test_build_pointer_and_workspace_checks(L):
    lib = L.lib()
    fake = ctypes.c_void_p(1 << 20)
    ix = L.IndexStruct()
    p = bp(L)
    # NULL K
    assert lib.wi_build_index(ctypes.byref(p), None, fake, ctypes.byref(ix), fake, 1 << 30,
                              None) == L.WI_ERR_INVALID_ARG
    # workspace too small
    assert lib.wi_build_index(ctypes.byref(p), fake, fake, ctypes.byref(ix), fake, 16,
                              None) == L.WI_ERR_WORKSPACE
    # misaligned K
    assert lib.wi_build_index(ctypes.byref(p), ctypes.c_void_p((1 << 20) + 8), fake,
                              ctypes.byref(ix), fake, 1 << 30, None) == L.WI_ERR_ALIGNMENT
    # index arrays not set (NULL)
    assert lib.wi_build_index(ctypes.byref(p), fake, fake, ctypes.byref(ix), fake, 1 << 30,
                              None) == L.WI_ERR_INVALID_ARG
    # an assign step on an index recorded for other parameters
    for name in L.FIELDS:
        setattr(ix, name, 1 << 20)
    ix.B, ix.Hkv, ix.N, ix.d = 1, 2, 4096, 128
    ix.sink, ix.window, ix.seg_len, ix.k_per_seg, ix.n_clusters = 4, 64, 1024, 64, 999
    assert lib.wi_kmeans_assign(ctypes.byref(p), fake, ctypes.byref(ix), fake, 1 << 30,
                                None) == L.WI_ERR_INDEX_MISMATCH


def dp(L, **kw):
    p = dict(B=1, Hq=8, Hkv=2, N=4096, d=128, sink=4, window=64, r=8, scale=0.088)
    p.update(kw)
    return L.DecodeParams(*[p[k] for k in ("B", "Hq", "Hkv", "N", "d", "sink", "window", "r")],
                          p["scale"])


def test_decode_layout(L):
    lib = L.lib()
    lay = L.DecodeLayout()
    assert lib.wi_decode_workspace_layout(ctypes.byref(dp(L)), 256, ctypes.byref(lay)) == 0
    assert lay.total == lib.wi_decode_workspace_bytes(ctypes.byref(dp(L)), 256)
    regions = [lay.counters, lay.scores, lay.head_max, lay.selected, lay.sel_rows,
               lay.sel_counts, lay.sel_prefix, lay.sel_scores, lay.head_tokens,
               lay.group_values, lay.partials, lay.total]
    assert regions == sorted(regions) and all(r % 256 == 0 for r in regions)
    assert lay.head_max - lay.scores >= 8 * 256 * 4
    # launch-wide words, then one scored-tile counter per KV group and one
    # partial counter per query head
    assert lay.scores - lay.counters == lay.counter_bytes >= 256 + (2 + 8) * 4
    for lo, hi in ((lay.selected, lay.sel_rows), (lay.sel_rows, lay.sel_counts),
                   (lay.sel_counts, lay.sel_prefix), (lay.sel_prefix, lay.sel_scores),
                   (lay.sel_scores, lay.head_tokens)):
        assert hi - lo >= 8 * 8 * 4
    assert lay.partials - lay.group_values >= 2 * 256 * 4  # [B, Hkv, C] f32
    # partials, (m, l, o[128]) each: estimate pieces (at most one per index
    # tile and KV group, G heads each), steady pieces (2 tiles per KV group, G
    # heads each), retrieval pieces (one per block and query head)
    part = (2 + 128) * 4
    tiles = 2 * (256 // 64)
    assert lay.total - lay.partials >= part * ((tiles + 2) * 4 + 2 * 2 * 4 + lay.max_blocks + 8)


@pytest.mark.parametrize("kw,code", [
    (dict(Hq=7), 1), (dict(Hq=6), 2), (dict(Hq=32, Hkv=2), 2), (dict(r=257), 1), (dict(r=-1), 1),
    (dict(d=96), 2), (dict(sink=5000), 1),
])
def test_decode_param_validation(L, kw, code):
    lib = L.lib()
    assert lib.wi_decode_workspace_bytes(ctypes.byref(dp(L, **kw)), 256) == 0
    ix = L.IndexStruct()
    for name in L.FIELDS:
        setattr(ix, name, 1 << 20)
    ix.B, ix.Hkv, ix.N, ix.d, ix.sink, ix.window, ix.n_clusters = 1, 2, 4096, 128, 4, 64, 256
    fake = ctypes.c_void_p(1 << 20)
    assert lib.wi_decode_attention(ctypes.byref(dp(L, **kw)), fake, fake, fake, ctypes.byref(ix),
                                   fake, None, None, fake, 1 << 30, None) == code


def test_decode_index_mismatch_and_workspace(L):
    lib = L.lib()
    ix = L.IndexStruct()
    for name in L.FIELDS:
        setattr(ix, name, 1 << 20)
    ix.B, ix.Hkv, ix.N, ix.d, ix.sink, ix.window, ix.n_clusters = 1, 2, 4096, 128, 4, 32, 256
    fake = ctypes.c_void_p(1 << 20)
    assert lib.wi_decode_attention(ctypes.byref(dp(L)), fake, fake, fake, ctypes.byref(ix), fake,
                                   None, None, fake, 1 << 30, None) == L.WI_ERR_INDEX_MISMATCH
    ix.window = 64
    assert lib.wi_decode_attention(ctypes.byref(dp(L)), fake, fake, fake, ctypes.byref(ix), fake,
                                   None, None, fake, 64, None) == L.WI_ERR_WORKSPACE
    assert lib.wi_decode_attention(ctypes.byref(dp(L)), fake, fake, fake, ctypes.byref(ix), None,
                                   None, None, fake, 1 << 30, None) == L.WI_ERR_INVALID_ARG
    assert lib.wi_decode_attention(ctypes.byref(dp(L)), fake, fake, fake, ctypes.byref(ix), fake,
                                   None, None, ctypes.c_void_p((1 << 20) + 16), 1 << 30,
                                   None) == L.WI_ERR_ALIGNMENT


def test_decode_option_validation(L):
    # the options are checked before anything else of the call
    lib = L.lib()
    ix = L.IndexStruct()
    for name in L.FIELDS:
        setattr(ix, name, 1 << 20)
    ix.B, ix.Hkv, ix.N, ix.d, ix.sink, ix.window, ix.n_clusters = 1, 2, 4096, 128, 4, 64, 256
    fake = ctypes.c_void_p(1 << 20)

    def call(**kw):
        o = L.DecodeOptions()
        for k, v in kw.items():
            setattr(o, k, v)
        return lib.wi_decode_attention_ex(ctypes.byref(dp(L)), ctypes.byref(o), fake, fake, fake,
                                          ctypes.byref(ix), fake, None, None, fake, 1 << 30, None)

    assert call(rank=2) == L.WI_ERR_INVALID_ARG
    assert call(share=2) == L.WI_ERR_INVALID_ARG
    assert call(rank=-1) == L.WI_ERR_INVALID_ARG
    assert call(prev_q=1 << 20) == L.WI_ERR_INVALID_ARG              # no prev_topk
    assert call(prev_q=1 << 20, prev_topk=1 << 20, tau=float("nan")) == L.WI_ERR_INVALID_ARG
    assert call(prev_q=(1 << 20) + 8, prev_topk=1 << 20) == L.WI_ERR_ALIGNMENT
    assert call(prev_q=1 << 20, prev_topk=(1 << 20) + 2) == L.WI_ERR_ALIGNMENT
    assert call(rank=1, reused=(1 << 20) + 1) == L.WI_ERR_ALIGNMENT
    # valid options reach the remaining checks (here the index mismatch)
    ix.window = 32
    assert call(rank=1, prev_q=1 << 20, prev_topk=1 << 20, tau=0.5) == L.WI_ERR_INDEX_MISMATCH
    assert lib.wi_decode_attention_ex(ctypes.byref(dp(L)), None, fake, fake, fake,
                                      ctypes.byref(ix), fake, None, None, fake, 1 << 30,
                                      None) == L.WI_ERR_INDEX_MISMATCH


def test_index_extend_host_checks(L):
    # shapes must match the earlier index; the context may not shrink; joining
    # positions must stay in segments the earlier index clustered
    lib = L.lib()
    fake = ctypes.c_void_p(1 << 20)

    def ix(N):
        t = L.IndexStruct()
        for name in L.FIELDS:
            setattr(t, name, 1 << 20)
        t.B, t.Hkv, t.N, t.d, t.sink, t.window, t.seg_len, t.k_per_seg = 1, 2, N, 128, 4, 64, 1024, 32
        t.n_clusters = -(-N // 1024) * 32
        return t

    def call(N1, old, **kw):
        p = bp(L, N=N1, seg_len=1024, k_per_seg=32, window=64, **kw)
        new = ix(N1)
        return lib.wi_index_extend(ctypes.byref(p), fake, fake, ctypes.byref(old),
                                   ctypes.byref(new), fake, 1 << 30, None)

    assert call(3000, ix(3100)) == L.WI_ERR_INDEX_MISMATCH     # shrank
    assert call(3000, ix(2900), sink=5) == L.WI_ERR_INDEX_MISMATCH
    assert call(3200, ix(3000)) == L.WI_ERR_UNSUPPORTED        # [2936, 3136) reaches segment 3
    assert call(3000, ix(40)) == L.WI_ERR_UNSUPPORTED          # nothing clustered before
    assert lib.wi_index_extend(ctypes.byref(bp(L)), fake, fake, None, ctypes.byref(ix(3000)),
                               fake, 1 << 30, None) == L.WI_ERR_INVALID_ARG
