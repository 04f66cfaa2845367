"""ctypes view of libwi's C ABI (include/wi.h).  Loading fails loudly when the
library has not been built: there is no fallback implementation."""

from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libwi.so")

WI_OK = 0
WI_ERR_INVALID_ARG = 1
WI_ERR_UNSUPPORTED = 2
WI_ERR_LAUNCH = 3
WI_ERR_INDEX_MISMATCH = 4
WI_ERR_DEVICE_TIMEOUT = 5
WI_ERR_WORKSPACE = 6
WI_ERR_ALIGNMENT = 7
WI_ERR_CUDA = 8

WI_HEAD_DIM = 128
WI_MAX_K_PER_SEG = 512
WI_MAX_SEG_LEN = 16384
WI_MAX_CLUSTERS = 1 << 20
WI_STATIC_SCRATCH_BYTES = 16 << 20

FIELDS = ["centroid_key", "unit_centroid", "value_sum", "size", "offset", "perm", "assign",
          "k_sorted", "v_sorted"]

# C ABI entry points, in header order (tests check the header against this).
SYMBOLS = [
    "wi_index_sizes", "wi_build_workspace_bytes", "wi_build_index", "wi_index_extend",
    "wi_build_init",
    "wi_kmeans_assign", "wi_kmeans_update", "wi_build_finalize", "wi_decode_workspace_bytes",
    "wi_decode_workspace_layout", "wi_decode_attention", "wi_index_round_bf16",
    "wi_decode_attention_ex",
    "wi_decode_score", "wi_decode_select", "wi_decode_attend", "wi_decode_attention_static",
    "wi_decode_static_status", "wi_sync_status", "wi_status_string", "wi_debug_inject",
    "wi_version",
]

WI_RANK_SCORE = 0
WI_RANK_MASS = 1
RANKS = {"score": WI_RANK_SCORE, "mass": WI_RANK_MASS}
WI_SHARE_HEAD = 0
WI_SHARE_GROUP = 1
SHARES = {"head": WI_SHARE_HEAD, "group": WI_SHARE_GROUP}


class DecodeOptions(ctypes.Structure):
    _fields_ = [("rank", ctypes.c_int), ("tau", ctypes.c_float), ("prev_q", ctypes.c_void_p),
                ("prev_topk", ctypes.c_void_p), ("reused", ctypes.c_void_p),
                ("share", ctypes.c_int), ("centroid_key_bf16", ctypes.c_void_p),
                ("value_sum_bf16", ctypes.c_void_p)]


class BuildParams(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in
                ("B", "Hkv", "N", "d", "sink", "window", "seg_len", "k_per_seg", "iters")]


class DecodeParams(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in ("B", "Hq", "Hkv", "N", "d", "sink", "window", "r")] + [
        ("scale", ctypes.c_float)]


class IndexStruct(ctypes.Structure):
    _fields_ = [
        ("centroid_key", ctypes.c_void_p),
        ("unit_centroid", ctypes.c_void_p),
        ("value_sum", ctypes.c_void_p),
        ("size", ctypes.c_void_p),
        ("offset", ctypes.c_void_p),
        ("perm", ctypes.c_void_p),
        ("assign", ctypes.c_void_p),
        ("k_sorted", ctypes.c_void_p),
        ("v_sorted", ctypes.c_void_p),
    ] + [(n, ctypes.c_int) for n in
         ("B", "Hkv", "N", "d", "sink", "window", "seg_len", "k_per_seg", "n_clusters")]


class DecodeLayout(ctypes.Structure):
    _fields_ = [(n, ctypes.c_size_t) for n in
                ("counters", "scores", "head_max", "selected", "sel_rows", "sel_counts",
                 "sel_prefix", "sel_scores", "head_tokens", "group_values", "partials",
                 "total")] + [
        (n, ctypes.c_int) for n in ("counter_bytes", "max_blocks", "reserved0", "reserved1")]


_lib = None


def lib() -> ctypes.CDLL:
    """The loaded libwi.so (raises if it is missing)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            "libwi.so is not built (%s); run `python -m cluster_indexed_sparse_wi_b300.build_lib`"
            % LIB_PATH)
    L = ctypes.CDLL(LIB_PATH)
    P = ctypes.POINTER
    vp, sz, i = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int
    bp, dp, ip = P(BuildParams), P(DecodeParams), P(IndexStruct)
    sig = {
        "wi_index_sizes": (i, [bp, P(sz)]),
        "wi_build_workspace_bytes": (sz, [bp]),
        "wi_build_index": (i, [bp, vp, vp, ip, vp, sz, vp]),
        "wi_index_extend": (i, [bp, vp, vp, ip, ip, vp, sz, vp]),
        "wi_build_init": (i, [bp, vp, ip, vp, sz, vp]),
        "wi_kmeans_assign": (i, [bp, vp, ip, vp, sz, vp]),
        "wi_kmeans_update": (i, [bp, vp, ip, vp, sz, vp]),
        "wi_build_finalize": (i, [bp, vp, vp, ip, vp, sz, vp]),
        "wi_decode_workspace_bytes": (sz, [dp, i]),
        "wi_decode_workspace_layout": (i, [dp, i, P(DecodeLayout)]),
        "wi_decode_attention": (i, [dp, vp, vp, vp, ip, vp, vp, vp, vp, sz, vp]),
        "wi_index_round_bf16": (i, [ip, vp, vp, vp]),
        "wi_decode_attention_ex": (i, [dp, P(DecodeOptions), vp, vp, vp, ip, vp, vp, vp, vp,
                                       sz, vp]),
        "wi_decode_score": (i, [dp, vp, ip, vp, sz, vp]),
        "wi_decode_select": (i, [dp, ip, vp, vp, sz, vp]),
        "wi_decode_attend": (i, [dp, vp, vp, vp, ip, vp, vp, vp, sz, vp]),
        "wi_decode_attention_static": (i, [dp, vp, vp, vp, ip, vp, vp, vp, vp]),
        "wi_decode_static_status": (i, [vp, P(i)]),
        "wi_sync_status": (i, [vp, vp, P(i)]),
        "wi_status_string": (ctypes.c_char_p, [i]),
        "wi_debug_inject": (i, [i]),
        "wi_version": (ctypes.c_char_p, []),
    }
    for name, (res, args) in sig.items():
        fn = getattr(L, name)
        fn.restype = res
        fn.argtypes = args
    _lib = L
    return L


class WIError(RuntimeError):
    def __init__(self, status: int, where: str = ""):
        self.status = status
        msg = lib().wi_status_string(status).decode()
        super().__init__("%s: libwi status %d (%s)" % (where or "libwi", status, msg))


def check(status: int, where: str = "") -> None:
    if status != WI_OK:
        raise WIError(status, where)
