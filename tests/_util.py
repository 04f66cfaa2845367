"""Shared test helpers: moving generator arrays and indices between NumPy (the
oracle's side) and torch device tensors (the library's side).  No method
arithmetic lives here."""

import numpy as np
import torch

from oracle import wave_index as wi


def bf16_tensor(bits: np.ndarray, device) -> torch.Tensor:
    """uint16 bf16 bit patterns -> torch.bfloat16 tensor on device (same bits)."""
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16))
    return t.view(torch.bfloat16).to(device)


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def f64(bits: np.ndarray) -> np.ndarray:
    return wi.bf16_bits_to_f64(bits)


def index_to_numpy(ix) -> dict:
    """Download a WaveIndex into the oracle's dict layout (float64 values)."""
    t = ix.tensors
    return {
        "centroid_key": t["centroid_key"].double().cpu().numpy(),
        "unit_centroid": t["unit_centroid"].double().cpu().numpy(),
        "value_sum": t["value_sum"].double().cpu().numpy(),
        "size": t["size"].cpu().numpy().astype(np.int64),
        "offset": t["offset"].cpu().numpy().astype(np.int64),
        "perm": t["perm"].cpu().numpy().astype(np.int64),
        "assign": t["assign"].cpu().numpy().astype(np.int64),
        "k_sorted": t["k_sorted"].double().cpu().numpy(),
        "v_sorted": t["v_sorted"].double().cpu().numpy(),
    }


def upload_oracle_index(ix, oidx: dict, b_h_axes: bool = True) -> None:
    """Fill a WaveIndex's device tensors from an oracle index (leading [B,Hkv]
    axes), so that decode can be tested independently of the GPU build.  The
    wi_index struct's scalar fields are recorded as a build would."""
    t = ix.tensors
    t["centroid_key"].copy_(torch.from_numpy(oidx["centroid_key"].astype(np.float32)))
    t["value_sum"].copy_(torch.from_numpy(oidx["value_sum"].astype(np.float32)))
    t["unit_centroid"].copy_(torch.from_numpy(oidx["unit_centroid"].astype(np.float32)).to(
        torch.bfloat16))
    for name in ("size", "offset", "perm", "assign"):
        t[name].copy_(torch.from_numpy(oidx[name].astype(np.int32)))
    t["k_sorted"].copy_(torch.from_numpy(oidx["k_sorted"].astype(np.float32)).to(torch.bfloat16))
    t["v_sorted"].copy_(torch.from_numpy(oidx["v_sorted"].astype(np.float32)).to(torch.bfloat16))
    c = ix.cfg
    s = ix.struct
    s.B, s.Hkv, s.N, s.d = c.B, c.Hkv, c.N, c.d
    s.sink, s.window, s.seg_len, s.k_per_seg, s.n_clusters = (c.sink, c.window, c.seg_len,
                                                               c.k_per_seg, c.n_clusters)


def head_index(idx: dict, b: int, g: int) -> dict:
    return {k: idx[k][b, g] for k in ("size", "centroid_key", "value_sum", "perm", "offset")}


def sets_match_mod_ties(got, ref, scores, tol):
    """Two index sets agree if every element of their symmetric difference
    scores within tol of the boundary (the reference set's lowest score)."""
    got, ref = set(int(x) for x in got), set(int(x) for x in ref)
    if got == ref:
        return True
    if len(got) != len(ref):
        return False
    boundary = min(scores[c] for c in ref) if ref else -np.inf
    return all(abs(scores[c] - boundary) < tol for c in got ^ ref)


def rel_err(a, b):
    return float(np.max(np.abs(np.asarray(a) - np.asarray(b))) / max(np.max(np.abs(b)), 1e-30))
