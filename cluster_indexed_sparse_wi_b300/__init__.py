"""Wave-index tripartite decode attention and its segmented spherical-k-means
index build for one NVIDIA B300 (sm_103a), as a C-ABI library (libwi.so,
declared in include/wi.h) with a thin PyTorch binding.

Method: "RetroInfer: A Vector Storage Engine for Scalable Long-Context LLM
Inference" (technical summary §2.A wave index, §3 segmented clustering).
"""

from . import _lib  # noqa: F401
from .api import (  # noqa: F401
    DecodeStep,
    Decoder,
    capture_graph,
    IndexConfig,
    WaveIndex,
    build_index,
    build_workspace_bytes,
    decode_attention,
    index_sizes,
    sync_status,
)
from ._lib import WIError, lib  # noqa: F401

__version__ = "0.1.0"
