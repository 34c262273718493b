"""Tiled, memory-efficient scaled-dot-product attention for GB300 (sm_103a).

The computation runs in hand-written CUDA kernels behind the C ABI of
include/attn.h (libattn.so); this package is a thin ctypes binding plus the
seeded synthetic input recipes.  Importing it does not load the library.
"""
from ._lib import AttnError, attn_bwd, attn_fwd, load, sync_status  # noqa: F401

__all__ = ["attn_fwd", "attn_bwd", "sync_status", "load", "AttnError"]
