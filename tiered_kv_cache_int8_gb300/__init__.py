"""Two-level KV cache for top-k sparse-attention decode on one GB300 (sm_103a).

The path (indexer + top-k, RESOLVE, attention, append) is CUDA in libhs.so,
reached through the C ABI in include/hs.h; ``hs`` is its ctypes binding.
"""
from .hs import HiSparseCache, HsError, lib  # noqa: F401
