"""GB300-native hot path of context-parallel attention (Ring, Ring Anything,
Ulysses, Ulysses Anything, Unified) on one GPU: hand-written sm_103a CUDA kernels behind the C ABI in
include/cpattn.h, with this thin PyTorch binding on top.

The shared library is loaded on first use and must exist (built by
``__graft_entry__.build()``); there is no CPU fallback.
"""
from .api import (CpattnError, grouped_as_bhsd, last_device_status, merge, partial,
                  prepare_ring, prepare_ulysses_anything, prepare_unified, ring,
                  ring_noalloc, ring_noalloc_max_workspace_bytes, ring_workspace_bytes,
                  set_wait_timeout_ns, ulysses_anything_attention, ulysses_anything_permute,
                  ulysses_anything_permute_batch, ulysses_attention, ulysses_permute,
                  ulysses_permute_batch, unified_attention)
from ._lib import EXPORTS, LIB_PATH, load as load_library

__all__ = ["partial", "merge", "ring", "ring_workspace_bytes", "ring_noalloc", "prepare_ring",
           "prepare_unified", "prepare_ulysses_anything",
           "ring_noalloc_max_workspace_bytes", "ulysses_permute", "unified_attention",
           "ulysses_attention", "ulysses_anything_permute", "ulysses_anything_attention",
           "ulysses_permute_batch", "ulysses_anything_permute_batch",
           "grouped_as_bhsd", "last_device_status", "set_wait_timeout_ns",
           "CpattnError", "EXPORTS", "LIB_PATH", "load_library"]
