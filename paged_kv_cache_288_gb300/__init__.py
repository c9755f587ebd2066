"""Paged KV-cache attention decode for GB300 (sm_103a).

The compute lives in ``libpa.so`` (hand-written CUDA kernels behind the C ABI
of ``include/pa.h``); this package only marshals torch tensors into those
calls. Build the library with ``python -m paged_kv_cache_288_gb300.build``.
Importing the package does not load the library; the first call does, and
raises if it has not been built.
"""

from ._binding import (
    PaError,
    F16,
    BF16,
    FP8_E4M3,
    DEVERR_SLOT_RANGE,
    DEVERR_BLOCK_RANGE,
    DEVERR_CONTEXT_RANGE,
    DEVERR_TIMEOUT,
    DEVERR_LAYOUT,
    DEVERR_QUERY_START,
    DEVERR_Q_RANGE,
    DEVERR_PREFIX,
    lib,
    library_path,
    reshape_and_cache,
    decode,
    decode_workspace_size,
    decode_split_noalloc,
    decode_shared_prefix,
    decode_shared_prefix_workspace_size,
    prefill,
    copy_blocks,
    swap_blocks,
    SWAP_MAX_LAYERS,
    pointer_array,
)
from .block_pool import BlockPool, OutOfBlocks, PrefixCache, block_key, shared_prefix_groups

__all__ = [
    "PaError", "F16", "BF16", "FP8_E4M3", "DEVERR_SLOT_RANGE", "DEVERR_BLOCK_RANGE",
    "DEVERR_CONTEXT_RANGE", "DEVERR_TIMEOUT", "DEVERR_LAYOUT", "DEVERR_QUERY_START",
    "DEVERR_Q_RANGE", "DEVERR_PREFIX", "lib", "library_path", "reshape_and_cache", "decode",
    "decode_workspace_size", "decode_split_noalloc", "decode_shared_prefix", "decode_shared_prefix_workspace_size", "prefill", "copy_blocks", "swap_blocks", "SWAP_MAX_LAYERS", "pointer_array", "BlockPool", "OutOfBlocks", "PrefixCache", "block_key", "shared_prefix_groups",
]
