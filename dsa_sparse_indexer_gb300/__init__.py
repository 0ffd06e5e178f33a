"""DCP sparse-indexer hot path for GB300 (sm_103a).

The path (PR #46076 report, "[Attention][DSA] support dcp for
FLASHINFER_MLA_SPARSE"): every shard's local top-K of fp32 indexer logits,
(score, global id) candidate packing into one [rows, S*K, 2] buffer, a stable
merge into the global top-K, conversion of the global ids to each shard's paged
KV slots with compaction, and the LSE combine of the shards' partial attention
outputs.  All compute runs in hand-written CUDA kernels behind the C ABI in
include/dsa.h (libdsa.so); this package only marshals torch tensors to it.
"""
from . import _lib
from .ops import (SUPPORTED_K, convert_index_compact, fused_norm_rope, indexer_fused,
                  indexer_logits, kv_cache_insert, lse_combine, merge_topk_stable,
                  new_error_flags, pack_candidates, shard_topk, shard_topk_pack, slot_mapping,
                  sparse_mla_decode)
from ._lib import DSAError, DSA_FLAG_BOUNDS, DSA_FLAG_TIMEOUT

__all__ = ["shard_topk", "pack_candidates", "shard_topk_pack", "merge_topk_stable",
           "convert_index_compact", "indexer_fused", "lse_combine", "slot_mapping",
           "sparse_mla_decode", "indexer_logits", "fused_norm_rope", "kv_cache_insert",
           "new_error_flags", "DSAError",
           "DSA_FLAG_BOUNDS", "DSA_FLAG_TIMEOUT", "SUPPORTED_K", "library"]


def library():
    """The loaded libdsa.so (ctypes handle); raises if it has not been built."""
    return _lib.load()
