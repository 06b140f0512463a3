"""GB300-native paged KV insert (RoPE + MXFP8) and dequant-gather.

The compute runs in libgkr.so (hand-written sm_103a CUDA kernels behind a C ABI,
declared in include/gkr.h); this package builds it in-tree and binds it with
ctypes.  PyTorch supplies device memory and streams only.

    kv_insert(kv, k_cache, slot_mapping, positions, cos_sin_cache, block_size, record,
              fp8_scale=None)
    kv_gather(k_cache, indices, out, fp8_scale=None)
    rope_quant_insert(kv, k_cache, slot_mapping, positions, cos_sin_cache, block_size,
                      compress_ratio, sanitize_nans)
    qnorm_rope_kv_insert(q, kv, k_cache, slot_mapping, positions, cos_sin_cache,
                         num_heads_padded, eps, block_size, apply_q_norm)
    sparse_logits(q, k_cache, indices, sm_scale)

Every call takes launch_opts=LaunchOpts(...); `with launch_policy(...)` sets them for
the calls of the current thread (context).
"""
from .build import build as _build_lib
from ._binding import (CacheDesc, ERR_INDEX, ERR_POS, ERR_SCALE, ERR_SLOT, ERR_TIMEOUT, GkrError,
                       LaunchOpts,
                       PACKED, RECORDS, alloc_cache, cache_bytes, get_early_metadata,
                       get_insert_staged_min, get_insert_stream_min, get_pdl,
                       insert_kernel_for, kv_gather, kv_insert, launch_policy, lib,
                       library_path, page_stride, qnorm_rope_kv_insert, record_rows,
                       rope_quant_insert, set_early_metadata, set_insert_staged_min,
                       set_insert_stream_min, set_pdl, sparse_logits, status_string)

__all__ = ["build", "kv_insert", "kv_gather", "rope_quant_insert", "qnorm_rope_kv_insert",
           "sparse_logits", "ERR_TIMEOUT",
           "LaunchOpts", "launch_policy", "page_stride", "record_rows",
           "alloc_cache", "cache_bytes", "status_string", "set_pdl", "get_pdl",
           "set_early_metadata", "get_early_metadata", "set_insert_stream_min",
           "get_insert_stream_min", "set_insert_staged_min", "get_insert_staged_min",
           "insert_kernel_for", "GkrError", "CacheDesc", "RECORDS", "PACKED", "ERR_SLOT",
           "ERR_POS", "ERR_INDEX", "ERR_SCALE", "lib", "library_path"]


def build(force: bool = False):
    """Compile libgkr.so for sm_103a in-tree (skipped when up to date)."""
    return _build_lib(force=force)
