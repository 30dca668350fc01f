"""Paged-KV exact attention for GB300 (sm_103a).

A small C-ABI library (``libpa.so``, declared in ``include/pa.h``) with
hand-written CUDA kernels for the KV-cache store (bf16, or FP8 E4M3 with
per-head scales), varlen causal prefill / extend attention over a page table,
split-KV decode and the log-sum-exp combine, and both attention halves of a
mixed batch in one launch; this package is its thin torch binding.  PyTorch
provides device memory and streams only.
"""
from .api import (PA_DEVERR_PAGE_RANGE, PA_DEVERR_POSITION, PA_DEVERR_SEQLENS, PA_DEVERR_TABLE_INDEX,
                  PA_DEVERR_TIMEOUT, PA_KV_BF16, PA_KV_FP8_E4M3, PA_MIXED_SCHEDULER_INTS, PagedAttentionError,
                  abi_version,
                  build_page_table,
                  build_seqlens, decode, decode_noalloc, decode_kv_chunk, decode_workspace_size,
                  device_error, lse_combine, mixed_batch, prefill, prefill_scheduler, rope_cos_sin_table,
                  rope_store_kv, store_kv, store_kv_fp8)

from .graphs import DecodeGraphRunner, bucket_for

__all__ = [
    "PagedAttentionError", "abi_version", "build_page_table", "build_seqlens", "decode",
    "decode_noalloc",
    "decode_kv_chunk", "decode_workspace_size", "device_error", "lse_combine", "mixed_batch", "prefill",
    "prefill_scheduler",
    "DecodeGraphRunner", "bucket_for",
    "store_kv", "store_kv_fp8", "PA_KV_BF16", "PA_KV_FP8_E4M3", "PA_MIXED_SCHEDULER_INTS",
    "rope_cos_sin_table", "rope_store_kv",
    "PA_DEVERR_PAGE_RANGE", "PA_DEVERR_SEQLENS", "PA_DEVERR_TIMEOUT", "PA_DEVERR_POSITION",
    "PA_DEVERR_TABLE_INDEX",
]
