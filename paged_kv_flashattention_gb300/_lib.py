"""ctypes loader for libpa.so: argument types of every C-ABI entry point.

The library must have been built (``paged_kv_flashattention_gb300.build``);
there is no other implementation to fall back to, so a missing library is an
ImportError at first use.
"""
from __future__ import annotations

import ctypes
import os
import threading

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libpa.so")

_lock = threading.Lock()
_lib = None

c_p = ctypes.c_void_p
c_i32 = ctypes.c_int32
c_i64 = ctypes.c_int64
c_f32 = ctypes.c_float
c_size = ctypes.c_size_t


class PrefillParams(ctypes.Structure):
    _fields_ = [
        ("q", c_p), ("k_cache", c_p), ("v_cache", c_p),
        ("page_table", c_p), ("page_table_stride", c_i32), ("total_q", c_i32),
        ("cu_seqlens_q", c_p), ("cu_seqlens_k", c_p),
        ("num_seqs", c_i32), ("max_seqlen_q", c_i32), ("max_seqlen_k", c_i32),
        ("num_q_heads", c_i32), ("num_kv_heads", c_i32), ("head_dim", c_i32),
        ("page_size", c_i32), ("num_pages", c_i64), ("causal", c_i32), ("scale", c_f32),
        ("out", c_p), ("lse", c_p), ("lse_stride", c_i64),
        ("kv_dtype", c_i32), ("k_scale", c_p), ("v_scale", c_p), ("sliding_window", c_i32),
        ("max_ctas", c_i32), ("scheduler", c_p), ("block_mask", c_p), ("block_mask_q_blocks", c_i32),
        ("block_mask_k_blocks", c_i32),
    ]


class DecodeParams(ctypes.Structure):
    _fields_ = [
        ("q", c_p), ("k_cache", c_p), ("v_cache", c_p),
        ("page_table", c_p), ("page_table_stride", c_i32),
        ("cache_seqlens", c_p), ("num_seqs", c_i32), ("max_seqlen_k", c_i32),
        ("num_q_heads", c_i32), ("num_kv_heads", c_i32), ("head_dim", c_i32),
        ("page_size", c_i32), ("num_pages", c_i64), ("scale", c_f32),
        ("out", c_p), ("lse", c_p), ("workspace", c_p), ("workspace_bytes", c_size),
        ("kv_chunk", c_i32), ("kv_dtype", c_i32), ("k_scale", c_p), ("v_scale", c_p),
        ("sliding_window", c_i32), ("max_ctas", c_i32), ("overlap_previous", c_i32),
    ]


class RopeStoreParams(ctypes.Structure):
    _fields_ = [
        ("q", c_p), ("q_out", c_p), ("k", c_p), ("v", c_p), ("positions", c_p), ("cos_sin", c_p),
        ("max_pos", c_i32), ("rot_dim", c_i32), ("interleaved", c_i32), ("slot_mapping", c_p),
        ("num_tokens", c_i64), ("num_q_heads", c_i32), ("num_kv_heads", c_i32), ("head_dim", c_i32),
        ("k_cache", c_p), ("v_cache", c_p), ("num_slots", c_i64), ("kv_dtype", c_i32),
        ("k_scale", c_p), ("v_scale", c_p),
    ]


# name -> (restype, argtypes)
SIGNATURES = {
    "pa_abi_version": (ctypes.c_int, []),
    "pa_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "pa_last_error": (ctypes.c_char_p, []),
    "pa_device_error": (ctypes.c_int, [ctypes.POINTER(c_i32), c_p]),
    "pa_store_kv": (ctypes.c_int, [c_p, c_p, c_p, c_i64, c_p, c_p, c_i64, c_i32, c_i32, c_p]),
    "pa_store_kv_fp8": (ctypes.c_int, [c_p, c_p, c_p, c_i64, c_p, c_p, c_i64, c_i32, c_i32, c_p, c_p, c_p]),
    "pa_rope_cos_sin_table": (ctypes.c_int, [c_p, c_i32, c_i32, ctypes.c_double]),
    "pa_rope_store_kv": (ctypes.c_int, [ctypes.POINTER(RopeStoreParams), c_p]),
    "pa_build_seqlens": (ctypes.c_int, [c_p, c_p, c_i32, c_p, c_p, c_p, c_p, c_p]),
    "pa_build_page_table": (ctypes.c_int, [c_p, c_i64, c_i64, c_p, c_i32, c_i32, c_i32, c_p, c_i32, c_p]),
    "pa_prefill": (ctypes.c_int, [ctypes.POINTER(PrefillParams), c_p]),
    "pa_decode_workspace_size": (c_size, [ctypes.POINTER(DecodeParams)]),
    "pa_decode_kv_chunk": (c_i32, [ctypes.POINTER(DecodeParams)]),
    "pa_decode": (ctypes.c_int, [ctypes.POINTER(DecodeParams), c_p]),
    "pa_decode_noalloc": (ctypes.c_int, [ctypes.POINTER(DecodeParams), c_p]),
    "pa_mixed_batch": (ctypes.c_int, [ctypes.POINTER(PrefillParams), ctypes.POINTER(DecodeParams), c_p]),
    "pa_lse_combine": (ctypes.c_int, [c_p, c_p, c_p, c_i32, c_i32, c_i32, c_p, c_p, c_p]),
}


def load(path: str | None = None):
    """Load libpa.so once and bind the signatures.  PA_LIBRARY_PATH selects
    another build of the library (e.g. one compiled with other flags)."""
    global _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        p = path or os.environ.get("PA_LIBRARY_PATH") or LIB_PATH
        if not os.path.exists(p):
            raise ImportError(
                f"libpa.so not found at {p}: build it first "
                "(python -m paged_kv_flashattention_gb300.build); there is no fallback path")
        lib = ctypes.CDLL(p)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        if path is None:
            _lib = lib
        return lib
