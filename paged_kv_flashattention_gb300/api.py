"""Thin torch binding of the C ABI (argument marshalling only).

Every function checks dtypes, devices and contiguity, passes raw pointers and
the current CUDA stream to libpa, and raises ``PagedAttentionError`` on a
non-zero status.  No arithmetic of the attention path happens here.
"""
from __future__ import annotations

import ctypes
import math
import threading

import numpy as np
import torch

from . import _lib

PA_OK = 0


class PagedAttentionError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(message)
        self.status = status


def _check(status: int, lib=None):
    if status != PA_OK:
        lib = lib or _lib.load()
        msg = lib.pa_last_error().decode(errors="replace")
        name = lib.pa_status_string(status).decode()
        raise PagedAttentionError(status, f"{name}: {msg}")


def _stream(t: torch.Tensor | None = None) -> int:
    dev = t.device if t is not None else None
    return torch.cuda.current_stream(dev).cuda_stream


def _ptr(t: torch.Tensor | None) -> int | None:
    return None if t is None else t.data_ptr()


def _need(t: torch.Tensor, name: str, dtype, device=None, contiguous=True):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if device is not None and t.device != device:
        raise ValueError(f"{name} must be on {device}, got {t.device}")
    if contiguous and not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


PA_KV_BF16, PA_KV_FP8_E4M3 = 0, 1
_FP8_DTYPES = (torch.uint8,) + ((torch.float8_e4m3fn,) if hasattr(torch, "float8_e4m3fn") else ())


def _kv_dtype(k_cache: torch.Tensor, v_cache: torch.Tensor) -> int:
    """PA_KV_BF16 for bf16 pools, PA_KV_FP8_E4M3 for E4M3 codes (uint8 or
    torch.float8_e4m3fn)."""
    if k_cache.dtype != v_cache.dtype:
        raise TypeError("k_cache and v_cache dtypes differ")
    if k_cache.dtype == torch.bfloat16:
        return PA_KV_BF16
    if k_cache.dtype in _FP8_DTYPES:
        return PA_KV_FP8_E4M3
    raise TypeError(f"pools must be bf16 or E4M3 (uint8 / float8_e4m3fn), got {k_cache.dtype}")


def _need_scales(k_scale, v_scale, Hkv: int, dev):
    for t, n in ((k_scale, "k_scale"), (v_scale, "v_scale")):
        if t is None:
            raise ValueError(f"{n} is required for FP8 pools")
        _need(t, n, torch.float32, dev)
        if t.numel() != Hkv:
            raise ValueError(f"{n} must hold one scale per KV head ({Hkv})")


def abi_version() -> int:
    return int(_lib.load().pa_abi_version())


# Device error bits (include/pa.h, PA_DEVERR_*).
PA_DEVERR_PAGE_RANGE = 1
PA_DEVERR_SEQLENS = 2
PA_DEVERR_TIMEOUT = 4
PA_DEVERR_POSITION = 8
PA_DEVERR_TABLE_INDEX = 16


def device_error() -> int:
    """Read and clear the device error word (synchronises the current stream).

    A launch whose bounded wait gave up (PA_DEVERR_TIMEOUT) may leave its
    scheduler counters non-zero, and the next launch sharing the array would
    skip work items: the scheduler arrays cached by ``prefill_scheduler``
    are cleared then (after the device has drained)."""
    lib = _lib.load()
    bits = ctypes.c_int32(0)
    _check(lib.pa_device_error(ctypes.byref(bits), _stream()), lib)
    if bits.value & PA_DEVERR_TIMEOUT:
        _reset_schedulers()
    return int(bits.value)


def store_kv(k: torch.Tensor, v: torch.Tensor, slot_mapping: torch.Tensor,
             k_cache: torch.Tensor, v_cache: torch.Tensor) -> None:
    """Write token t's K/V rows into row slot_mapping[t] of the pools.
    k, v: bf16 [T, Hkv, d]; caches: bf16 [num_pages, page_size, Hkv, d] or
    [num_slots, Hkv, d]; slot_mapping: int32 [T] (negative = skip)."""
    dev = k_cache.device
    for t, n in ((k, "k"), (v, "v"), (k_cache, "k_cache"), (v_cache, "v_cache")):
        _need(t, n, torch.bfloat16, dev)
    _need(slot_mapping, "slot_mapping", torch.int32, dev)
    Hkv, d = k_cache.shape[-2], k_cache.shape[-1]
    T = slot_mapping.numel()
    if k.numel() != T * Hkv * d or v.numel() != T * Hkv * d:
        raise ValueError("k/v must hold num_tokens rows of Hkv*d")
    if v_cache.shape != k_cache.shape:
        raise ValueError("k_cache and v_cache shapes differ")
    num_slots = k_cache.numel() // (Hkv * d)
    lib = _lib.load()
    _check(lib.pa_store_kv(_ptr(k), _ptr(v), _ptr(slot_mapping), T, _ptr(k_cache), _ptr(v_cache),
                           num_slots, Hkv, d, _stream(k_cache)), lib)


def store_kv_fp8(k: torch.Tensor, v: torch.Tensor, slot_mapping: torch.Tensor,
                 k_cache: torch.Tensor, v_cache: torch.Tensor, k_scale: torch.Tensor,
                 v_scale: torch.Tensor) -> None:
    """Write token t's K/V rows into row slot_mapping[t] of E4M3 pools:
    code = E4M3(x / scale[kv head]).  k, v: bf16 [T, Hkv, d]; caches: uint8
    or float8_e4m3fn [num_pages, page_size, Hkv, d] or [num_slots, Hkv, d];
    k_scale, v_scale: fp32 [Hkv]."""
    dev = k_cache.device
    for t, n in ((k, "k"), (v, "v")):
        _need(t, n, torch.bfloat16, dev)
    if _kv_dtype(k_cache, v_cache) != PA_KV_FP8_E4M3:
        raise TypeError("store_kv_fp8 needs E4M3 pools")
    for t, n in ((k_cache, "k_cache"), (v_cache, "v_cache")):
        _need(t, n, k_cache.dtype, dev)
    _need(slot_mapping, "slot_mapping", torch.int32, dev)
    Hkv, d = k_cache.shape[-2], k_cache.shape[-1]
    _need_scales(k_scale, v_scale, Hkv, dev)
    T = slot_mapping.numel()
    if k.numel() != T * Hkv * d or v.numel() != T * Hkv * d:
        raise ValueError("k/v must hold num_tokens rows of Hkv*d")
    if v_cache.shape != k_cache.shape:
        raise ValueError("k_cache and v_cache shapes differ")
    num_slots = k_cache.numel() // (Hkv * d)
    lib = _lib.load()
    _check(lib.pa_store_kv_fp8(_ptr(k), _ptr(v), _ptr(slot_mapping), T, _ptr(k_cache), _ptr(v_cache),
                               num_slots, Hkv, d, _ptr(k_scale), _ptr(v_scale), _stream(k_cache)), lib)


def rope_cos_sin_table(max_pos: int, rot_dim: int, base: float = 10000.0) -> torch.Tensor:
    """Host fp32 [max_pos, rot_dim] rotary table (cos of the rot_dim/2 angles
    p * base^(-2i/rot_dim), then their sin), computed by the C library."""
    t = torch.empty((int(max_pos), int(rot_dim)), dtype=torch.float32)
    lib = _lib.load()
    _check(lib.pa_rope_cos_sin_table(t.data_ptr() if t.numel() else None, int(max_pos), int(rot_dim),
                                     float(base)), lib)
    return t


def rope_store_kv(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, positions: torch.Tensor,
                  cos_sin: torch.Tensor, slot_mapping: torch.Tensor, k_cache: torch.Tensor,
                  v_cache: torch.Tensor, *, q_out: torch.Tensor | None = None,
                  interleaved: bool = False, k_scale: torch.Tensor | None = None,
                  v_scale: torch.Tensor | None = None) -> torch.Tensor:
    """Rotary embedding of q and k at ``positions`` fused with the K/V store.
    q bf16 [T, Hq, d]; k, v bf16 [T, Hkv, d]; cos_sin fp32 [max_pos, rot_dim]
    on the device; pools bf16 or E4M3 (with ``k_scale``/``v_scale``).  Returns
    the rotated q (``q_out``, which may be ``q``)."""
    dev = q.device
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _need(t, n, torch.bfloat16, dev)
    _need(positions, "positions", torch.int32, dev)
    _need(slot_mapping, "slot_mapping", torch.int32, dev)
    _need(cos_sin, "cos_sin", torch.float32, dev)
    kvd = _kv_dtype(k_cache, v_cache)
    for t, n in ((k_cache, "k_cache"), (v_cache, "v_cache")):
        _need(t, n, k_cache.dtype, dev)
    T, Hq, d = q.shape
    Hkv = k_cache.shape[-2]
    if k_cache.shape[-1] != d or k.numel() != T * Hkv * d or v.numel() != T * Hkv * d:
        raise ValueError("k/v/pool shapes do not match q")
    if positions.numel() != T or slot_mapping.numel() != T:
        raise ValueError("positions and slot_mapping must hold one entry per token")
    if kvd == PA_KV_FP8_E4M3:
        _need_scales(k_scale, v_scale, Hkv, dev)
    if q_out is None:
        q_out = torch.empty_like(q)
    _need(q_out, "q_out", torch.bfloat16, dev)
    p = _lib.RopeStoreParams(
        q=_ptr(q), q_out=_ptr(q_out), k=_ptr(k), v=_ptr(v), positions=_ptr(positions),
        cos_sin=_ptr(cos_sin), max_pos=cos_sin.shape[0], rot_dim=cos_sin.shape[1],
        interleaved=int(bool(interleaved)), slot_mapping=_ptr(slot_mapping), num_tokens=T,
        num_q_heads=Hq, num_kv_heads=Hkv, head_dim=d, k_cache=_ptr(k_cache), v_cache=_ptr(v_cache),
        num_slots=k_cache.numel() // (Hkv * d), kv_dtype=kvd,
        k_scale=_ptr(k_scale) if kvd == PA_KV_FP8_E4M3 else None,
        v_scale=_ptr(v_scale) if kvd == PA_KV_FP8_E4M3 else None)
    lib = _lib.load()
    _check(lib.pa_rope_store_kv(ctypes.byref(p), _stream(q)), lib)
    return q_out


def build_seqlens(cached_len, extend_len):
    """Host metadata: (cu_seqlens_q, cu_seqlens_k, cache_seqlens, max_q, max_k)
    as int32 numpy arrays (the C entry point does the arithmetic)."""
    c = np.ascontiguousarray(cached_len, dtype=np.int32)
    e = np.ascontiguousarray(extend_len, dtype=np.int32)
    B = c.shape[0]
    cu_q = np.zeros(B + 1, np.int32)
    cu_k = np.zeros(B + 1, np.int32)
    cs = np.zeros(max(B, 1), np.int32)
    mq = ctypes.c_int32(0)
    mk = ctypes.c_int32(0)
    lib = _lib.load()
    _check(lib.pa_build_seqlens(c.ctypes.data, e.ctypes.data, B, cu_q.ctypes.data,
                                cu_k.ctypes.data, cs.ctypes.data, ctypes.byref(mq),
                                ctypes.byref(mk)), lib)
    return cu_q, cu_k, cs[:B], int(mq.value), int(mk.value)


def build_page_table(token_table: torch.Tensor, table_idx: torch.Tensor, max_seqlen_k: int,
                     page_size: int, out: torch.Tensor | None = None) -> torch.Tensor:
    """Device metadata: page table [B, ceil(max_seqlen_k / page_size)] from the
    token-granular global table (sliced with step page_size, floor-divided)."""
    dev = token_table.device
    _need(token_table, "token_table", torch.int32, dev)
    _need(table_idx, "table_idx", torch.int32, dev)
    B = table_idx.numel()
    ncols = -(-int(max_seqlen_k) // int(page_size))
    if token_table.dim() != 2 or token_table.stride(1) != 1:
        raise ValueError("token_table must be 2-D with unit column stride")
    if out is None:
        out = torch.empty((B, max(ncols, 1)), dtype=torch.int32, device=dev)
    _need(out, "out", torch.int32, dev, contiguous=False)
    if out.dim() != 2 or out.stride(1) != 1 or out.shape[0] < B or out.shape[1] < ncols:
        raise ValueError(f"out must be 2-D with unit column stride and at least [{B}, {ncols}]")
    lib = _lib.load()
    _check(lib.pa_build_page_table(_ptr(token_table), token_table.stride(0), token_table.shape[0],
                                   _ptr(table_idx), B,
                                   int(max_seqlen_k), int(page_size), _ptr(out), out.stride(0),
                                   _stream(token_table)), lib)
    return out


def _pool_geometry(k_cache: torch.Tensor, v_cache: torch.Tensor, page_size: int | None):
    if v_cache.shape != k_cache.shape:
        raise ValueError("k_cache and v_cache shapes differ")
    if k_cache.dim() == 4:
        num_pages, P, Hkv, d = k_cache.shape
        if page_size is not None and page_size != P:
            raise ValueError("page_size does not match the pool shape")
    elif k_cache.dim() == 3:
        if page_size is None:
            raise ValueError("page_size is required for a [slots, Hkv, d] pool")
        slots, Hkv, d = k_cache.shape
        P = page_size
        num_pages = slots // P
    else:
        raise ValueError("pool must be [pages, page_size, Hkv, d] or [slots, Hkv, d]")
    return int(num_pages), int(P), int(Hkv), int(d)


# Zeroed scheduler arrays of pa_prefill, one per (device, stream): launches on
# one stream run one after the other, so they can share one array (each
# launch leaves it at zero); launches on different streams get their own.
_sched_lock = threading.Lock()
_sched_arrays: dict = {}
PA_PREFILL_SCHEDULER_INTS = 2
PA_MIXED_SCHEDULER_INTS = 4


def _reset_schedulers() -> None:
    """Zero every cached scheduler array once the work in flight has ended."""
    with _sched_lock:
        arrays = list(_sched_arrays.values())
    for t in arrays:
        if t.is_cuda:
            torch.cuda.synchronize(t.device)
        t.zero_()
        if t.is_cuda:
            torch.cuda.synchronize(t.device)


def prefill_scheduler(device=None, stream=None) -> torch.Tensor:
    """The cached zeroed int32 [4] scheduler array for (device, stream):
    the default of ``prefill(scheduler=None)`` and ``mixed_batch``.  Create
    it before capturing a CUDA graph that calls either on that stream."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    if stream is None:
        stream = torch.cuda.current_stream(dev)
    key = (dev.index, int(stream.cuda_stream))
    with _sched_lock:
        t = _sched_arrays.get(key)
        if t is None:
            t = torch.zeros(PA_MIXED_SCHEDULER_INTS, dtype=torch.int32, device=dev)
            _sched_arrays[key] = t
        return t


def prefill(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor, page_table: torch.Tensor,
            cu_seqlens_q: torch.Tensor, cu_seqlens_k: torch.Tensor, max_seqlen_q: int,
            max_seqlen_k: int, *, causal: bool = True, scale: float | None = None,
            page_size: int | None = None, out: torch.Tensor | None = None,
            lse: torch.Tensor | None = None, k_scale: torch.Tensor | None = None,
            v_scale: torch.Tensor | None = None, sliding_window: int = 0,
            max_ctas: int = 0, scheduler: torch.Tensor | None = None,
            block_mask: torch.Tensor | None = None) -> torch.Tensor:
    """Varlen prefill / extend attention.  q: bf16 [total_q, Hq, d];
    returns out bf16 [total_q, Hq, d]; lse (optional) fp32 [Hq, total_q].
    Pools are bf16, or E4M3 codes (uint8 / float8_e4m3fn) with fp32
    per-KV-head ``k_scale`` and ``v_scale``.  ``scheduler`` is the int32 [2]
    work-counter array of the launch (zero between launches); by default the
    array cached for the current stream (``prefill_scheduler``).
    ``block_mask``: optional uint8 [B, nq, nk] on the device; entry
    [b, i // 128, j // 128] == 0 hides key j from request b's query row i
    (rows counted from the request's first row)."""
    p, out = _prefill_params(q, k_cache, v_cache, page_table, cu_seqlens_q, cu_seqlens_k, max_seqlen_q,
                             max_seqlen_k, causal, scale, page_size, out, lse, k_scale, v_scale, sliding_window,
                             max_ctas, scheduler, block_mask, PA_PREFILL_SCHEDULER_INTS)
    lib = _lib.load()
    _check(lib.pa_prefill(ctypes.byref(p), _stream(q)), lib)
    return out


def _prefill_params(q, k_cache, v_cache, page_table, cu_seqlens_q, cu_seqlens_k, max_seqlen_q, max_seqlen_k,
                    causal, scale, page_size, out, lse, k_scale, v_scale, sliding_window, max_ctas, scheduler,
                    block_mask, sched_ints):
    dev = q.device
    num_pages, P, Hkv, d = _pool_geometry(k_cache, v_cache, page_size)
    _need(q, "q", torch.bfloat16, dev)
    kvd = _kv_dtype(k_cache, v_cache)
    for t, n in ((k_cache, "k_cache"), (v_cache, "v_cache")):
        _need(t, n, k_cache.dtype, dev)
    if kvd == PA_KV_FP8_E4M3:
        _need_scales(k_scale, v_scale, Hkv, dev)
    for t, n in ((page_table, "page_table"), (cu_seqlens_q, "cu_seqlens_q"), (cu_seqlens_k, "cu_seqlens_k")):
        _need(t, n, torch.int32, dev, contiguous=(n != "page_table"))
    if page_table.dim() != 2 or page_table.stride(1) != 1:
        raise ValueError("page_table must be 2-D with unit column stride")
    total_q, Hq, dq = q.shape
    if dq != d:
        raise ValueError("head_dim of q and the pool differ")
    if out is None:
        out = torch.empty_like(q)
    _need(out, "out", torch.bfloat16, dev)
    if lse is not None:
        _need(lse, "lse", torch.float32, dev, contiguous=False)
        if lse.dim() != 2 or lse.shape[0] != Hq or lse.stride(1) != 1:
            raise ValueError("lse must be [Hq, >= total_q] with unit inner stride")
    if block_mask is not None:
        _need(block_mask, "block_mask", torch.uint8, dev)
        if block_mask.dim() != 3 or block_mask.shape[0] != cu_seqlens_q.numel() - 1:
            raise ValueError("block_mask must be [num_seqs, q_blocks, k_blocks]")
    if scheduler is None:
        scheduler = prefill_scheduler(dev)
    _need(scheduler, "scheduler", torch.int32, dev)
    if scheduler.numel() < sched_ints:
        raise ValueError(f"scheduler must hold {sched_ints} int32")
    p = _lib.PrefillParams(
        q=_ptr(q), k_cache=_ptr(k_cache), v_cache=_ptr(v_cache), page_table=_ptr(page_table),
        page_table_stride=page_table.stride(0), total_q=total_q, cu_seqlens_q=_ptr(cu_seqlens_q),
        cu_seqlens_k=_ptr(cu_seqlens_k), num_seqs=cu_seqlens_q.numel() - 1,
        max_seqlen_q=int(max_seqlen_q), max_seqlen_k=int(max_seqlen_k), num_q_heads=Hq,
        num_kv_heads=Hkv, head_dim=d, page_size=P, num_pages=num_pages, causal=int(bool(causal)),
        scale=float(1.0 / math.sqrt(d) if scale is None else scale), out=_ptr(out),
        lse=_ptr(lse), lse_stride=(lse.stride(0) if lse is not None else 0), kv_dtype=kvd,
        k_scale=_ptr(k_scale) if kvd == PA_KV_FP8_E4M3 else None,
        v_scale=_ptr(v_scale) if kvd == PA_KV_FP8_E4M3 else None, sliding_window=int(sliding_window),
        max_ctas=int(max_ctas), scheduler=_ptr(scheduler), block_mask=_ptr(block_mask),
        block_mask_q_blocks=int(block_mask.shape[1]) if block_mask is not None else 0,
        block_mask_k_blocks=int(block_mask.shape[2]) if block_mask is not None else 0)
    return p, out


def _decode_params(q, k_cache, v_cache, page_table, cache_seqlens, max_seqlen_k, scale, page_size,
                   out, lse, workspace, kv_chunk, k_scale=None, v_scale=None, sliding_window=0,
                   max_ctas=0, overlap_previous=False):
    num_pages, P, Hkv, d = _pool_geometry(k_cache, v_cache, page_size)
    B, Hq, dq = q.shape
    if dq != d:
        raise ValueError("head_dim of q and the pool differ")
    kvd = _kv_dtype(k_cache, v_cache)
    if kvd == PA_KV_FP8_E4M3:
        _need_scales(k_scale, v_scale, Hkv, q.device)
    return _lib.DecodeParams(
        q=_ptr(q), k_cache=_ptr(k_cache), v_cache=_ptr(v_cache), page_table=_ptr(page_table),
        page_table_stride=page_table.stride(0) if page_table is not None else 0,
        cache_seqlens=_ptr(cache_seqlens), num_seqs=B, max_seqlen_k=int(max_seqlen_k),
        num_q_heads=Hq, num_kv_heads=Hkv, head_dim=d, page_size=P, num_pages=num_pages,
        scale=float(1.0 / math.sqrt(d) if scale is None else scale), out=_ptr(out), lse=_ptr(lse),
        workspace=_ptr(workspace), workspace_bytes=(workspace.numel() * workspace.element_size()
                                                    if workspace is not None else 0),
        kv_chunk=int(kv_chunk), kv_dtype=kvd,
        k_scale=_ptr(k_scale) if kvd == PA_KV_FP8_E4M3 else None,
        v_scale=_ptr(v_scale) if kvd == PA_KV_FP8_E4M3 else None, sliding_window=int(sliding_window),
        max_ctas=int(max_ctas), overlap_previous=int(bool(overlap_previous)))


def decode_workspace_size(q_shape, k_cache: torch.Tensor, max_seqlen_k: int, *,
                          page_size: int | None = None, kv_chunk: int = 0) -> int:
    """Workspace bytes pa_decode needs (0 when a single split suffices)."""
    B, Hq, d = q_shape
    num_pages, P, Hkv, dk = _pool_geometry(k_cache, k_cache, page_size)
    p = _lib.DecodeParams(num_seqs=B, max_seqlen_k=int(max_seqlen_k), num_q_heads=Hq,
                          num_kv_heads=Hkv, head_dim=d, page_size=P, num_pages=num_pages,
                          scale=1.0, kv_chunk=int(kv_chunk))
    return int(_lib.load().pa_decode_workspace_size(ctypes.byref(p)))


def decode_kv_chunk(q_shape, k_cache: torch.Tensor, max_seqlen_k: int, *,
                    page_size: int | None = None, kv_chunk: int = 0) -> int:
    B, Hq, d = q_shape
    num_pages, P, Hkv, dk = _pool_geometry(k_cache, k_cache, page_size)
    p = _lib.DecodeParams(num_seqs=B, max_seqlen_k=int(max_seqlen_k), num_q_heads=Hq,
                          num_kv_heads=Hkv, head_dim=d, page_size=P, num_pages=num_pages,
                          scale=1.0, kv_chunk=int(kv_chunk))
    return int(_lib.load().pa_decode_kv_chunk(ctypes.byref(p)))


def decode(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor, page_table: torch.Tensor,
           cache_seqlens: torch.Tensor, max_seqlen_k: int, *, scale: float | None = None,
           page_size: int | None = None, out: torch.Tensor | None = None,
           lse: torch.Tensor | None = None, workspace: torch.Tensor | None = None,
           kv_chunk: int = 0, k_scale: torch.Tensor | None = None,
           v_scale: torch.Tensor | None = None, sliding_window: int = 0,
           max_ctas: int = 0, overlap_previous: bool = False) -> torch.Tensor:
    """Split-KV decode: q bf16 [B, Hq, d] -> out bf16 [B, Hq, d]; lse fp32 [B, Hq].
    Pools are bf16, or E4M3 codes (uint8 / float8_e4m3fn) with fp32 per-KV-head
    ``k_scale`` and ``v_scale``.  ``workspace`` (a uint8 CUDA tensor) is
    allocated here when not given."""
    dev = q.device
    _need(q, "q", torch.bfloat16, dev)
    kvd = _kv_dtype(k_cache, v_cache)
    for t, n in ((k_cache, "k_cache"), (v_cache, "v_cache")):
        _need(t, n, k_cache.dtype, dev)
    _need(cache_seqlens, "cache_seqlens", torch.int32, dev)
    _need(page_table, "page_table", torch.int32, dev, contiguous=False)
    if page_table.dim() != 2 or page_table.stride(1) != 1:
        raise ValueError("page_table must be 2-D with unit column stride")
    if out is None:
        out = torch.empty_like(q)
    _need(out, "out", torch.bfloat16, dev)
    if lse is not None:
        _need(lse, "lse", torch.float32, dev)
    need = decode_workspace_size(q.shape, k_cache, max_seqlen_k, page_size=page_size, kv_chunk=kv_chunk)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    p = _decode_params(q, k_cache, v_cache, page_table, cache_seqlens, max_seqlen_k, scale, page_size,
                       out, lse, workspace, kv_chunk, k_scale, v_scale, sliding_window, max_ctas,
                       overlap_previous)
    lib = _lib.load()
    _check(lib.pa_decode(ctypes.byref(p), _stream(q)), lib)
    return out


def mixed_batch(q_prefill: torch.Tensor, q_decode: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                page_table_prefill: torch.Tensor, cu_seqlens_q: torch.Tensor, cu_seqlens_k: torch.Tensor,
                max_seqlen_q: int, max_seqlen_k_prefill: int, page_table_decode: torch.Tensor,
                cache_seqlens: torch.Tensor, max_seqlen_k_decode: int, *, causal: bool = True,
                scale: float | None = None, out_prefill: torch.Tensor | None = None,
                out_decode: torch.Tensor | None = None, lse_prefill: torch.Tensor | None = None,
                lse_decode: torch.Tensor | None = None, workspace: torch.Tensor | None = None,
                kv_chunk: int = 0, scheduler: torch.Tensor | None = None, prefill_ctas: int = 0,
                decode_sliding_window: int = 0, k_scale: torch.Tensor | None = None,
                v_scale: torch.Tensor | None = None):
    """One continuous batch in one launch (``pa_mixed_batch``): prefill /
    extend of ``q_prefill`` [total_q, Hq, d] (cu_seqlens_q/k, its page table)
    and decode of ``q_decode`` [B, Hq, d] (cache_seqlens, its page table)
    over the same bf16 pools.  ``prefill_ctas`` > 0: that many CTAs take
    prefill tiles before decode key ranges (the others start on decode at
    once); 0: the kernel chooses the count from the work of both halves.
    ``decode_sliding_window`` W > 0: each decode query sees its sequence's
    last W keys only (the prefill half takes no window).  FP8 (uint8 E4M3)
    pools take their per-KV-head ``k_scale`` / ``v_scale`` for both halves.
    Returns (out_prefill, out_decode)."""
    dev = q_prefill.device
    p, out_prefill = _prefill_params(q_prefill, k_cache, v_cache, page_table_prefill, cu_seqlens_q, cu_seqlens_k,
                                     max_seqlen_q, max_seqlen_k_prefill, causal, scale, None, out_prefill,
                                     lse_prefill, k_scale, v_scale, 0, int(prefill_ctas), scheduler, None,
                                     PA_MIXED_SCHEDULER_INTS)
    _need(q_decode, "q_decode", torch.bfloat16, dev)
    _need(cache_seqlens, "cache_seqlens", torch.int32, dev)
    _need(page_table_decode, "page_table_decode", torch.int32, dev, contiguous=False)
    if out_decode is None:
        out_decode = torch.empty_like(q_decode)
    need = decode_workspace_size(q_decode.shape, k_cache, max_seqlen_k_decode, kv_chunk=kv_chunk)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    dp = _decode_params(q_decode, k_cache, v_cache, page_table_decode, cache_seqlens, max_seqlen_k_decode, scale,
                        None, out_decode, lse_decode, workspace, kv_chunk, k_scale, v_scale,
                        sliding_window=int(decode_sliding_window))
    lib = _lib.load()
    _check(lib.pa_mixed_batch(ctypes.byref(p), ctypes.byref(dp), _stream(q_prefill)), lib)
    return out_prefill, out_decode


def decode_noalloc(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                   page_table: torch.Tensor, cache_seqlens: torch.Tensor, max_seqlen_k: int, *,
                   scale: float | None = None, page_size: int | None = None,
                   out: torch.Tensor | None = None, lse: torch.Tensor | None = None,
                   kv_chunk: int = 0, k_scale: torch.Tensor | None = None,
                   v_scale: torch.Tensor | None = None, sliding_window: int = 0) -> torch.Tensor:
    """Split-KV decode through ``pa_decode_noalloc``: the split partials go to
    the library's fixed 32 MiB device scratch, so no workspace is allocated
    (for callers that may not allocate device memory).  Calls on one device
    must not overlap on the GPU; sizes whose scratch would exceed 32 MiB raise
    PagedAttentionError.  ``out`` (and ``lse``) must be given by a caller that
    cannot allocate; they are created here only for convenience."""
    dev = q.device
    _need(q, "q", torch.bfloat16, dev)
    _kv_dtype(k_cache, v_cache)
    for t, n in ((k_cache, "k_cache"), (v_cache, "v_cache")):
        _need(t, n, k_cache.dtype, dev)
    _need(cache_seqlens, "cache_seqlens", torch.int32, dev)
    _need(page_table, "page_table", torch.int32, dev, contiguous=False)
    if page_table.dim() != 2 or page_table.stride(1) != 1:
        raise ValueError("page_table must be 2-D with unit column stride")
    if out is None:
        out = torch.empty_like(q)
    _need(out, "out", torch.bfloat16, dev)
    if lse is not None:
        _need(lse, "lse", torch.float32, dev)
    p = _decode_params(q, k_cache, v_cache, page_table, cache_seqlens, max_seqlen_k, scale, page_size,
                       out, lse, None, kv_chunk, k_scale, v_scale, sliding_window)
    lib = _lib.load()
    _check(lib.pa_decode_noalloc(ctypes.byref(p), _stream(q)), lib)
    return out


def lse_combine(o_partial: torch.Tensor, lse_partial: torch.Tensor,
                splits_per_row: torch.Tensor | None = None, *, out: torch.Tensor | None = None,
                lse: torch.Tensor | None = None) -> torch.Tensor:
    """Merge split partials: o_partial fp32 [R, S, d], lse_partial fp32 [R, S]
    -> out bf16 [R, d] (and lse fp32 [R] if given)."""
    dev = o_partial.device
    _need(o_partial, "o_partial", torch.float32, dev)
    _need(lse_partial, "lse_partial", torch.float32, dev)
    R, S, d = o_partial.shape
    if lse_partial.shape != (R, S):
        raise ValueError("lse_partial must be [R, S]")
    if splits_per_row is not None:
        _need(splits_per_row, "splits_per_row", torch.int32, dev)
    if out is None:
        out = torch.empty((R, d), dtype=torch.bfloat16, device=dev)
    _need(out, "out", torch.bfloat16, dev)
    if lse is not None:
        _need(lse, "lse", torch.float32, dev)
    lib = _lib.load()
    _check(lib.pa_lse_combine(_ptr(o_partial), _ptr(lse_partial), _ptr(splits_per_row), R, S, d,
                              _ptr(out), _ptr(lse), _stream(o_partial)), lib)
    return out
