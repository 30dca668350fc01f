"""Paged-KV exact attention oracle (fp64, CPU).

TEST INFRASTRUCTURE ONLY.  Only the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg may import this package.  The product path (the
CUDA library and its Python binding) never imports, links or runs it, and the
two share no code.

``oracle.c`` holds the plain C implementation (see its header for the passages
of "Transformer inference kernels: GEMM·Attention·FlashAttention·Fusion (3/10)"
and "code-series sgl-project mini-sglang 07" each function follows); this
module compiles it with gcc and wraps it for numpy arrays.  ``online.py`` holds
the online-softmax block merge and the split-KV merge written from sections 12
and 16 of the first page; ``brute.py`` a tiny pure-Python brute force.

All bf16 tensors cross this interface as ``numpy.uint16`` bit patterns, FP8
(E4M3) pools as ``numpy.uint8`` codes with float32 per-KV-head scales.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``oracle.c`` into ``_oracle.so`` (gcc, -O2, OpenMP)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    # -O2 without fast-math: every operation stays IEEE double.
    cmd = ["gcc", "-O2", "-fno-fast-math", "-ffp-contract=off", "-fopenmp", "-fPIC",
           "-shared", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _bind(lib):
    P = ctypes.c_void_p
    i32, i64, dbl = ctypes.c_int32, ctypes.c_int64, ctypes.c_double
    lib.oracle_store_kv.argtypes = [P, P, P, i64, P, P, i64, i64]
    lib.oracle_store_kv.restype = ctypes.c_int
    lib.oracle_page_table_from_token_table.argtypes = [P, i64, P, i32, i32, i32, P, i64]
    lib.oracle_page_table_from_token_table.restype = ctypes.c_int
    lib.oracle_seqlens.argtypes = [P, P, i32, P, P, P, P, P]
    lib.oracle_seqlens.restype = ctypes.c_int
    lib.oracle_attention.argtypes = [P, P, P, P, i64, P, P, i32, i32, i32, i32, i32,
                                     i64, ctypes.c_int, i32, dbl, P, i64, P, P]
    lib.oracle_attention.restype = ctypes.c_int
    lib.oracle_attention_fp8.argtypes = [P, P, P, P, P, P, i64, P, P, i32, i32, i32, i32, i32,
                                         i64, ctypes.c_int, i32, dbl, P, i64, P, P]
    lib.oracle_attention_fp8.restype = ctypes.c_int
    lib.oracle_attention_bm.argtypes = [P, P, P, P, i64, P, P, i32, i32, i32, i32, i32,
                                        i64, ctypes.c_int, i32, P, i32, i32, dbl, P, i64, P, P]
    lib.oracle_attention_bm.restype = ctypes.c_int
    lib.oracle_attention_fp8_bm.argtypes = [P, P, P, P, P, P, i64, P, P, i32, i32, i32, i32, i32,
                                            i64, ctypes.c_int, i32, P, i32, i32, dbl, P, i64, P, P]
    lib.oracle_attention_fp8_bm.restype = ctypes.c_int
    lib.oracle_e4m3_value.argtypes = [ctypes.c_uint8]
    lib.oracle_e4m3_value.restype = dbl
    lib.oracle_e4m3_encode.argtypes = [ctypes.c_float]
    lib.oracle_e4m3_encode.restype = ctypes.c_uint8
    lib.oracle_store_kv_fp8.argtypes = [P, P, P, i64, P, P, i64, i32, i32, P, P]
    lib.oracle_store_kv_fp8.restype = ctypes.c_int
    lib.oracle_rope_table.argtypes = [P, P, i32, i32, dbl]
    lib.oracle_rope_table.restype = ctypes.c_int
    lib.oracle_rope_rotate.argtypes = [P, P, i64, i32, i32, i32, ctypes.c_int, P, P, i32, P]
    lib.oracle_rope_rotate.restype = ctypes.c_int
    lib.oracle_round_bf16.argtypes = [P, i64, P]
    lib.oracle_round_bf16.restype = ctypes.c_int
    lib.oracle_num_threads.restype = ctypes.c_int
    lib.oracle_set_threads.argtypes = [ctypes.c_int]
    return lib


def load_variant(so_path: str):
    """Load another build of the oracle's C source (the tests compile
    deliberately broken copies to show that the pins catch each mistake)."""
    return _bind(ctypes.CDLL(os.path.abspath(so_path)))


def _load(lib=None):
    global _lib
    if lib is not None:
        return lib
    with _lock:
        if _lib is None:
            build()
            _lib = _bind(ctypes.CDLL(_LIB_PATH))
    return _lib


def _ptr(a: np.ndarray):
    return ctypes.c_void_p(a.ctypes.data)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def num_threads() -> int:
    return int(_load().oracle_num_threads())


def set_threads(n: int) -> None:
    _load().oracle_set_threads(int(n))


class OracleError(RuntimeError):
    pass


def _check(status: int, what: str):
    if status != 0:
        raise OracleError(f"{what} failed with oracle status {status}")


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns (uint16) to float64."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def store_kv(k, v, slot_mapping, k_cache, v_cache, *, lib=None) -> None:
    """KV-cache store into ``k_cache``/``v_cache`` in place (uint16 arrays,
    first axis = slot, the rest = one token's row)."""
    k = _c(k, np.uint16)
    v = _c(v, np.uint16)
    sm = _c(slot_mapping, np.int32)
    assert k_cache.dtype == np.uint16 and k_cache.flags.c_contiguous
    assert v_cache.dtype == np.uint16 and v_cache.flags.c_contiguous
    T = sm.shape[0]
    row = int(np.prod(k_cache.shape[1:])) if k_cache.ndim > 1 else 1
    slots = k_cache.shape[0]
    assert k.size == T * row and v.size == T * row
    _check(_load(lib).oracle_store_kv(_ptr(k), _ptr(v), _ptr(sm), T, _ptr(k_cache), _ptr(v_cache),
                                   slots, row), "oracle_store_kv")


def e4m3_value(codes, *, lib=None) -> np.ndarray:
    """float64 values of E4M3 codes (uint8), NaN for the NaN codes."""
    c = np.asarray(codes, dtype=np.uint8)
    lib = _load(lib)
    table = np.array([lib.oracle_e4m3_value(i) for i in range(256)], dtype=np.float64)
    return table[c]


def e4m3_encode(x, *, lib=None) -> np.ndarray:
    """Nearest E4M3 codes (uint8) of float32 values (ties to even, saturating)."""
    xf = np.asarray(x, dtype=np.float32)
    lib = _load(lib)
    flat = [lib.oracle_e4m3_encode(float(v)) for v in xf.ravel()]
    return np.array(flat, dtype=np.uint8).reshape(xf.shape)


def store_kv_fp8(k, v, slot_mapping, k_cache, v_cache, k_scale, v_scale, *, lib=None) -> None:
    """FP8 KV-cache store into uint8 ``k_cache``/``v_cache`` ([slots, Hkv, d])
    in place; k, v: bf16 bits [T, Hkv, d]; scales float32 [Hkv]."""
    assert k_cache.dtype == np.uint8 and k_cache.flags.c_contiguous and k_cache.ndim == 3
    assert v_cache.dtype == np.uint8 and v_cache.flags.c_contiguous and v_cache.shape == k_cache.shape
    slots, Hkv, d = k_cache.shape
    k = _c(k, np.uint16)
    v = _c(v, np.uint16)
    sm = _c(slot_mapping, np.int32)
    ks = _c(k_scale, np.float32)
    vs = _c(v_scale, np.float32)
    T = sm.shape[0]
    assert k.size == T * Hkv * d and v.size == T * Hkv * d and ks.size == Hkv and vs.size == Hkv
    _check(_load(lib).oracle_store_kv_fp8(_ptr(k), _ptr(v), _ptr(sm), T, _ptr(k_cache), _ptr(v_cache),
                                          slots, Hkv, d, _ptr(ks), _ptr(vs)), "oracle_store_kv_fp8")


def rope_table(max_pos: int, rot_dim: int, base: float, *, lib=None):
    """(cos, sin) float64 [max_pos, rot_dim/2] of angle p * base^(-2i/rot_dim)."""
    h = int(rot_dim) // 2
    c = np.zeros((int(max_pos), h), np.float64)
    s_ = np.zeros((int(max_pos), h), np.float64)
    _check(_load(lib).oracle_rope_table(_ptr(c), _ptr(s_), int(max_pos), int(rot_dim), float(base)),
           "oracle_rope_table")
    return c, s_


def rope_rotate(x, positions, cos, sin, *, rot_dim: int, interleaved: bool = False, lib=None):
    """Rotary embedding of bf16 bits x [T, H, d] at positions [T]; exact
    float64 result [T, H, d] (elements past rot_dim unchanged)."""
    x = _c(x, np.uint16)
    pos = _c(positions, np.int32)
    c = _c(cos, np.float64)
    s_ = _c(sin, np.float64)
    T, H, d = x.shape
    out = np.zeros((T, H, d), np.float64)
    _check(_load(lib).oracle_rope_rotate(_ptr(x), _ptr(pos), T, H, d, int(rot_dim), int(bool(interleaved)),
                                         _ptr(c), _ptr(s_), c.shape[0], _ptr(out)), "oracle_rope_rotate")
    return out


def round_bf16(x, *, lib=None) -> np.ndarray:
    """Nearest bf16 bits (ties to even) of float64 values, in one rounding."""
    xf = _c(x, np.float64)
    out = np.zeros(xf.shape, np.uint16)
    _check(_load(lib).oracle_round_bf16(_ptr(xf), xf.size, _ptr(out)), "oracle_round_bf16")
    return out


def page_table_from_token_table(token_table, table_idx, max_seqlen_k: int, page_size: int,
                                out_cols: int | None = None, *, lib=None) -> np.ndarray:
    tt = _c(token_table, np.int32)
    ti = _c(table_idx, np.int32)
    cols = -(-int(max_seqlen_k) // int(page_size))
    out_cols = cols if out_cols is None else int(out_cols)
    out = np.zeros((ti.shape[0], out_cols), dtype=np.int32)
    _check(_load(lib).oracle_page_table_from_token_table(
        _ptr(tt), tt.shape[1], _ptr(ti), ti.shape[0], int(max_seqlen_k), int(page_size),
        _ptr(out), out_cols), "oracle_page_table_from_token_table")
    return out


def seqlens(cached_len, extend_len, *, lib=None):
    """(cu_seqlens_q, cu_seqlens_k, cache_seqlens, max_seqlen_q, max_seqlen_k)."""
    c = _c(cached_len, np.int32)
    e = _c(extend_len, np.int32)
    B = c.shape[0]
    cu_q = np.zeros(B + 1, np.int32)
    cu_k = np.zeros(B + 1, np.int32)
    cs = np.zeros(max(B, 1), np.int32)
    mq = np.zeros(1, np.int32)
    mk = np.zeros(1, np.int32)
    _check(_load(lib).oracle_seqlens(_ptr(c), _ptr(e), B, _ptr(cu_q), _ptr(cu_k), _ptr(cs),
                                     _ptr(mq), _ptr(mk)), "oracle_seqlens")
    return cu_q, cu_k, cs[:B], int(mq[0]), int(mk[0])


def attention(q, k_cache, v_cache, page_table, cu_seqlens_q, cu_seqlens_k, *,
              num_q_heads: int, num_kv_heads: int, head_dim: int, page_size: int,
              causal: bool, scale: float, rows=None, k_scale=None, v_scale=None, window_left: int = -1,
              block_mask=None, lib=None):
    """fp64 attention over paged K/V.

    q: uint16 [Tq, Hq, d]; caches: uint16 [num_pages*page_size, Hkv, d] (any
    shape with that element order), or uint8 E4M3 codes with float32
    ``k_scale``/``v_scale`` [Hkv]; page_table int32 [B, stride].
    block_mask: optional uint8 [B, nq, nk]; entry [b, i // 128, j // 128] == 0
    hides key j from query row i of request b.
    Returns (out, lse): float64 [Tq, Hq, d] and [Tq, Hq], or, when ``rows`` (an
    int64 [n, 2] array of (token, head)) is given, [n, d] and [n].
    """
    q = _c(q, np.uint16)
    fp8 = k_scale is not None
    kt = np.uint8 if fp8 else np.uint16
    kc = k_cache if (k_cache.dtype == kt and k_cache.flags.c_contiguous) else _c(k_cache, kt)
    vc = v_cache if (v_cache.dtype == kt and v_cache.flags.c_contiguous) else _c(v_cache, kt)
    pt = _c(page_table, np.int32)
    if pt.ndim == 1:
        pt = pt.reshape(-1, 1)
    cq = _c(cu_seqlens_q, np.int32)
    ck = _c(cu_seqlens_k, np.int32)
    B = cq.shape[0] - 1
    Hq, Hkv, d, P = int(num_q_heads), int(num_kv_heads), int(head_dim), int(page_size)
    num_pages = kc.size // (P * Hkv * d)
    Tq = int(cq[-1]) if B > 0 else 0
    if rows is None:
        out = np.zeros((Tq, Hq, d), dtype=np.float64)
        lse = np.zeros((Tq, Hq), dtype=np.float64)
        rp, nr = None, 0
    else:
        rws = _c(rows, np.int64).reshape(-1, 2)
        out = np.zeros((rws.shape[0], d), dtype=np.float64)
        lse = np.zeros((rws.shape[0],), dtype=np.float64)
        rp, nr = _ptr(rws), rws.shape[0]
    if block_mask is not None:
        bm = _c(block_mask, np.uint8)
        assert bm.ndim == 3 and bm.shape[0] == B
        if fp8:
            ks = _c(k_scale, np.float32)
            vs = _c(v_scale, np.float32)
            _check(_load(lib).oracle_attention_fp8_bm(
                _ptr(q), _ptr(kc), _ptr(vc), _ptr(ks), _ptr(vs), _ptr(pt), pt.shape[1], _ptr(cq), _ptr(ck),
                B, Hq, Hkv, d, P, num_pages, int(bool(causal)), int(window_left), _ptr(bm), bm.shape[1],
                bm.shape[2], float(scale), rp, nr, _ptr(out), _ptr(lse)), "oracle_attention_fp8_bm")
        else:
            _check(_load(lib).oracle_attention_bm(
                _ptr(q), _ptr(kc), _ptr(vc), _ptr(pt), pt.shape[1], _ptr(cq), _ptr(ck), B,
                Hq, Hkv, d, P, num_pages, int(bool(causal)), int(window_left), _ptr(bm), bm.shape[1],
                bm.shape[2], float(scale), rp, nr, _ptr(out), _ptr(lse)), "oracle_attention_bm")
        return out, lse
    if fp8:
        ks = _c(k_scale, np.float32)
        vs = _c(v_scale, np.float32)
        assert ks.size == Hkv and vs.size == Hkv
        _check(_load(lib).oracle_attention_fp8(
            _ptr(q), _ptr(kc), _ptr(vc), _ptr(ks), _ptr(vs), _ptr(pt), pt.shape[1], _ptr(cq), _ptr(ck),
            B, Hq, Hkv, d, P, num_pages, int(bool(causal)), int(window_left), float(scale), rp, nr,
            _ptr(out), _ptr(lse)), "oracle_attention_fp8")
        return out, lse
    _check(_load(lib).oracle_attention(
        _ptr(q), _ptr(kc), _ptr(vc), _ptr(pt), pt.shape[1], _ptr(cq), _ptr(ck), B,
        Hq, Hkv, d, P, num_pages, int(bool(causal)), int(window_left), float(scale), rp, nr,
        _ptr(out), _ptr(lse)), "oracle_attention")
    return out, lse


def decode(q, k_cache, v_cache, page_table, cache_seqlens, *, num_q_heads: int,
           num_kv_heads: int, head_dim: int, page_size: int, scale: float, rows=None,
           k_scale=None, v_scale=None, window_left: int = -1, lib=None):
    """Decode attention: one query token per sequence attending to all
    cache_seqlens[b] keys (the new token already stored).  q: [B, Hq, d]."""
    cs = np.asarray(cache_seqlens, dtype=np.int64)
    B = cs.shape[0]
    cu_q = np.arange(B + 1, dtype=np.int32)
    cu_k = np.zeros(B + 1, dtype=np.int64)
    cu_k[1:] = np.cumsum(cs)
    return attention(q, k_cache, v_cache, page_table, cu_q, cu_k.astype(np.int32),
                     num_q_heads=num_q_heads, num_kv_heads=num_kv_heads, head_dim=head_dim,
                     page_size=page_size, causal=True, scale=scale, rows=rows, k_scale=k_scale,
                     v_scale=v_scale, window_left=window_left, lib=lib)


from . import online  # noqa: E402,F401  (re-export)
