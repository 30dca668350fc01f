"""C-ABI checks that need no GPU: the library loads, exports every entry point
include/pa.h declares, computes host metadata exactly like the oracle, and
rejects malformed calls before any launch."""
import ctypes
import os
import re

import numpy as np
import pytest

import oracle
import workloads as W

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from paged_kv_flashattention_gb300 import build, _lib
    build.build()
    return _lib.load()


def declared_functions():
    src = open(os.path.join(ROOT, "include", "pa.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(pa_[a-z0-9_]+)\s*\(", src)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for must in ("pa_store_kv", "pa_prefill", "pa_decode", "pa_decode_workspace_size",
                 "pa_lse_combine", "pa_build_seqlens", "pa_build_page_table"):
        assert must in names


def test_exports_every_declared_symbol(lib):
    from paged_kv_flashattention_gb300 import _lib
    for name in declared_functions():
        assert hasattr(lib, name), f"libpa.so does not export {name}"
        assert name in _lib.SIGNATURES, f"binding has no signature for {name}"
    assert lib.pa_abi_version() == 1


@pytest.mark.parametrize("cfg", [1, 2, 3, 4])
def test_build_seqlens_matches_oracle(lib, cfg):
    import paged_kv_flashattention_gb300 as pa
    p = W.config(cfg, with_data=False)
    got = pa.build_seqlens(p.cached_len, p.extend_len)
    want = oracle.seqlens(p.cached_len, p.extend_len)
    for g, w in zip(got[:3], want[:3]):
        assert np.array_equal(g, w)
    assert got[3:] == want[3:]


def test_build_seqlens_edges(lib):
    import paged_kv_flashattention_gb300 as pa
    for cached, ext in (([], []), ([0], [0]), ([5, 0, 0], [0, 0, 7]), ([2**30], [2**30 - 1])):
        got = pa.build_seqlens(cached, ext)
        want = oracle.seqlens(cached, ext)
        for g, w in zip(got[:3], want[:3]):
            assert np.array_equal(g, w)
        assert got[3:] == want[3:]
    with pytest.raises(pa.PagedAttentionError):
        pa.build_seqlens([-1], [3])
    with pytest.raises(pa.PagedAttentionError):
        pa.build_seqlens([2**30, 2**30], [2**30, 0])    # total keys overflow int32


def _prefill(lib, **kw):
    from paged_kv_flashattention_gb300 import _lib
    base = dict(q=0x1000, k_cache=0x2000, v_cache=0x3000, page_table=0x4000, page_table_stride=64,
                total_q=64, cu_seqlens_q=0x5000, cu_seqlens_k=0x6000, num_seqs=2, max_seqlen_q=16,
                max_seqlen_k=32, num_q_heads=8, num_kv_heads=2, head_dim=128, page_size=16,
                num_pages=100, causal=1, scale=0.1, out=0x7000, lse=None, lse_stride=0)
    base.update(kw)
    p = _lib.PrefillParams(**base)
    return lib.pa_prefill(ctypes.byref(p), None)


def _decode(lib, **kw):
    from paged_kv_flashattention_gb300 import _lib
    base = dict(q=0x1000, k_cache=0x2000, v_cache=0x3000, page_table=0x4000, page_table_stride=64,
                cache_seqlens=0x5000, num_seqs=2, max_seqlen_k=4096, num_q_heads=8,
                num_kv_heads=2, head_dim=128, page_size=16, num_pages=1000, scale=0.1,
                out=0x7000, lse=None, workspace=0x8000, workspace_bytes=16, kv_chunk=0)
    base.update(kw)
    p = _lib.DecodeParams(**base)
    return lib.pa_decode(ctypes.byref(p), None)


INVALID, UNSUPPORTED = 1, 2


@pytest.mark.parametrize("kw,status", [
    (dict(head_dim=96), UNSUPPORTED),
    (dict(page_size=8), UNSUPPORTED),
    (dict(num_q_heads=6, num_kv_heads=4), INVALID),
    (dict(num_q_heads=32, num_kv_heads=2), UNSUPPORTED),     # group 16
    (dict(q=0x1001), INVALID),                               # misaligned
    (dict(out=0), INVALID),
    (dict(max_seqlen_q=64, max_seqlen_k=32), INVALID),
    (dict(causal=2), INVALID),
    (dict(page_table_stride=1), INVALID),
    (dict(scale=float("nan")), INVALID),
    (dict(scale=0.0), INVALID),
    (dict(scale=-0.1), INVALID),
    (dict(scale=float("inf")), INVALID),
    (dict(sliding_window=-3), INVALID),
])
def test_prefill_rejects_before_launch(lib, kw, status):
    assert _prefill(lib, **kw) == status
    assert lib.pa_last_error()


@pytest.mark.parametrize("kw,status", [
    (dict(head_dim=80), UNSUPPORTED),
    (dict(kv_chunk=24), INVALID),
    (dict(kv_chunk=-16), INVALID),
    (dict(workspace=0), INVALID),
    (dict(workspace_bytes=16), INVALID),                      # far too small for 4096 keys
    (dict(k_cache=0x2008), INVALID),
    (dict(page_table_stride=8), INVALID),
    (dict(num_seqs=20000), UNSUPPORTED),
    (dict(kv_dtype=2), INVALID),
    (dict(kv_dtype=1), INVALID),                              # FP8 without scales
    (dict(sliding_window=-1), INVALID),
    (dict(scale=-0.125), INVALID),
    (dict(scale=float("inf")), INVALID),
])
def test_decode_rejects_before_launch(lib, kw, status):
    assert _decode(lib, **kw) == status


def test_store_rejects_before_launch(lib):
    assert lib.pa_store_kv(0x1001, 0x2000, 0x3000, 4, 0x4000, 0x5000, 64, 2, 64, None) == INVALID
    assert lib.pa_store_kv(0x1000, 0x2000, 0x3000, -1, 0x4000, 0x5000, 64, 2, 64, None) == INVALID
    assert lib.pa_store_kv(0x1000, 0x2000, 0x3000, 4, 0x4000, 0x5000, 64, 1, 4, None) == UNSUPPORTED
    # zero tokens: nothing to do, nothing launched
    assert lib.pa_store_kv(0, 0, 0, 0, 0, 0, 0, 2, 64, None) == 0
    # FP8 store: scales required, head_dim a multiple of 16
    assert lib.pa_store_kv_fp8(0x1000, 0x2000, 0x3000, 4, 0x4000, 0x5000, 64, 2, 64, None, 0x6000, None) == INVALID
    assert lib.pa_store_kv_fp8(0x1000, 0x2000, 0x3000, 4, 0x4000, 0x5000, 64, 2, 72, 0x6000, 0x7000, None) == UNSUPPORTED
    assert lib.pa_store_kv_fp8(0x1008, 0x2000, 0x3000, 4, 0x4000, 0x5000, 64, 2, 64, 0x6000, 0x7000, None) == INVALID
    assert lib.pa_store_kv_fp8(0, 0, 0, 0, 0, 0, 0, 2, 64, None, None, None) == 0


def test_decode_workspace_size_host_only(lib):
    from paged_kv_flashattention_gb300 import _lib
    p = _lib.DecodeParams(num_seqs=64, max_seqlen_k=4096, num_q_heads=32, num_kv_heads=8,
                          head_dim=64, page_size=16, num_pages=10000, scale=0.125, kv_chunk=256)
    n = lib.pa_decode_workspace_size(ctypes.byref(p))
    # a row of 4096 keys cut into ranges of >= 256 keys touches at most 17 of them
    splits = 4096 // 256 + 1
    rows = 64 * 32 * splits
    assert n >= rows * 64 * 4 + rows * 4 + (64 + 1) * 4
    assert lib.pa_decode_kv_chunk(ctypes.byref(p)) == 256
    p.kv_chunk = 4096
    small = lib.pa_decode_workspace_size(ctypes.byref(p))
    assert 0 < small < n and small >= 64 * 32 * 2 * (64 + 1) * 4


@pytest.mark.parametrize("max_k,want", [(1, 64), (1000, 64), (2048, 64), (4096, 128), (5000, 160),
                                         (32768, 1024)])
def test_decode_automatic_split(lib, max_k, want):
    """kv_chunk = 0 takes 1/32 of the longest context, a multiple of 16, at
    least 64 keys."""
    from paged_kv_flashattention_gb300 import _lib
    p = _lib.DecodeParams(num_seqs=8, max_seqlen_k=max_k, num_q_heads=32, num_kv_heads=8,
                          head_dim=128, page_size=16, num_pages=10000, scale=0.1, kv_chunk=0)
    assert lib.pa_decode_kv_chunk(ctypes.byref(p)) == want


def test_rope_table_host(lib):
    """The host rotary table equals the oracle's fp64 table rounded to fp32
    (within half an fp32 step of values <= 1)."""
    import paged_kv_flashattention_gb300 as pa
    for r, base in ((128, 10000.0), (64, 500000.0)):
        t = pa.rope_cos_sin_table(2048, r, base).numpy().astype(np.float64)
        c, s = oracle.rope_table(2048, r, base)
        assert np.abs(t[:, :r // 2] - c).max() <= 2.0 ** -25 and np.abs(t[:, r // 2:] - s).max() <= 2.0 ** -25
    with pytest.raises(pa.PagedAttentionError):
        pa.rope_cos_sin_table(16, 7, 10000.0)


def test_rope_store_rejects_before_launch(lib):
    from paged_kv_flashattention_gb300 import _lib
    base = dict(q=0x1000, q_out=0x1000, k=0x2000, v=0x3000, positions=0x4000, cos_sin=0x5000, max_pos=64,
                rot_dim=128, interleaved=0, slot_mapping=0x6000, num_tokens=4, num_q_heads=8,
                num_kv_heads=2, head_dim=128, k_cache=0x7000, v_cache=0x8000, num_slots=64, kv_dtype=0)
    for kw, status in ((dict(rot_dim=72), UNSUPPORTED), (dict(rot_dim=256), UNSUPPORTED),
                       (dict(interleaved=2), INVALID), (dict(kv_dtype=1), INVALID),
                       (dict(q=0x1008), INVALID), (dict(head_dim=72), UNSUPPORTED)):
        p = _lib.RopeStoreParams(**{**base, **kw})
        assert lib.pa_rope_store_kv(ctypes.byref(p), None) == status, kw


def test_graph_bucket_selection():
    from paged_kv_flashattention_gb300.graphs import bucket_for
    assert bucket_for((1, 2, 4, 8, 16), 5) == 8
    assert bucket_for((16, 1, 4), 1) == 1
    assert bucket_for((1, 2, 4), 4) == 4
    with pytest.raises(ValueError):
        bucket_for((1, 2, 4), 5)
