"""C-ABI checks that need no GPU: the library loads, exports every entry point
include/pa.h declares, computes host metadata exactly like the oracle, and
rejects malformed calls before any launch."""
import ctypes
import os
import re

import numpy as np
import pytest

import abi_reject_cases
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
    assert lib.pa_abi_version() == 3


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


@pytest.fixture(scope="module")
def rejections(lib):
    """Every malformed call of tests/abi_reject_cases.py, run in a child
    process that sees no GPU (CUDA_VISIBLE_DEVICES=''): the calls carry
    made-up device addresses, so a check that failed to reject one would only
    meet a CUDA error there, never a real GPU."""
    import json
    import subprocess
    import sys
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "tests", "abi_reject_cases.py")],
                       capture_output=True, text=True, env=env, timeout=300)
    assert r.returncode == 0, r.stderr
    return json.loads(r.stdout.strip().splitlines()[-1])


@pytest.mark.parametrize("case", abi_reject_cases.all_case_ids())
def test_rejects_before_launch(rejections, case):
    status, message = rejections[case]
    want = abi_reject_cases.expected()[case]
    assert status == want, f"{case}: status {status} ({message}), expected {want}"
    if want != 0:
        assert message, f"{case}: no error message"


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


def test_graph_bucket_selection():
    from paged_kv_flashattention_gb300.graphs import bucket_for
    assert bucket_for((1, 2, 4, 8, 16), 5) == 8
    assert bucket_for((16, 1, 4), 1) == 1
    assert bucket_for((1, 2, 4), 4) == 4
    with pytest.raises(ValueError):
        bucket_for((1, 2, 4), 5)


def test_page_table_binding_checks_shapes():
    """The binding rejects a page-table output too small for the rows and
    columns it would write, on the host, before any call into the library."""
    import torch
    from paged_kv_flashattention_gb300 import api
    tt = torch.zeros((4, 64), dtype=torch.int32)
    idx = torch.arange(3, dtype=torch.int32)
    with pytest.raises(ValueError):
        api.build_page_table(tt, idx, 64, 16, out=torch.zeros((2, 4), dtype=torch.int32))
    with pytest.raises(ValueError):
        api.build_page_table(tt, idx, 64, 16, out=torch.zeros((3, 3), dtype=torch.int32))
    with pytest.raises(ValueError):
        api.build_page_table(tt.t(), idx, 64, 16, out=torch.zeros((3, 4), dtype=torch.int32))


def test_device_error_bits_match_header():
    """The binding's PA_DEVERR_* constants are the header's."""
    import paged_kv_flashattention_gb300 as pa
    text = open(os.path.join(ROOT, "include", "pa.h")).read()
    defs = dict(re.findall(r"#define (PA_DEVERR_\w+) (\d+)", text))
    assert defs, "no PA_DEVERR_* defines found"
    for name, value in defs.items():
        assert getattr(pa, name) == int(value), name


def test_timeout_clears_cached_schedulers(monkeypatch):
    """After a device error word with PA_DEVERR_TIMEOUT, the cached scheduler
    arrays are zero again (a timed-out launch may leave its counters set);
    other error bits leave them alone.  The library call is a fake that
    reports the bits, so nothing runs on a device."""
    import torch
    from paged_kv_flashattention_gb300 import api

    class FakeLib:
        bits = 0

        def pa_device_error(self, out, stream):
            ctypes.cast(out, ctypes.POINTER(ctypes.c_int32))[0] = self.bits
            return 0

    fake = FakeLib()
    monkeypatch.setattr(api._lib, "load", lambda: fake)
    monkeypatch.setattr(api, "_stream", lambda t=None: 0)
    arrays = {("cpu", 1): torch.tensor([5, 3, 0, 0], dtype=torch.int32),
              ("cpu", 2): torch.tensor([0, 0, 7, 1], dtype=torch.int32)}
    monkeypatch.setattr(api, "_sched_arrays", arrays)
    fake.bits = api.PA_DEVERR_PAGE_RANGE
    assert api.device_error() == api.PA_DEVERR_PAGE_RANGE
    assert int(arrays[("cpu", 1)].sum()) == 8 and int(arrays[("cpu", 2)].sum()) == 8
    fake.bits = api.PA_DEVERR_TIMEOUT | api.PA_DEVERR_SEQLENS
    assert api.device_error() == api.PA_DEVERR_TIMEOUT | api.PA_DEVERR_SEQLENS
    assert all(int(t.abs().sum()) == 0 for t in arrays.values())
