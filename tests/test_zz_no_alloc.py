"""pa_decode_noalloc: decode for callers that may not allocate device memory
(graph capture, host-owned memory arenas, hard memory budgets).  It must agree
with pa_decode within the parity tolerance on two calls in a row (the shared
scratch keeps the previous call's contents), and reject sizes beyond its fixed
32 MiB scratch without launching.  This file is collected last on purpose."""
import ctypes

import numpy as np
import pytest
import torch

import workloads as W
from pa_harness import DeviceProblem, TOL_MAX_ABS, TOL_MEAN_ABS

pytestmark = pytest.mark.gpu


def _inputs(p, dev):
    from paged_kv_flashattention_gb300 import metadata
    d = DeviceProblem(p, dev)
    d.store()
    m = metadata.prepare(p.cached_len, p.extend_len, d.token_table, d.table_idx, p.page_size)
    return d, m


def _close(a, b, what):
    diff = (a.float() - b.float()).abs()
    assert torch.isfinite(a.float()).all(), f"{what}: non-finite output"
    assert diff.max().item() <= TOL_MAX_ABS, f"{what}: max abs diff {diff.max().item()}"
    assert diff.mean().item() <= TOL_MEAN_ABS, f"{what}: mean abs diff {diff.mean().item()}"


def test_noalloc_matches_decode_twice(cuda_device):
    import paged_kv_flashattention_gb300 as pa
    cases = [(W.config(2), 0), (W.config(1), 16)]   # a split batch, then a smaller one
    for rep in range(2):                             # two calls in a row per case
        for p, chunk in cases:
            d, m = _inputs(p, cuda_device)
            B, Hq = p.num_seqs, p.num_q_heads
            lse_ref = torch.empty((B, Hq), dtype=torch.float32, device=cuda_device)
            ref = pa.decode(d.q, d.k_cache, d.v_cache, m.page_table, m.cache_seqlens, m.max_seqlen_k,
                            scale=p.scale, lse=lse_ref, kv_chunk=chunk)
            out = torch.full_like(d.q, float("nan"))
            lse = torch.full((B, Hq), float("nan"), dtype=torch.float32, device=cuda_device)
            pa.decode_noalloc(d.q, d.k_cache, d.v_cache, m.page_table, m.cache_seqlens,
                              m.max_seqlen_k, scale=p.scale, out=out, lse=lse, kv_chunk=chunk)
            torch.cuda.synchronize()
            _close(out, ref, f"{p.name} call {rep}")
            assert (lse - lse_ref).abs().max().item() <= 2e-3
            assert pa.device_error() == 0


def test_noalloc_rejects_oversized_scratch(cuda_device):
    import paged_kv_flashattention_gb300 as pa
    from paged_kv_flashattention_gb300 import _lib
    lib = _lib.load()
    # 4096 sequences of 32768 keys with 128-key splits need far more than 32 MiB
    p = _lib.DecodeParams(q=0x1000, k_cache=0x2000, v_cache=0x3000, page_table=0x4000,
                          page_table_stride=2048, cache_seqlens=0x5000, num_seqs=4096,
                          max_seqlen_k=32768, num_q_heads=32, num_kv_heads=8, head_dim=128,
                          page_size=16, num_pages=1 << 20, scale=0.1, out=0x6000, kv_chunk=128)
    assert lib.pa_decode_workspace_size(ctypes.byref(p)) > (32 << 20)
    assert lib.pa_decode_noalloc(ctypes.byref(p), None) == 2
    assert b"32" in lib.pa_last_error()
