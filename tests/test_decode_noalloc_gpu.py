"""pa_decode_noalloc: decode for callers that may not allocate device memory
(graph capture, host-owned memory arenas, hard memory budgets).  It must agree
with pa_decode within the parity tolerance on two calls in a row (the shared
scratch keeps the previous call's contents), and with the fp64 oracle.  Its
rejection of sizes beyond the fixed 32 MiB scratch is checked without a GPU
(tests/abi_reject_cases.py), so nothing here depends on the order in which
the test files run."""
import pytest
import torch

import workloads as W
from pa_harness import DeviceProblem, TOL_MAX_ABS, TOL_MEAN_ABS, compare, oracle_ref

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
    refs = {p.name: oracle_ref(p) for p, _ in cases}
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
            # and against the oracle itself, not only the other entry point
            o_ref, l_ref = refs[p.name]
            compare(out, o_ref, f"{p.name} no-alloc vs oracle, call {rep}", lse_gpu=lse, lse_ref=l_ref)
            assert pa.device_error() == 0
