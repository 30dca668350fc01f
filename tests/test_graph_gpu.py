"""Decode through captured CUDA graphs (one per batch-size bucket, dummy
requests padding the batch): the real rows agree with the fp64 oracle, the
dummy rows are O = 0 / lse = -inf, and one graph serves new lengths and new
contents of the fixed buffers."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from oracle_pins import _meta, stored_caches
from pa_harness import DeviceProblem, compare, oracle_ref

pytestmark = pytest.mark.gpu


def test_decode_graph_runner(cuda_device):
    import paged_kv_flashattention_gb300 as pa
    p = W.config(2)                                   # 64 sequences, Hq 32 / Hkv 8, d 64
    d = DeviceProblem(p, cuda_device)
    d.store()
    m = d.metadata()
    ref, ref_lse = oracle_ref(p)
    runner = pa.DecodeGraphRunner(d.k_cache, d.v_cache, num_q_heads=p.num_q_heads,
                                  max_seqlen_k=m.max_seqlen_k, buckets=(1, 4, 16, 64), scale=p.scale)
    runner.capture()
    lengths = p.device_len.astype(np.int32)
    for B in (3, 17, 64, 1, 16):
        out, lse = runner.run(lengths[:B], q=d.q[:B], page_table=m.page_table[:B])
        torch.cuda.synchronize()
        compare(out, ref[:B], f"graph B={B}", lse_gpu=lse, lse_ref=ref_lse[:B])
        bucket = pa.bucket_for(runner.buckets, B)
        assert torch.count_nonzero(runner.out[B:bucket]).item() == 0, "dummy rows must be zero"
        assert torch.all(torch.isneginf(runner.lse[B:bucket])), "dummy rows must have lse = -inf"


def test_decode_graph_new_lengths(cuda_device):
    """The same graph after the lengths change: every sequence now attends to
    a shorter prefix of its keys."""
    import paged_kv_flashattention_gb300 as pa
    p = W.config(2)
    d = DeviceProblem(p, cuda_device)
    d.store()
    m = d.metadata()
    runner = pa.DecodeGraphRunner(d.k_cache, d.v_cache, num_q_heads=p.num_q_heads,
                                  max_seqlen_k=m.max_seqlen_k, buckets=(32,), scale=p.scale)
    runner.capture()
    rng = np.random.default_rng(61)
    B = 29
    short = (p.device_len[:B] * rng.uniform(0.1, 1.0, B)).astype(np.int32).clip(1)
    out, lse = runner.run(short, q=d.q[:B], page_table=m.page_table[:B])
    torch.cuda.synchronize()
    _, _, _, pt = _meta(p)
    kc, vc = stored_caches(p)                          # the oracle's own store
    want, want_lse = oracle.decode(p.q[:B], kc, vc, pt[:B], short, num_q_heads=p.num_q_heads,
                                   num_kv_heads=p.num_kv_heads, head_dim=p.head_dim,
                                   page_size=p.page_size, scale=p.scale)
    compare(out, want, "graph with shorter lengths", lse_gpu=lse, lse_ref=want_lse)
