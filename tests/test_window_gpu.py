"""GPU parity of sliding-window attention (a query at position p sees keys
p - (W - 1) .. p) against the fp64 oracle, for prefill / extend and decode,
bf16 and FP8 pools, both page sizes."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from oracle_pins import _meta, stored_caches
from pa_harness import DeviceProblem, compare

pytestmark = pytest.mark.gpu


def _oracle_window(p, window, rows=None):
    cu_q, cu_k, _, pt = _meta(p)
    kc, vc = stored_caches(p)
    return oracle.attention(p.q, kc, vc, pt, cu_q, cu_k, num_q_heads=p.num_q_heads,
                            num_kv_heads=p.num_kv_heads, head_dim=p.head_dim, page_size=p.page_size,
                            causal=p.causal, scale=p.scale, window_left=window - 1, rows=rows)


def _prefill_window(p, dev, window, what):
    import paged_kv_flashattention_gb300 as pa
    d = DeviceProblem(p, dev)
    d.store()
    m = d.metadata()
    Tq = d.q.shape[0]
    lse = torch.empty((p.num_q_heads, max(Tq, 1)), dtype=torch.float32, device=dev)
    out = pa.prefill(d.q, d.k_cache, d.v_cache, m.page_table, m.cu_seqlens_q, m.cu_seqlens_k,
                     m.max_seqlen_q, m.max_seqlen_k, causal=p.causal, scale=p.scale, lse=lse,
                     sliding_window=window)
    torch.cuda.synchronize()
    ref, ref_lse = _oracle_window(p, window)
    compare(out, ref, what, lse_gpu=lse[:, :ref.shape[0]].T.contiguous(), lse_ref=ref_lse)


CASES = [
    ([0, 0, 0], [300, 129, 17]),            # no cache hit: the window cuts inside the prompt
    ([200, 1000, 3], [160, 40, 260]),        # cached prefix + extend: the window cuts the prefix
]


@pytest.mark.parametrize("window", [1, 16, 100, 128, 129, 300])
@pytest.mark.parametrize("page", [1, 16])
def test_prefill_sliding_window(cuda_device, window, page):
    for n, (cached, ext) in enumerate(CASES):
        for hq, hkv, d in ((8, 2, 128), (4, 4, 64)):
            p = W.small_problem(3300 + 11 * n + window + page + hq, cached, ext, num_q_heads=hq,
                                num_kv_heads=hkv, head_dim=d, page_size=page)
            _prefill_window(p, cuda_device, window, f"prefill W{window} P{page} d{d} g{hq // hkv} case{n}")


def test_prefill_sliding_window_non_causal(cuda_device):
    p = W.build("noncausal-window", cached_len=[0, 40, 200], extend_len=[33, 130, 64], num_q_heads=8,
                num_kv_heads=2, head_dim=128, page_size=16, seed=3401, causal=False)
    _prefill_window(p, cuda_device, 50, "non-causal W50")


def _decode_window(p, dev, window, kv_chunk=0, what=""):
    d = DeviceProblem(p, dev)
    d.store()
    out, lse = None, None
    import paged_kv_flashattention_gb300 as pa
    m = d.metadata()
    lse = torch.empty((p.num_seqs, p.num_q_heads), dtype=torch.float32, device=dev)
    out = pa.decode(d.q, d.k_cache, d.v_cache, m.page_table, m.cache_seqlens, m.max_seqlen_k,
                    scale=p.scale, lse=lse, kv_chunk=kv_chunk, sliding_window=window)
    torch.cuda.synchronize()
    ref, ref_lse = _oracle_window(p, window)
    compare(out, ref.reshape(out.shape), what, lse_gpu=lse, lse_ref=ref_lse.reshape(lse.shape))


@pytest.mark.parametrize("window", [1, 16, 17, 100, 1024])
@pytest.mark.parametrize("page", [1, 16])
def test_decode_sliding_window(cuda_device, window, page):
    Lk = np.array([1, 15, 16, 17, 33, 100, 257, 2000], np.int32)
    p = W.small_problem(3500 + window + page, Lk - 1, np.ones_like(Lk), num_q_heads=32, num_kv_heads=8,
                        head_dim=128, page_size=page)
    for chunk in (0, 16):
        _decode_window(p, cuda_device, window, chunk, f"decode W{window} P{page} C{chunk}")


def test_decode_sliding_window_llama(cuda_device):
    _decode_window(W.config(2), cuda_device, 1024, what="llama32 decode W1024")


def test_fp8_sliding_window(cuda_device):
    """FP8 pools with a window, decode and prefill."""
    from test_fp8_gpu import FP8Problem
    import paged_kv_flashattention_gb300 as pa
    Lk = np.array([40, 300, 1500], np.int32)
    p = W.small_problem(3600, Lk - 1, np.ones_like(Lk), num_q_heads=32, num_kv_heads=8, head_dim=128,
                        page_size=16)
    f = FP8Problem(p, cuda_device, 3601)
    lse = torch.empty((p.num_seqs, p.num_q_heads), dtype=torch.float32, device=cuda_device)
    out = pa.decode(f.q, f.k_cache, f.v_cache, f.meta.page_table, f.meta.cache_seqlens, f.meta.max_seqlen_k,
                    scale=p.scale, lse=lse, k_scale=f.k_scale, v_scale=f.v_scale, sliding_window=200)
    torch.cuda.synchronize()
    cu_q, cu_k, _, pt = _meta(p)
    ref, ref_lse = oracle.attention(p.q, f.kc, f.vc, pt, cu_q, cu_k, num_q_heads=32, num_kv_heads=8,
                                    head_dim=128, page_size=16, causal=True, scale=p.scale,
                                    k_scale=f.ks, v_scale=f.vs, window_left=199)
    compare(out, ref.reshape(out.shape), "fp8 decode W200", lse_gpu=lse, lse_ref=ref_lse.reshape(lse.shape))
    p2 = W.small_problem(3602, [100, 0], [300, 200], num_q_heads=8, num_kv_heads=2, head_dim=128, page_size=16)
    f2 = FP8Problem(p2, cuda_device, 3603)
    m = f2.meta
    Tq = f2.q.shape[0]
    lse2 = torch.empty((8, Tq), dtype=torch.float32, device=cuda_device)
    out2 = pa.prefill(f2.q, f2.k_cache, f2.v_cache, m.page_table, m.cu_seqlens_q, m.cu_seqlens_k,
                      m.max_seqlen_q, m.max_seqlen_k, scale=p2.scale, lse=lse2, k_scale=f2.k_scale,
                      v_scale=f2.v_scale, sliding_window=150)
    torch.cuda.synchronize()
    cu_q, cu_k, _, pt = _meta(p2)
    ref2, ref2_lse = oracle.attention(p2.q, f2.kc, f2.vc, pt, cu_q, cu_k, num_q_heads=8, num_kv_heads=2,
                                      head_dim=128, page_size=16, causal=True, scale=p2.scale,
                                      k_scale=f2.ks, v_scale=f2.vs, window_left=149)
    compare(out2, ref2, "fp8 prefill W150", lse_gpu=lse2.T.contiguous(), lse_ref=ref2_lse)
