"""GPU parity of block-sparse masks in prefill / extend attention (a byte per
block of 128 of a request's query rows x 128 keys; a zero block is hidden, on
top of the causal and window limits) against the fp64 oracle: bf16 and FP8
pools, page sizes 16 and 1, causal and not, with and without a window, and
the closed forms (an all-ones mask changes nothing, an all-zero mask leaves
every row empty)."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from oracle_pins import _meta, stored_caches
from pa_harness import DeviceProblem, compare

pytestmark = pytest.mark.gpu


def _oracle(p, mask, window=0, rows=None, caches=None, scales=None):
    cu_q, cu_k, _, pt = _meta(p)
    kc, vc = caches if caches is not None else stored_caches(p)
    ks, vs = scales if scales is not None else (None, None)
    return oracle.attention(p.q, kc, vc, pt, cu_q, cu_k, num_q_heads=p.num_q_heads,
                            num_kv_heads=p.num_kv_heads, head_dim=p.head_dim, page_size=p.page_size,
                            causal=p.causal, scale=p.scale, window_left=window - 1, rows=rows,
                            block_mask=mask, k_scale=ks, v_scale=vs)


def _prefill(d, p, dev, mask_t, window=0, **kw):
    import paged_kv_flashattention_gb300 as pa
    m = d.metadata() if hasattr(d, "metadata") else d.meta
    Tq = d.q.shape[0]
    lse = torch.empty((p.num_q_heads, max(Tq, 1)), dtype=torch.float32, device=dev)
    out = pa.prefill(d.q, d.k_cache, d.v_cache, m.page_table, m.cu_seqlens_q, m.cu_seqlens_k,
                     m.max_seqlen_q, m.max_seqlen_k, causal=p.causal, scale=p.scale, lse=lse,
                     page_size=p.page_size, sliding_window=window, block_mask=mask_t, **kw)
    torch.cuda.synchronize()
    return out, lse


def _check(p, dev, mask, window=0, what=""):
    d = DeviceProblem(p, dev)
    d.store()
    out, lse = _prefill(d, p, dev, torch.from_numpy(mask).to(dev), window)
    ref, ref_lse = _oracle(p, mask, window)
    compare(out, ref, what, lse_gpu=lse[:, :ref.shape[0]].T.contiguous(), lse_ref=ref_lse)
    import paged_kv_flashattention_gb300 as pa
    assert pa.device_error() == 0


CASES = [
    ([0, 0, 0], [300, 129, 17]),             # no cache hit, blocks cut inside the prompts
    ([200, 1000, 3, 0], [160, 40, 260, 0]),  # cached prefix + extend, an empty request
]


@pytest.mark.parametrize("density", [0.3, 0.7])
@pytest.mark.parametrize("page", [1, 16])
def test_prefill_block_mask(cuda_device, density, page):
    rng = np.random.default_rng(int(100 * density) + page)
    for n, (cached, ext) in enumerate(CASES):
        for hq, hkv, d in ((8, 2, 128), (4, 4, 64)):
            p = W.small_problem(4100 + 11 * n + page + hq, cached, ext, num_q_heads=hq, num_kv_heads=hkv,
                                head_dim=d, page_size=page)
            mask = W.block_mask(rng, p.extend_len, p.device_len, density=density, keep_diagonal=(n == 0))
            _check(p, cuda_device, mask, what=f"mask {density} P{page} d{d} g{hq // hkv} case{n}")


def test_prefill_block_mask_with_window_and_non_causal(cuda_device):
    rng = np.random.default_rng(4200)
    p = W.small_problem(4201, [200, 1000, 3], [160, 40, 260], num_q_heads=8, num_kv_heads=2, head_dim=128,
                        page_size=16)
    _check(p, cuda_device, W.block_mask(rng, p.extend_len, p.device_len, 0.6), window=300, what="mask + W300")
    q = W.build("noncausal-mask", cached_len=[0, 300, 200], extend_len=[33, 130, 300], num_q_heads=8,
                num_kv_heads=2, head_dim=128, page_size=16, seed=4202, causal=False)
    _check(q, cuda_device, W.block_mask(rng, q.extend_len, q.device_len, 0.5, keep_diagonal=False),
           what="non-causal mask")


def test_prefill_block_mask_closed_forms(cuda_device):
    """All ones: bit-identical to no mask (the masked kernel does the same
    arithmetic).  All zeros: every output row is 0 and every lse -inf."""
    import paged_kv_flashattention_gb300 as pa
    p = W.small_problem(4300, [200, 0, 57], [160, 300, 70], num_q_heads=8, num_kv_heads=2, head_dim=128,
                        page_size=16)
    d = DeviceProblem(p, cuda_device)
    d.store()
    nq = -(-int(p.extend_len.max()) // 128)
    nk = -(-int(p.device_len.max()) // 128)
    ones = torch.ones((p.num_seqs, nq, nk), dtype=torch.uint8, device=cuda_device)
    plain, plain_lse = _prefill(d, p, cuda_device, None)
    o1, l1 = _prefill(d, p, cuda_device, ones)
    assert torch.equal(plain.view(torch.int16), o1.view(torch.int16)), "all-ones mask changed the output"
    assert torch.equal(plain_lse, l1)
    o0, l0 = _prefill(d, p, cuda_device, torch.zeros_like(ones))
    Tq = d.q.shape[0]
    assert torch.all(o0.float() == 0) and torch.all(l0[:, :Tq] == -float("inf"))
    assert pa.device_error() == 0


def test_prefill_block_mask_fp8(cuda_device):
    from test_fp8_gpu import FP8Problem
    rng = np.random.default_rng(4400)
    for page in (16, 1):
        p = W.small_problem(4401 + page, [200, 1000, 3], [160, 40, 260], num_q_heads=8, num_kv_heads=2,
                            head_dim=128, page_size=page)
        f = FP8Problem(p, cuda_device, 4402 + page)
        mask = W.block_mask(rng, p.extend_len, p.device_len, 0.5)
        out, lse = _prefill(f, p, cuda_device, torch.from_numpy(mask).to(cuda_device),
                            k_scale=f.k_scale, v_scale=f.v_scale)
        ref, ref_lse = _oracle(p, mask, caches=(f.kc, f.vc), scales=(f.ks, f.vs))
        compare(out, ref, f"fp8 mask P{page}", lse_gpu=lse[:, :ref.shape[0]].T.contiguous(), lse_ref=ref_lse)


def test_prefill_block_mask_extend_workload(cuda_device):
    """The extend-with-partial-hit workload (8 requests, prefixes up to 4096)
    under a half-density mask, on sampled rows at full size."""
    rng = np.random.default_rng(4500)
    p = W.config(4)
    mask = W.block_mask(rng, p.extend_len, p.device_len, 0.5)
    d = DeviceProblem(p, cuda_device)
    d.store()
    out, lse = _prefill(d, p, cuda_device, torch.from_numpy(mask).to(cuda_device))
    Tq = d.q.shape[0]
    rows = np.stack([rng.choice(Tq, 400), rng.integers(0, p.num_q_heads, 400)], 1).astype(np.int64)
    ref, ref_lse = _oracle(p, mask, rows=rows)
    rt = torch.from_numpy(rows).to(cuda_device)
    compare(out[rt[:, 0], rt[:, 1]], ref, "extend workload, mask 0.5", lse_gpu=lse[rt[:, 1], rt[:, 0]],
            lse_ref=ref_lse)
