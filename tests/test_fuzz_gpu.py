"""Seeded random parity cases that mix the features the other GPU tests cover
one at a time: prefill or decode, bf16 or FP8 pools, page size 1 or 16,
head_dim 64 or 128, GQA groups 1 to 8, sliding windows, causal or not,
forced split sizes, prefill requests with no new tokens.  Each case is checked against the fp64 oracle with the
contract's tolerances (max abs <= 2e-2, mean abs <= 1e-3, lse within 2e-3)."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from oracle_pins import _meta, stored_caches
from pa_harness import DeviceProblem, compare

pytestmark = pytest.mark.gpu

HEADS = [(4, 4), (8, 4), (16, 4), (32, 4), (8, 2), (32, 8), (12, 6)]


def _case(seed, big=False):
    """One random configuration (a dict), drawn from its own seed; ``big``
    draws longer contexts and larger batches."""
    rng = np.random.default_rng(seed)
    scale = 4 if big else 1
    c = {
        "op": ("prefill", "decode")[int(rng.integers(0, 2))],
        "fp8": bool(rng.integers(0, 3) == 0),
        "page": (1, 16)[int(rng.integers(0, 2))],
        "d": (64, 128)[int(rng.integers(0, 2))],
        "heads": HEADS[int(rng.integers(0, len(HEADS)))],
        "window": int(rng.integers(1, 400)) if rng.integers(0, 3) == 0 else 0,
        "causal": bool(rng.integers(0, 5) != 0),
        "chunk": (0, 16, 64)[int(rng.integers(0, 3))],
        "B": int(rng.integers(1, 7 * scale)),
    }
    if c["op"] == "decode":
        c["cached"] = [int(x) for x in rng.integers(0, 1500 * scale, size=c["B"])]
        c["extend"] = [1] * c["B"]
    else:
        c["B"] = min(c["B"], 8)                 # keeps the oracle's share of the test short
        c["cached"] = [int(x) if rng.integers(0, 3) else 0 for x in rng.integers(0, 700 * scale, size=c["B"])]
        c["extend"] = [int(x) for x in rng.integers(1, 300 if not big else 500, size=c["B"])]
        if c["B"] > 1 and rng.integers(0, 3) == 0:     # a request with no new tokens
            c["extend"][int(rng.integers(0, c["B"]))] = 0
    return c


def _problem(c, seed):
    hq, hkv = c["heads"]
    return W.build(f"fuzz{seed}", cached_len=c["cached"], extend_len=c["extend"], num_q_heads=hq,
                   num_kv_heads=hkv, head_dim=c["d"], page_size=c["page"], seed=seed,
                   causal=c["causal"] or c["op"] == "decode")


@pytest.mark.parametrize("seed", list(range(7000, 7032)) + [-s for s in range(7100, 7112)])
def test_fuzz_parity(cuda_device, seed):
    """A negative seed draws a big case (its absolute value is the seed)."""
    import paged_kv_flashattention_gb300 as pa
    big = seed < 0
    seed = abs(seed)
    c = _case(seed, big)
    p = _problem(c, seed)
    pa.device_error()                       # start from a clear device error word
    what = f"fuzz {seed}: {c}"
    dev = cuda_device
    win = c["window"]
    if c["fp8"]:
        from test_fp8_gpu import FP8Problem
        f = FP8Problem(p, dev, seed + 1)
        q, kd, vd, m = f.q, f.k_cache, f.v_cache, f.meta
        kc, vc, ks, vs = f.kc, f.vc, f.ks, f.vs
        extra = {"k_scale": f.k_scale, "v_scale": f.v_scale}
    else:
        d = DeviceProblem(p, dev)
        d.store()
        q, kd, vd, m = d.q, d.k_cache, d.v_cache, d.metadata()
        kc, vc = stored_caches(p)
        ks = vs = None
        extra = {}
    cu_q, cu_k, _, pt = _meta(p)
    ref, ref_lse = oracle.attention(p.q, kc, vc, pt, cu_q, cu_k, num_q_heads=p.num_q_heads,
                                    num_kv_heads=p.num_kv_heads, head_dim=p.head_dim,
                                    page_size=p.page_size, causal=p.causal, scale=p.scale,
                                    k_scale=ks, v_scale=vs, window_left=win - 1 if win > 0 else -1)
    if c["op"] == "decode":
        lse = torch.empty((p.num_seqs, p.num_q_heads), dtype=torch.float32, device=dev)
        out = pa.decode(q, kd, vd, m.page_table, m.cache_seqlens, m.max_seqlen_k, scale=p.scale,
                        lse=lse, kv_chunk=c["chunk"], sliding_window=win, **extra)
        torch.cuda.synchronize()
        compare(out, ref.reshape(out.shape), what, lse_gpu=lse, lse_ref=ref_lse.reshape(lse.shape))
    else:
        Tq = q.shape[0]
        lse = torch.empty((p.num_q_heads, max(Tq, 1)), dtype=torch.float32, device=dev)
        out = pa.prefill(q, kd, vd, m.page_table, m.cu_seqlens_q, m.cu_seqlens_k, m.max_seqlen_q,
                         m.max_seqlen_k, causal=p.causal, scale=p.scale, lse=lse,
                         sliding_window=win, **extra)
        torch.cuda.synchronize()
        compare(out, ref, what, lse_gpu=lse[:, :ref.shape[0]].T.contiguous(), lse_ref=ref_lse)
    assert pa.device_error() == 0, what
