"""GPU parity of varlen prefill / extend attention (tcgen05 kernel) against the
fp64 oracle: max abs <= 2e-2, mean abs <= 1e-3 on bf16 outputs, lse within
2e-3, on the workloads and the edge-case matrix."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from pa_harness import DeviceProblem, compare, oracle_ref

pytestmark = pytest.mark.gpu


def _prefill_check(p, dev, what="", rows=None):
    d = DeviceProblem(p, dev)
    d.store()
    out, lse = d.prefill()
    torch.cuda.synchronize()
    if rows is None:
        ref, ref_lse = oracle_ref(p)
        return compare(out, ref, what or p.name, lse_gpu=lse[:, :ref.shape[0]].T.contiguous(),
                       lse_ref=ref_lse)
    ref, ref_lse = oracle_ref(p, rows=rows)
    o = out[torch.from_numpy(rows[:, 0]).to(dev), torch.from_numpy(rows[:, 1]).to(dev)]
    l = lse[torch.from_numpy(rows[:, 1]).to(dev), torch.from_numpy(rows[:, 0]).to(dev)]
    return compare(o, ref, what or p.name, lse_gpu=l, lse_ref=ref_lse)


def test_varlen_prefill_16x512_full(cuda_device):
    """16 requests x 512 prompt tokens, no cache hit, Hq 32 / Hkv 8, d 128, page 16."""
    _prefill_check(W.config(3), cuda_device)


def _sample_rows(p, frac, seed):
    """Every request's first and last 3 rows, plus a random fraction; all heads."""
    rng = np.random.default_rng(seed)
    cu = np.concatenate([[0], np.cumsum(p.extend_len)])
    toks = set()
    for b in range(p.num_seqs):
        for t in list(range(cu[b], min(cu[b] + 3, cu[b + 1]))) + list(range(max(cu[b], cu[b + 1] - 3), cu[b + 1])):
            toks.add(int(t))
    T = int(cu[-1])
    toks.update(int(t) for t in rng.choice(T, size=max(1, int(T * frac)), replace=False))
    toks = np.array(sorted(toks), np.int64)
    heads = np.arange(p.num_q_heads, dtype=np.int64)
    return np.stack(np.meshgrid(toks, heads, indexing="ij"), axis=-1).reshape(-1, 2)


@pytest.mark.parametrize("variant", [None, "p1"])
def test_extend_partial_hit(cuda_device, variant):
    """8 requests, cached U[0,4096], extend U[64,1024], end-aligned causal mask;
    page size 16 and the token-granular page size 1 table."""
    p = W.config(4, variant)
    _prefill_check(p, cuda_device, rows=_sample_rows(p, 0.25, 4), what=p.name)


EDGE = [
    ([0, 0, 0, 0, 0], [1, 15, 16, 17, 129]),            # no hit; lengths at page/tile edges
    ([3, 16, 127, 128, 1000], [1, 16, 1, 129, 255]),   # cached prefix + extend
    ([0, 7, 0], [300, 0, 128]),                          # an empty request in the batch
]


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("hq,hkv", [(4, 4), (8, 4), (16, 4), (32, 4)])
@pytest.mark.parametrize("page", [1, 16])
def test_prefill_edge_matrix(cuda_device, d, hq, hkv, page):
    for n, (cached, ext) in enumerate(EDGE):
        p = W.small_problem(2000 + 7 * n + d + hq + page, cached, ext, num_q_heads=hq,
                            num_kv_heads=hkv, head_dim=d, page_size=page)
        _prefill_check(p, cuda_device, what=f"d{d} g{hq // hkv} P{page} case{n}")


@pytest.mark.parametrize("page", [1, 16])
def test_prefill_non_causal(cuda_device, page):
    p = W.build("noncausal", cached_len=[0, 40, 200], extend_len=[33, 130, 64], num_q_heads=8,
                num_kv_heads=2, head_dim=128, page_size=page, seed=3001, causal=False)
    _prefill_check(p, cuda_device, what=f"non-causal P{page}")


def test_prefill_deterministic(cuda_device):
    p = W.config(3)
    d = DeviceProblem(p, cuda_device)
    d.store()
    a, la = d.prefill()
    b, lb = d.prefill()
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    assert torch.equal(la, lb)


@pytest.mark.parametrize("page", [1, 16])
def test_prefill_physical_permutation_invariance(cuda_device, page):
    """The same logical K/V on other physical pages (slots for page size 1)
    gives the identical output and LSE: the page-table indexing is exact and
    the kernel's arithmetic depends on the logical order only."""
    import paged_kv_flashattention_gb300 as pa
    p = W.small_problem(91 + page, [300, 17, 0, 1000], [40, 130, 200, 7], num_q_heads=16,
                        num_kv_heads=4, head_dim=128, page_size=page)
    d = DeviceProblem(p, cuda_device)
    d.store()
    out1, lse1 = d.prefill()
    m = d.metadata()
    # the poison page stays last, so unused table entries still point at it
    perm = np.concatenate([np.random.default_rng(4).permutation(p.num_pages - 1), [p.num_pages - 1]])
    permt = torch.from_numpy(perm).to(cuda_device)
    kc2 = torch.empty_like(d.k_cache)
    vc2 = torch.empty_like(d.v_cache)
    kc2[permt] = d.k_cache
    vc2[permt] = d.v_cache
    tt = p.token_table.astype(np.int64)
    tt2 = (perm[tt // page] * page + tt % page).astype(np.int32)
    pt2 = pa.build_page_table(torch.from_numpy(tt2).to(cuda_device), d.table_idx, m.max_seqlen_k, page)
    lse2 = torch.empty_like(lse1)
    out2 = pa.prefill(d.q, kc2, vc2, pt2, m.cu_seqlens_q, m.cu_seqlens_k, m.max_seqlen_q,
                      m.max_seqlen_k, causal=True, scale=p.scale, lse=lse2)
    torch.cuda.synchronize()
    assert torch.equal(out1.view(torch.int16), out2.view(torch.int16))
    assert torch.equal(lse1, lse2)


def test_decode_via_prefill_matches_decode(cuda_device):
    """A decode batch run through prefill (Lq = 1 per request, cu_seqlens_q =
    arange) agrees with the decode kernel and with the oracle."""
    p = W.config(2)
    d = DeviceProblem(p, cuda_device)
    d.store()
    o_dec, l_dec = d.decode()
    o_pre, l_pre = d.prefill()
    torch.cuda.synchronize()
    ref, ref_lse = oracle_ref(p)
    compare(o_pre, ref, "decode through prefill", lse_gpu=l_pre.T.contiguous(), lse_ref=ref_lse)
    diff = (o_dec.float() - o_pre.float()).abs().max().item()
    assert diff <= 2e-2


def test_prefill_skewed_batch(cuda_device):
    """One long request among many short ones: most (tile, request) work
    slots of the longest-tile-first order are empty and the work counter
    skips them; every row still agrees with the oracle."""
    cached = [0] * 41 + [300]
    ext = [1, 2, 3, 17, 5] * 8 + [9, 1500]
    p = W.build("skewed", cached_len=cached, extend_len=ext, num_q_heads=8, num_kv_heads=2,
                head_dim=128, page_size=16, seed=3101)
    _prefill_check(p, cuda_device, rows=_sample_rows(p, 0.2, 5), what="skewed batch")


def test_prefill_scheduler_counters_are_reset(cuda_device):
    """The caller's scheduler array is left at zero by every launch, so one
    array serves many launches in a row: each output is bit-identical to the
    first launch's, and the array reads back as zeros at the end."""
    import paged_kv_flashattention_gb300 as pa
    p = W.small_problem(3111, [0, 20, 0], [130, 40, 7], num_q_heads=8, num_kv_heads=2,
                        head_dim=64, page_size=16)
    d = DeviceProblem(p, cuda_device)
    d.store()
    m = d.metadata()
    sched = torch.zeros(2, dtype=torch.int32, device=cuda_device)
    first = None
    for i in range(64):
        out = pa.prefill(d.q, d.k_cache, d.v_cache, m.page_table, m.cu_seqlens_q, m.cu_seqlens_k,
                         m.max_seqlen_q, m.max_seqlen_k, causal=True, scale=p.scale, scheduler=sched)
        if first is None:
            first = out.clone()
        else:
            assert torch.equal(first.view(torch.int16), out.view(torch.int16)), f"launch {i} differs"
    torch.cuda.synchronize()
    assert sched.tolist() == [0, 0]
    ref, _ = oracle_ref(p)
    compare(out, ref, "after counter reuse")


def test_prefill_concurrent_streams(cuda_device):
    """Two prefill launches in flight at once on two streams use separate
    scheduler arrays (the binding keeps one per stream) and both agree with
    the oracle."""
    import paged_kv_flashattention_gb300 as pa
    probs = [W.config(3), W.small_problem(3121, [0, 500, 64], [700, 300, 900], num_q_heads=32,
                                          num_kv_heads=8, head_dim=128, page_size=16)]
    devs = [DeviceProblem(p, cuda_device) for p in probs]
    for d in devs:
        d.store()
    metas = [d.metadata() for d in devs]
    torch.cuda.synchronize()
    streams = [torch.cuda.Stream(cuda_device) for _ in devs]
    outs = []
    for d, m, s in zip(devs, metas, streams):
        with torch.cuda.stream(s):
            outs.append(pa.prefill(d.q, d.k_cache, d.v_cache, m.page_table, m.cu_seqlens_q,
                                   m.cu_seqlens_k, m.max_seqlen_q, m.max_seqlen_k, causal=True,
                                   scale=d.p.scale))
    torch.cuda.synchronize()
    ref0, _ = oracle_ref(probs[0])
    compare(outs[0], ref0, "stream 0")
    rows = _sample_rows(probs[1], 0.1, 6)
    ref1, _ = oracle_ref(probs[1], rows=rows)
    o1 = outs[1][torch.from_numpy(rows[:, 0]).to(cuda_device), torch.from_numpy(rows[:, 1]).to(cuda_device)]
    compare(o1, ref1, "stream 1")


def test_prefill_and_decode_overlapped(cuda_device):
    """Prefill on a few SMs with decode launched as its programmatic
    dependent on the rest (the benchmark's schedule): both agree with the
    oracle, and so does a decode capped to a handful of CTAs."""
    import paged_kv_flashattention_gb300 as pa
    pp, pd = W.config(3), W.config(2)
    dp, dd = DeviceProblem(pp, cuda_device), DeviceProblem(pd, cuda_device)
    dp.store()
    dd.store()
    mp, md = dp.metadata(), dd.metadata()
    torch.cuda.synchronize()
    sms = torch.cuda.get_device_properties(cuda_device).multi_processor_count
    out_p = pa.prefill(dp.q, dp.k_cache, dp.v_cache, mp.page_table, mp.cu_seqlens_q, mp.cu_seqlens_k,
                       mp.max_seqlen_q, mp.max_seqlen_k, causal=True, scale=pp.scale, max_ctas=12)
    out_d = pa.decode(dd.q, dd.k_cache, dd.v_cache, md.page_table, md.cache_seqlens, md.max_seqlen_k,
                      scale=pd.scale, max_ctas=2 * (sms - 12), overlap_previous=True)
    small = pa.decode(dd.q, dd.k_cache, dd.v_cache, md.page_table, md.cache_seqlens, md.max_seqlen_k,
                      scale=pd.scale, max_ctas=5)
    torch.cuda.synchronize()
    ref_p, _ = oracle_ref(pp)
    ref_d, _ = oracle_ref(pd)
    compare(out_p, ref_p, "prefill on 12 SMs")
    compare(out_d, ref_d, "decode overlapped with prefill")
    compare(small, ref_d, "decode on 5 CTAs")


def test_prefill_device_lengths_out_of_bounds(cuda_device):
    """cu_seqlens on the device that break the call's bounds (rows past
    total_q, more keys than max_seqlen_k) skip that request: nothing is read
    or written out of bounds, PA_DEVERR_SEQLENS is raised, and the other
    requests are still exact."""
    import paged_kv_flashattention_gb300 as pa
    p = W.small_problem(940, [100, 0, 40, 7], [50, 130, 20, 9], num_q_heads=8, num_kv_heads=2, head_dim=128,
                        page_size=16)
    d = DeviceProblem(p, cuda_device)
    d.store()
    m = d.metadata()
    ref, _ = oracle_ref(p)
    cu_q, cu_k = m.cu_seqlens_q.clone(), m.cu_seqlens_k.clone()
    # request 1: 200 more keys than max_seqlen_k allows (request 2 keeps its length)
    cu_k[2:] += 200
    # request 3: its rows run past total_q
    cu_q[4] += 64
    Tq = d.q.shape[0]
    out = torch.zeros_like(d.q)
    pa.device_error()
    pa.prefill(d.q, d.k_cache, d.v_cache, m.page_table, cu_q, cu_k, m.max_seqlen_q, m.max_seqlen_k, causal=True,
               scale=p.scale, out=out)
    torch.cuda.synchronize()
    assert pa.device_error() & 2
    cq = np.concatenate([[0], np.cumsum(p.extend_len)])
    for b in (0, 2):
        rows = slice(int(cq[b]), int(cq[b + 1]))
        compare(out[rows], ref[rows], f"request {b} beside out-of-bounds lengths")
    assert torch.all(out[int(cq[1]):int(cq[2])] == 0) and torch.all(out[int(cq[3]):Tq] == 0)
