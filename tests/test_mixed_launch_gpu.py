"""One continuous batch in one launch (pa_mixed_batch): prefill / extend
requests and decode sequences over the same paged pool.  Both halves must
agree with the fp64 oracle within the contract; the prefill half is
bit-identical to pa_prefill (the same work items, computed the same way) and
the decode half agrees with pa_decode within the tolerance (its key ranges
may be cut elsewhere).  Repeated launches reuse one scheduler array."""
import numpy as np
import pytest
import torch

import workloads as W
from pa_harness import bf16_dev, compare, oracle_ref

pytestmark = pytest.mark.gpu


class Mixed:
    """A batch whose first n_pre requests are prefill / extend requests and the
    rest decode sequences (one new token each), sharing one pool and one
    token table; every new token is stored before attention."""

    def __init__(self, seed, pre_cached, pre_ext, dec_len, *, hq=32, hkv=8, d=128, page=16):
        import paged_kv_flashattention_gb300 as pa
        from paged_kv_flashattention_gb300 import metadata
        self.n_pre = len(pre_cached)
        cached = list(pre_cached) + [int(L) - 1 for L in dec_len]
        ext = list(pre_ext) + [1] * len(dec_len)
        self.p = p = W.small_problem(seed, cached, ext, num_q_heads=hq, num_kv_heads=hkv, head_dim=d,
                                     page_size=page)
        dev = torch.device("cuda:0")
        self.dev = dev
        self.k_cache, self.v_cache = bf16_dev(p.k_cache, dev), bf16_dev(p.v_cache, dev)
        pa.store_kv(bf16_dev(p.k_new, dev), bf16_dev(p.v_new, dev), torch.from_numpy(p.slot_mapping).to(dev),
                    self.k_cache, self.v_cache)
        q = bf16_dev(p.q, dev)
        self.tp = int(p.extend_len[:self.n_pre].sum())
        self.q_pre, self.q_dec = q[:self.tp], q[self.tp:]
        tt = torch.from_numpy(p.token_table).to(dev)
        idx = torch.from_numpy(p.table_idx).to(dev)
        self.mp = metadata.prepare(p.cached_len[:self.n_pre], p.extend_len[:self.n_pre], tt, idx[:self.n_pre], page)
        self.md = metadata.prepare(p.cached_len[self.n_pre:], p.extend_len[self.n_pre:], tt, idx[self.n_pre:], page)
        torch.cuda.synchronize()

    def mixed(self, scheduler=None, prefill_ctas=0):
        import paged_kv_flashattention_gb300 as pa
        mp, md = self.mp, self.md
        lse_p = torch.empty((self.p.num_q_heads, self.tp), dtype=torch.float32, device=self.dev)
        lse_d = torch.empty((self.q_dec.shape[0], self.p.num_q_heads), dtype=torch.float32, device=self.dev)
        op, od = pa.mixed_batch(self.q_pre, self.q_dec, self.k_cache, self.v_cache, mp.page_table, mp.cu_seqlens_q,
                                mp.cu_seqlens_k, mp.max_seqlen_q, mp.max_seqlen_k, md.page_table,
                                md.cache_seqlens, md.max_seqlen_k, scale=self.p.scale, lse_prefill=lse_p,
                                lse_decode=lse_d, scheduler=scheduler, prefill_ctas=prefill_ctas)
        torch.cuda.synchronize()
        return op, od, lse_p, lse_d

    def separate(self):
        import paged_kv_flashattention_gb300 as pa
        mp, md = self.mp, self.md
        op = pa.prefill(self.q_pre, self.k_cache, self.v_cache, mp.page_table, mp.cu_seqlens_q, mp.cu_seqlens_k,
                        mp.max_seqlen_q, mp.max_seqlen_k, causal=True, scale=self.p.scale)
        od = pa.decode(self.q_dec, self.k_cache, self.v_cache, md.page_table, md.cache_seqlens, md.max_seqlen_k,
                       scale=self.p.scale)
        torch.cuda.synchronize()
        return op, od

    def check(self, what, prefill_ctas=0):
        import paged_kv_flashattention_gb300 as pa
        op, od, lp, ld = self.mixed(prefill_ctas=prefill_ctas)
        ref, ref_lse = oracle_ref(self.p)                  # every row of the whole batch
        compare(op, ref[:self.tp], f"{what}: prefill half", lse_gpu=lp.T.contiguous(), lse_ref=ref_lse[:self.tp])
        compare(od, ref[self.tp:], f"{what}: decode half", lse_gpu=ld, lse_ref=ref_lse[self.tp:])
        sp, sd = self.separate()
        assert torch.equal(op.view(torch.int16), sp.view(torch.int16)), f"{what}: prefill half != pa_prefill"
        assert (od.float() - sd.float()).abs().max().item() <= 2e-2, f"{what}: decode half vs pa_decode"
        assert pa.device_error() == 0


@pytest.mark.parametrize("page", [16, 1])
@pytest.mark.parametrize("d,hq,hkv", [(128, 32, 8), (64, 16, 4), (128, 8, 4), (64, 32, 4)])
def test_mixed_batch_launch(cuda_device, page, d, hq, hkv):
    rng = np.random.default_rng(600 + page + d + hq)
    dec_len = rng.integers(1, 2000, size=24)
    m = Mixed(610 + page + d + hq, [0, 300, 1000], [700, 130, 5], dec_len, hq=hq, hkv=hkv, d=d, page=page)
    m.check(f"mixed P{page} d{d} g{hq // hkv}")
    m.check(f"mixed P{page} d{d} g{hq // hkv}, prefill on 5 CTAs", prefill_ctas=5)


def test_mixed_batch_repeated_and_edges(cuda_device):
    """Repeated launches on one scheduler array (reset by every launch; the
    prefill share chosen by the kernel, one CTA or three) give the same
    results; decode sequences of one key and long ones."""
    dec_len = np.array([1, 1, 40, 5000, 17, 3000], np.int64)
    m = Mixed(650, [0, 64], [129, 64], dec_len, hq=32, hkv=8, d=128, page=16)
    sched = torch.zeros(4, dtype=torch.int32, device=cuda_device)
    bits = lambda t: t.view(torch.int16) if t.dtype == torch.bfloat16 else t.view(torch.int32)
    firsts = {n: m.mixed(sched, prefill_ctas=n) for n in (0, 1, 3)}
    for n in (0, 1, 3, 0, 1, 3):
        again = m.mixed(sched, prefill_ctas=n)
        # with one prefill share the work items and the decode key ranges are
        # fixed by the batch, whatever CTA takes them: the same bits
        for a, b in zip(firsts[n], again):
            assert torch.equal(bits(a), bits(b))
        # another share may cut the decode rows into other partials: the
        # prefill half is the same, the decode half equal up to rounding
        op, od, lp, ld = firsts[0]
        assert torch.equal(bits(op), bits(again[0])) and torch.equal(bits(lp), bits(again[2]))
        assert (od.float() - again[1].float()).abs().max().item() <= 2e-2
        assert (ld - again[3]).abs().max().item() <= 2e-3
        assert sched.tolist() == [0, 0, 0, 0]
    m.check("edges")
    m.check("edges, prefill on one CTA", prefill_ctas=1)


def test_mixed_metadata_builder(cuda_device):
    """MixedMetadataBuilder (one copy of both halves' lengths, one page-table
    launch for both halves' rows, two buffer sets used in turn): the same
    lengths and page-table rows as preparing each half on its own, and the
    same mixed-batch result, over repeated batches."""
    import paged_kv_flashattention_gb300 as pa
    from paged_kv_flashattention_gb300.metadata import MixedMetadataBuilder
    dec_len = np.array([1, 33, 700, 2500, 16, 17, 4000], np.int64)
    m = Mixed(670, [0, 300, 64], [129, 200, 1], dec_len, hq=32, hkv=8, d=128, page=16)
    p, n = m.p, m.n_pre
    tt = torch.from_numpy(p.token_table).to(cuda_device)
    idx = torch.from_numpy(np.concatenate([p.table_idx[n:], p.table_idx[:n]]).astype(np.int32)).to(cuda_device)
    builder = MixedMetadataBuilder(cuda_device, 4, 16)
    ref = m.mixed()
    sched = torch.zeros(4, dtype=torch.int32, device=cuda_device)
    for rep in range(5):
        mp, md = builder.prepare(p.cached_len[:n], p.extend_len[:n], p.cached_len[n:], p.extend_len[n:], tt, idx,
                                 p.page_size)
        for got, want in ((mp, m.mp), (md, m.md)):
            assert (got.num_seqs, got.max_seqlen_q, got.max_seqlen_k) == (want.num_seqs, want.max_seqlen_q,
                                                                           want.max_seqlen_k)
            for f in ("cu_seqlens_q", "cu_seqlens_k", "cache_seqlens"):
                assert torch.equal(getattr(got, f), getattr(want, f)), f
            cols = want.page_table.shape[1]
            assert torch.equal(got.page_table[:, :cols], want.page_table)
        lse_p = torch.empty((p.num_q_heads, m.tp), dtype=torch.float32, device=cuda_device)
        lse_d = torch.empty((m.q_dec.shape[0], p.num_q_heads), dtype=torch.float32, device=cuda_device)
        out = pa.mixed_batch(m.q_pre, m.q_dec, m.k_cache, m.v_cache, mp.page_table, mp.cu_seqlens_q,
                             mp.cu_seqlens_k, mp.max_seqlen_q, mp.max_seqlen_k, md.page_table, md.cache_seqlens,
                             md.max_seqlen_k, scale=p.scale, lse_prefill=lse_p, lse_decode=lse_d, scheduler=sched)
        torch.cuda.synchronize()
        for a, b in zip((out[0], out[1], lse_p, lse_d), ref):
            assert torch.equal(a.view(torch.int16) if a.dtype == torch.bfloat16 else a.view(torch.int32),
                               b.view(torch.int16) if b.dtype == torch.bfloat16 else b.view(torch.int32))
    assert pa.device_error() == 0


def _bits(t):
    return t.view(torch.int16) if t.dtype == torch.bfloat16 else t.view(torch.int32)


def test_mixed_batch_one_kind_only(cuda_device):
    """With no decode sequences the call is pa_prefill, with no prefill rows it
    is pa_decode: the same bits as those calls."""
    import paged_kv_flashattention_gb300 as pa
    m = Mixed(680, [0, 300], [200, 40], np.array([10, 900, 3000]), hq=32, hkv=8, d=128, page=16)
    mp, md = m.mp, m.md
    sp, sd = m.separate()
    op, od = pa.mixed_batch(m.q_pre, m.q_dec[:0], m.k_cache, m.v_cache, mp.page_table, mp.cu_seqlens_q,
                            mp.cu_seqlens_k, mp.max_seqlen_q, mp.max_seqlen_k, md.page_table[:0],
                            md.cache_seqlens[:0], 1, scale=m.p.scale)
    torch.cuda.synchronize()
    assert od.shape[0] == 0 and torch.equal(_bits(op), _bits(sp))
    zero = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    op, od = pa.mixed_batch(m.q_pre[:0], m.q_dec, m.k_cache, m.v_cache, mp.page_table[:0], zero, zero, 0, 0,
                            md.page_table, md.cache_seqlens, md.max_seqlen_k, scale=m.p.scale)
    torch.cuda.synchronize()
    assert op.shape[0] == 0 and torch.equal(_bits(od), _bits(sd))
    assert pa.device_error() == 0


def test_mixed_batch_decode_rows_without_keys(cuda_device):
    """Decode sequences of length 0 in a mixed launch: O = 0 and lse = -inf for
    them; the other rows still match the oracle."""
    import paged_kv_flashattention_gb300 as pa
    m = Mixed(690, [0, 100], [300, 60], np.array([50, 1200, 7, 2600, 300]), hq=32, hkv=8, d=128, page=16)
    mp, md = m.mp, m.md
    cs = md.cache_seqlens.clone()
    empty = [0, 3]
    cs[empty] = 0
    lse_d = torch.empty((m.q_dec.shape[0], m.p.num_q_heads), dtype=torch.float32, device=cuda_device)
    op, od = pa.mixed_batch(m.q_pre, m.q_dec, m.k_cache, m.v_cache, mp.page_table, mp.cu_seqlens_q,
                            mp.cu_seqlens_k, mp.max_seqlen_q, mp.max_seqlen_k, md.page_table, cs,
                            md.max_seqlen_k, scale=m.p.scale, lse_decode=lse_d)
    torch.cuda.synchronize()
    ref, ref_lse = oracle_ref(m.p)
    keep = [i for i in range(m.q_dec.shape[0]) if i not in empty]
    assert torch.all(od[empty].float() == 0) and torch.all(lse_d[empty] == -float("inf"))
    compare(od[keep], ref[m.tp:][keep], "decode rows with keys", lse_gpu=lse_d[keep], lse_ref=ref_lse[m.tp:][keep])
    compare(op, ref[:m.tp], "prefill half beside empty decode rows")
    assert pa.device_error() == 0


def test_mixed_batch_decode_sliding_window(cuda_device):
    """A sliding window on the decode half (its queries see their sequences'
    last W keys) against the oracle with that window."""
    import oracle
    import paged_kv_flashattention_gb300 as pa
    from oracle_pins import _meta, stored_caches
    m = Mixed(700, [0, 64], [250, 100], np.array([40, 300, 1500, 5000, 257]), hq=32, hkv=8, d=128, page=16)
    mp, md = m.mp, m.md
    W = 256
    lse_d = torch.empty((m.q_dec.shape[0], m.p.num_q_heads), dtype=torch.float32, device=cuda_device)
    op, od = pa.mixed_batch(m.q_pre, m.q_dec, m.k_cache, m.v_cache, mp.page_table, mp.cu_seqlens_q,
                            mp.cu_seqlens_k, mp.max_seqlen_q, mp.max_seqlen_k, md.page_table, md.cache_seqlens,
                            md.max_seqlen_k, scale=m.p.scale, lse_decode=lse_d, decode_sliding_window=W)
    torch.cuda.synchronize()
    p = m.p
    cu_q, cu_k, _, pt = _meta(p)
    kc, vc = stored_caches(p)
    rows = np.stack(np.meshgrid(np.arange(m.tp, p.q.shape[0]), np.arange(p.num_q_heads), indexing="ij"),
                    -1).reshape(-1, 2).astype(np.int64)
    ref, ref_lse = oracle.attention(p.q, kc, vc, pt, cu_q, cu_k, num_q_heads=p.num_q_heads,
                                    num_kv_heads=p.num_kv_heads, head_dim=p.head_dim, page_size=p.page_size,
                                    causal=p.causal, scale=p.scale, window_left=W - 1, rows=rows)
    nd = m.q_dec.shape[0]
    compare(od.reshape(nd * p.num_q_heads, -1), ref, "decode half, window 256", lse_gpu=lse_d.reshape(-1),
            lse_ref=ref_lse)
    ref_full, _ = oracle_ref(p)
    compare(op, ref_full[:m.tp], "prefill half (no window)")
    assert pa.device_error() == 0


@pytest.mark.parametrize("d,hq,hkv,page", [(128, 32, 8, 16), (64, 16, 4, 1)])
def test_mixed_batch_fp8(cuda_device, d, hq, hkv, page):
    """One mixed launch over FP8 (E4M3) pools with per-KV-head scales: both
    halves against the fp64 oracle on the same codes, the prefill half
    bit-identical to pa_prefill over the same pools."""
    import oracle
    import paged_kv_flashattention_gb300 as pa
    from paged_kv_flashattention_gb300 import metadata
    from oracle_pins import _meta
    from test_fp8_gpu import FP8Problem
    rng = np.random.default_rng(710 + d + page)
    dec_len = rng.integers(1, 3000, size=12)
    pre_c, pre_e = [0, 500], [300, 77]
    p = W.small_problem(711 + d + page, pre_c + [int(L) - 1 for L in dec_len], pre_e + [1] * len(dec_len),
                        num_q_heads=hq, num_kv_heads=hkv, head_dim=d, page_size=page)
    f = FP8Problem(p, cuda_device, 712 + d)
    n = len(pre_c)
    tp = int(p.extend_len[:n].sum())
    tt = torch.from_numpy(p.token_table).to(cuda_device)
    idx = torch.from_numpy(p.table_idx).to(cuda_device)
    mp = metadata.prepare(p.cached_len[:n], p.extend_len[:n], tt, idx[:n], page)
    md = metadata.prepare(p.cached_len[n:], p.extend_len[n:], tt, idx[n:], page)
    lse_p = torch.empty((hq, tp), dtype=torch.float32, device=cuda_device)
    lse_d = torch.empty((len(dec_len), hq), dtype=torch.float32, device=cuda_device)
    sc = dict(k_scale=f.k_scale, v_scale=f.v_scale)
    op, od = pa.mixed_batch(f.q[:tp], f.q[tp:], f.k_cache, f.v_cache, mp.page_table, mp.cu_seqlens_q,
                            mp.cu_seqlens_k, mp.max_seqlen_q, mp.max_seqlen_k, md.page_table, md.cache_seqlens,
                            md.max_seqlen_k, scale=p.scale, lse_prefill=lse_p, lse_decode=lse_d, **sc)
    torch.cuda.synchronize()
    cu_q, cu_k, _, pt = _meta(p)
    ref, ref_lse = oracle.attention(p.q, f.kc, f.vc, pt, cu_q, cu_k, num_q_heads=hq, num_kv_heads=hkv,
                                    head_dim=d, page_size=page, causal=True, scale=p.scale, k_scale=f.ks,
                                    v_scale=f.vs)
    compare(op, ref[:tp], f"fp8 mixed d{d} P{page}: prefill half", lse_gpu=lse_p.T.contiguous(), lse_ref=ref_lse[:tp])
    compare(od, ref[tp:], f"fp8 mixed d{d} P{page}: decode half", lse_gpu=lse_d, lse_ref=ref_lse[tp:])
    sp = pa.prefill(f.q[:tp], f.k_cache, f.v_cache, mp.page_table, mp.cu_seqlens_q, mp.cu_seqlens_k,
                    mp.max_seqlen_q, mp.max_seqlen_k, causal=True, scale=p.scale, **sc)
    torch.cuda.synchronize()
    assert torch.equal(op.view(torch.int16), sp.view(torch.int16))
    assert pa.device_error() == 0
