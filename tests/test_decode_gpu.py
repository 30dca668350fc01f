"""GPU parity of split-KV decode and the LSE combine against the fp64 oracle
(max abs <= 2e-2, mean abs <= 1e-3 on bf16 outputs; lse within 2e-3)."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from oracle import online
from pa_harness import DeviceProblem, compare, oracle_ref

pytestmark = pytest.mark.gpu


def _decode_check(p, dev, kv_chunk=0, what=""):
    d = DeviceProblem(p, dev)
    d.store()
    out, lse = d.decode(kv_chunk=kv_chunk)
    torch.cuda.synchronize()
    ref, ref_lse = oracle_ref(p)
    return compare(out, ref, what or p.name, lse_gpu=lse, lse_ref=ref_lse)


def test_tiny_decode(cuda_device):
    _decode_check(W.config(1), cuda_device)


@pytest.mark.parametrize("kv_chunk", [0, 16, 48])
def test_tiny_decode_forced_splits(cuda_device, kv_chunk):
    _decode_check(W.config(1), cuda_device, kv_chunk=kv_chunk)


def test_llama32_1b_decode_full(cuda_device):
    """B=64, Hq 32 / Hkv 8, d 64, contexts U[128, 4096], every output row."""
    _decode_check(W.config(2), cuda_device)


EDGE_LENGTHS = [1, 15, 16, 17, 33, 100, 257]


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("hq,hkv", [(4, 4), (8, 4), (16, 4), (32, 4), (12, 6)])
@pytest.mark.parametrize("page", [1, 16])
def test_decode_edge_matrix(cuda_device, d, hq, hkv, page):
    Lk = np.array(EDGE_LENGTHS, np.int32)
    p = W.small_problem(1000 + d + hq + page, Lk - 1, np.ones_like(Lk), num_q_heads=hq,
                        num_kv_heads=hkv, head_dim=d, page_size=page)
    for chunk in (0, 16, 64):
        _decode_check(p, cuda_device, kv_chunk=chunk, what=f"d{d} g{hq // hkv} P{page} C{chunk}")


def test_decode_empty_sequences(cuda_device):
    """cache_seqlens = 0 (a padded dummy request): O = 0, lse = -inf; the other
    rows are unaffected."""
    p = W.small_problem(77, [0, 20, 0, 5], [0, 1, 0, 1], num_q_heads=8, num_kv_heads=2,
                        head_dim=128, page_size=16)
    # decode rows: requests 0 and 2 have no keys at all
    import paged_kv_flashattention_gb300 as pa
    d = DeviceProblem(p, cuda_device)
    d.store()
    cs = torch.tensor(p.device_len, dtype=torch.int32, device=cuda_device)
    pt = pa.build_page_table(d.token_table, d.table_idx, int(p.device_len.max()), 16)
    q = torch.from_numpy(W.normal_bf16(np.random.default_rng(1), (4, 8, 128)).view(np.int16)).to(cuda_device).view(torch.bfloat16)
    for chunk in (0, 16):
        lse = torch.empty((4, 8), dtype=torch.float32, device=cuda_device)
        out = pa.decode(q, d.k_cache, d.v_cache, pt, cs, int(p.device_len.max()), scale=p.scale,
                        lse=lse, kv_chunk=chunk)
        kc, vc = p.k_cache.copy(), p.v_cache.copy()
        row = 2 * 128
        oracle.store_kv(p.k_new.reshape(-1, row), p.v_new.reshape(-1, row), p.slot_mapping,
                        kc.reshape(-1, row), vc.reshape(-1, row))
        qh = q.view(torch.int16).cpu().numpy().view(np.uint16)
        ptn = oracle.page_table_from_token_table(p.token_table, p.table_idx, int(p.device_len.max()), 16)
        ref, ref_lse = oracle.decode(qh, kc, vc, ptn, p.device_len, num_q_heads=8, num_kv_heads=2,
                                     head_dim=128, page_size=16, scale=p.scale)
        compare(out, ref, f"empty seqs C{chunk}", lse_gpu=lse, lse_ref=ref_lse)
        o = out.float().cpu().numpy()
        assert np.all(o[[0, 2]] == 0.0)


def test_decode_deterministic(cuda_device):
    p = W.config(2)
    d = DeviceProblem(p, cuda_device)
    d.store()
    a, la = d.decode()
    b, lb = d.decode()
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    assert torch.equal(la, lb)


def test_decode_physical_permutation_invariance(cuda_device):
    """Re-packing the same logical K/V on other physical pages gives the
    identical output (the kernel's arithmetic depends on logical order only)."""
    import paged_kv_flashattention_gb300 as pa
    p = W.small_problem(88, [300, 17, 64, 1000], [1, 1, 1, 1], num_q_heads=32, num_kv_heads=8,
                        head_dim=128, page_size=16)
    d = DeviceProblem(p, cuda_device)
    d.store()
    out1, _ = d.decode(kv_chunk=64)
    perm = np.concatenate([np.random.default_rng(3).permutation(p.num_pages - 1), [p.num_pages - 1]])
    permt = torch.from_numpy(perm).to(cuda_device)
    kc2 = torch.empty_like(d.k_cache)
    vc2 = torch.empty_like(d.v_cache)
    kc2[permt] = d.k_cache
    vc2[permt] = d.v_cache
    tt = p.token_table.astype(np.int64)
    tt2 = (perm[tt // 16] * 16 + tt % 16).astype(np.int32)
    pt2 = pa.build_page_table(torch.from_numpy(tt2).to(cuda_device), d.table_idx,
                              int(p.device_len.max()), 16)
    cs = torch.from_numpy(p.device_len).to(cuda_device)
    out2 = pa.decode(d.q, kc2, vc2, pt2, cs, int(p.device_len.max()), scale=p.scale, kv_chunk=64)
    torch.cuda.synchronize()
    assert torch.equal(out1.view(torch.int16), out2.view(torch.int16))


def test_decode_workspace_reuse(cuda_device):
    """One zero-filled workspace serves a run of calls with other length mixes
    and split sizes.  Outputs start as NaN, so a split row whose merge did not
    run (an arrival count left over from an earlier call) shows up."""
    import paged_kv_flashattention_gb300 as pa
    rng = np.random.default_rng(5)
    cases = []
    for i, chunk in enumerate((16, 0, 64, 16, 32)):
        L = rng.integers(1, 900, size=12).astype(np.int32)
        p = W.small_problem(500 + i, L - 1, np.ones_like(L), num_q_heads=16, num_kv_heads=4,
                            head_dim=128, page_size=16)
        d = DeviceProblem(p, cuda_device)
        d.store()
        cases.append((p, d, chunk, oracle_ref(p)))
    need = max(pa.decode_workspace_size(d.q.shape, d.k_cache, d.metadata().max_seqlen_k, kv_chunk=c)
               for _, d, c, _ in cases)
    ws = torch.zeros(need, dtype=torch.uint8, device=cuda_device)
    for rep in range(2):
        for p, d, chunk, (ref, ref_lse) in cases:
            m = d.metadata()
            out = torch.full_like(d.q, float("nan"))
            lse = torch.full((p.num_seqs, p.num_q_heads), float("nan"), dtype=torch.float32,
                             device=cuda_device)
            pa.decode(d.q, d.k_cache, d.v_cache, m.page_table, m.cache_seqlens, m.max_seqlen_k,
                      scale=p.scale, out=out, lse=lse, workspace=ws, kv_chunk=chunk)
            torch.cuda.synchronize()
            compare(out, ref, f"reuse {rep} C{chunk}", lse_gpu=lse, lse_ref=ref_lse)


@pytest.mark.parametrize("d", [64, 128])
def test_lse_combine(cuda_device, d):
    import paged_kv_flashattention_gb300 as pa
    rng = np.random.default_rng(d)
    R, S = 300, 13
    o = rng.standard_normal((R, S, d)).astype(np.float32)
    l = (rng.standard_normal((R, S)) * 5).astype(np.float32)
    l[rng.random((R, S)) < 0.2] = -np.inf
    l[5] = -np.inf                       # a row with only empty splits
    n = rng.integers(0, S + 1, size=R).astype(np.int32)
    n[7] = 0
    lse = torch.empty(R, dtype=torch.float32, device=cuda_device)
    out = pa.lse_combine(torch.from_numpy(o).to(cuda_device), torch.from_numpy(l).to(cuda_device),
                         torch.from_numpy(n).to(cuda_device), lse=lse)
    mask = np.arange(S)[None, :] < n[:, None]
    ref_o, ref_l = online.merge_partials(np.where(mask[..., None], o, 0.0), np.where(mask, l, -np.inf))
    compare(out, ref_o, f"lse_combine d{d}", lse_gpu=lse, lse_ref=ref_l)


def _shared_prefix_problem(seed, decode, page, d=128):
    """Requests 1 and 3 start with request 0's pages (a cached prefix shared
    through the page table, PagedAttention's block sharing), request 2 with
    request 1's; each then continues on pages of its own."""
    cached = [300, 310, 350, 20] if not decode else [300, 333, 400, 40]
    ext = [1, 1, 1, 1] if decode else [40, 130, 64, 17]
    n = 256 // page                                      # shared pages: the first 256 keys
    return W.small_problem(seed, cached, ext, num_q_heads=8, num_kv_heads=2, head_dim=d, page_size=page,
                           shared_prefix_pages={1: (0, n), 2: (1, n), 3: (0, 1)})


@pytest.mark.parametrize("page", [1, 16])
@pytest.mark.parametrize("fp8", [False, True])
def test_shared_prefix_pages(cuda_device, page, fp8):
    """Several requests whose page tables point at the same physical pages,
    through pa_decode and pa_prefill, against the oracle (which reads them
    through the same tables)."""
    for decode in (True, False):
        p = _shared_prefix_problem(900 + page + 2 * fp8 + 4 * decode, decode, page)
        pl = p.meta["page_lists"]
        assert pl[1][:256 // page] == pl[0][:256 // page] and pl[2][:256 // page] == pl[1][:256 // page]
        what = f"shared prefix {'decode' if decode else 'prefill'} P{page}{' fp8' if fp8 else ''}"
        if fp8:
            from test_fp8_gpu import FP8Problem
            f = FP8Problem(p, cuda_device, 950 + page)
            out, lse = f.decode() if decode else f.prefill()
            torch.cuda.synchronize()
            ref, ref_lse = f.oracle()
        else:
            dp = DeviceProblem(p, cuda_device)
            dp.store()
            out, lse = dp.decode() if decode else dp.prefill()
            torch.cuda.synchronize()
            ref, ref_lse = oracle_ref(p)
        if decode:
            compare(out, ref.reshape(out.shape), what, lse_gpu=lse, lse_ref=ref_lse.reshape(lse.shape))
        else:
            compare(out, ref, what, lse_gpu=lse[:, :ref.shape[0]].T.contiguous(), lse_ref=ref_lse)
