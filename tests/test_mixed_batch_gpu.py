"""Parity at full size on the benchmark's own workload and launch path: the
mixed continuous batch (256 decode sequences with contexts log-uniform in
[512, 32768] and two 2048-token prefill chunks over a 40 GB pool), run by
bench.MixedBatch.step() exactly as bench.py times it: the headline's single
mixed-batch launch (12 prefill CTAs, 256-key T-ranges), and the PDL overlap
schedule its schedule comparison also times.  Sampled outputs are
checked one by one against the oracle: for a handful of sequences the pages
they read are copied to the host before the step, the oracle applies the
step's KV store to them and computes those rows."""
import numpy as np
import pytest
import torch

import oracle
from pa_harness import compare

pytestmark = pytest.mark.gpu


def _bits(t):
    return t.detach().view(torch.int16).cpu().numpy().view(np.uint16)


def _oracle_rows(prob, k_pages, v_pages, page_ids, seqs, q_rows, new_k, new_v, new_slots, decode,
                 rows=None):
    """Oracle output for requests `seqs` of `prob`, with their pages packed
    into a compact host pool (the result does not depend on placement)."""
    P, Hkv, d = prob.page_size, prob.num_kv_heads, prob.head_dim
    remap = {int(p): i for i, p in enumerate(page_ids)}
    kc, vc = k_pages.copy(), v_pages.copy()
    # the step's store, restricted to the sampled requests' new tokens
    row = Hkv * d
    slots = np.array([remap[s // P] * P + s % P for s in new_slots], np.int32)
    oracle.store_kv(new_k.reshape(-1, row), new_v.reshape(-1, row), slots,
                    kc.reshape(-1, row), vc.reshape(-1, row))
    width = max(len(prob.meta["page_lists"][b]) for b in seqs)
    pt = np.zeros((len(seqs), width), np.int32)
    for i, b in enumerate(seqs):
        pl = [remap[p] for p in prob.meta["page_lists"][b]]
        pt[i, :len(pl)] = pl
    if decode:
        return oracle.decode(q_rows, kc, vc, pt, prob.device_len[seqs], num_q_heads=prob.num_q_heads,
                             num_kv_heads=Hkv, head_dim=d, page_size=P, scale=prob.scale)
    cu = np.concatenate([[0], np.cumsum(prob.extend_len[seqs])]).astype(np.int32)
    ck = np.concatenate([[0], np.cumsum(prob.device_len[seqs])]).astype(np.int32)
    return oracle.attention(q_rows, kc, vc, pt, cu, ck, num_q_heads=prob.num_q_heads,
                            num_kv_heads=Hkv, head_dim=d, page_size=P, causal=True,
                            scale=prob.scale, rows=rows)


@pytest.mark.parametrize("schedule", ["fused", "overlap"])
def test_mixed_batch_full_size_sampled(cuda_device, schedule):
    import bench
    mb = bench.MixedBatch(cuda_device)
    mb.schedule = schedule
    dec, pre = mb.dec, mb.pre
    L = dec.device_len
    order = np.argsort(L)
    dseqs = sorted({int(order[0]), int(order[1]), int(order[len(order) // 2]), int(order[-2]),
                    int(order[-1])})
    pseqs = [0, 1]
    pages_d = sorted({p for b in dseqs for p in dec.meta["page_lists"][b]})
    pages_p = sorted({p for b in pseqs for p in pre.meta["page_lists"][b]})
    idx_d = torch.tensor(pages_d, dtype=torch.long, device=cuda_device)
    idx_p = torch.tensor(pages_p, dtype=torch.long, device=cuda_device)
    kd, vd = _bits(mb.k_cache.index_select(0, idx_d)), _bits(mb.v_cache.index_select(0, idx_d))
    kp, vp = _bits(mb.k_cache.index_select(0, idx_p)), _bits(mb.v_cache.index_select(0, idx_p))
    mb.step()
    torch.cuda.synchronize()
    import paged_kv_flashattention_gb300 as pa
    assert pa.device_error() == 0

    # decode rows: the new token of request b is row b of the store inputs
    knew, vnew = _bits(mb.k_new), _bits(mb.v_new)
    ref, _ = _oracle_rows(dec, kd, vd, pages_d, dseqs, _bits(mb.q_dec)[dseqs], knew[dseqs],
                          vnew[dseqs], dec.slot_mapping[dseqs], decode=True)
    compare(mb.out_dec[torch.tensor(dseqs, device=cuda_device)], ref, f"{schedule}: decode (sampled)")

    # prefill rows: a sample of each chunk's rows (first, last, random), all heads
    rng = np.random.default_rng(3)
    nd = dec.num_new_tokens
    rows = np.unique(np.concatenate([[0, 1, 127, 128, 2047, 2048, 2049, 4095],
                                     rng.choice(4096, size=120, replace=False)]))
    pairs = np.stack(np.meshgrid(rows, np.arange(pre.num_q_heads), indexing="ij"), -1).reshape(-1, 2)
    ref_rows, _ = _oracle_rows(pre, kp, vp, pages_p, pseqs, _bits(mb.q_pre), knew[nd:], vnew[nd:],
                               pre.slot_mapping, decode=False, rows=pairs)
    got = mb.out_pre[torch.from_numpy(pairs[:, 0]).to(cuda_device), torch.from_numpy(pairs[:, 1]).to(cuda_device)]
    compare(got, ref_rows, f"{schedule}: prefill (sampled rows)")
    del mb
    torch.cuda.empty_cache()
