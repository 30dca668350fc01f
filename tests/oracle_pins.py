"""Checks that pin the fp64 oracle to facts other than itself.

Each ``check_*`` takes an optional ``lib`` (another build of the oracle's C
source) and raises AssertionError when the oracle disagrees with:

* a pure-Python brute force written the other way round (gather first,
  unshifted textbook softmax, exactly rounded sums);
* closed forms: equal scores give the mean of the visible values, a single
  visible key returns its value, a dominant score returns its value, no
  visible key returns zeros;
* the library routine torch.nn.functional.scaled_dot_product_attention in
  float64 on contiguous K/V gathered with the allocator's own token table and
  an explicit end-aligned causal mask;
* invariants of the method: decode equals the last row of causal prefill,
  extend equals the tail of a full causal prefill, grouped-query heads equal
  multi-head attention with the KV heads repeated, page size 1 and 16 give
  the same result, physical page permutation and prefix sharing change
  nothing, the online block merge and the split merge equal the two-pass
  softmax.

The FP8 (E4M3) KV path is pinned by closed-form code values from the
format's definition, by a second rounding procedure written the other way
(binade quantum and numpy's round-half-even instead of the oracle's
bisection over the code table), by an elementwise quantisation reference for
the store, and by the identity "attention over FP8 pools = attention over
bf16 pools holding the same values" (every E4M3 value times a power-of-two
scale is a bf16 value, so both paths see identical numbers).

The rotary embedding is pinned by numpy's cos / sin of p * base^(-2i/r) for
the table, by complex multiplication (pairs as complex numbers times e^(i
angle)) for the rotation, by its defining property (q(m) . k(n) depends only
on m - n) and by position 0 being the identity; the bf16 rounding by the
input generator's float32 -> bf16 rounding on float32 values and exact ties.

The block-sparse mask (128 x 128 blocks of a request's query rows and keys)
is pinned by the brute force filtering keys by the mask byte, by the all-ones
and all-zero masks, by a block-diagonal mask equalling independent 128-token
requests, and by a hidden first key block equalling a page table shifted by
128 keys.

The hand-worked golden cases live in tests/golden/.
"""
from __future__ import annotations

import json
import math
import os

import numpy as np

import oracle
from oracle import brute, online
import workloads as W

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _meta(p: W.Problem, lib=None):
    cu_q, cu_k, cs, mq, mk = oracle.seqlens(p.cached_len, p.extend_len, lib=lib)
    pt = oracle.page_table_from_token_table(p.token_table, p.table_idx, max(mk, 1), p.page_size,
                                            lib=lib)
    return cu_q, cu_k, cs, pt


def stored_caches(p: W.Problem, lib=None):
    kc = p.k_cache.copy()
    vc = p.v_cache.copy()
    row = p.num_kv_heads * p.head_dim
    oracle.store_kv(p.k_new.reshape(-1, row), p.v_new.reshape(-1, row), p.slot_mapping,
                    kc.reshape(-1, row), vc.reshape(-1, row), lib=lib)
    return kc, vc


def run_oracle(p: W.Problem, lib=None, rows=None, caches=None):
    cu_q, cu_k, _, pt = _meta(p, lib)
    kc, vc = caches if caches is not None else stored_caches(p, lib)
    return oracle.attention(p.q, kc, vc, pt, cu_q, cu_k, num_q_heads=p.num_q_heads,
                            num_kv_heads=p.num_kv_heads, head_dim=p.head_dim,
                            page_size=p.page_size, causal=p.causal, scale=p.scale,
                            rows=rows, lib=lib)


def _assert_close(a, b, tol, what):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    assert a.shape == b.shape, (what, a.shape, b.shape)
    fin = np.isfinite(b)
    assert np.array_equal(np.isfinite(a), fin), f"{what}: finiteness differs"
    err = float(np.max(np.abs(a[fin] - b[fin]))) if fin.any() else 0.0
    assert err <= tol, f"{what}: max abs err {err:.3e} > {tol:.1e}"


# --------------------------------------------------------------------------
def edge_problems(head_dim=8, page_size=4):
    """Small shapes over the edge-case matrix of section 24 of the first page:
    lengths 1, page-1, page, page+1; empty KV; partial pages; cached prefix +
    extend; a shared prefix; decode."""
    P = page_size
    cases = [
        ([0, 0, 0, 0], [1, P - 1, P, P + 1]),       # no cache hit, lengths at page edges
        ([P - 1, P, P + 1, 2 * P + 3], [1, 1, 1, 1]),  # decode rows
        ([0, 3, 2 * P, 5], [0, 2, 3, P + 2]),      # empty request, partial hits
    ]
    out = []
    for n, (c, e) in enumerate(cases):
        out.append(W.small_problem(100 + n, c, e, num_q_heads=4, num_kv_heads=2,
                                   head_dim=head_dim, page_size=P))
    # shared prefix: request 1's first two pages are request 0's
    out.append(W.small_problem(200, [2 * P + 1, 2 * P + 3], [2, 1], num_q_heads=4, num_kv_heads=2,
                               head_dim=head_dim, page_size=P, shared_prefix_pages={1: (0, 2)}))
    return out


def _brute(p: W.Problem, kc, vc, lib=None, window_left=-1, causal=None):
    cu_q, cu_k, _, pt = _meta(p, lib)
    kcr = kc.reshape(-1, p.num_kv_heads, p.head_dim)
    vcr = vc.reshape(-1, p.num_kv_heads, p.head_dim)
    return np.array(brute.attention(p.q, kcr, vcr, pt, cu_q, cu_k, num_q_heads=p.num_q_heads,
                                    num_kv_heads=p.num_kv_heads, head_dim=p.head_dim,
                                    page_size=p.page_size, causal=p.causal if causal is None else causal,
                                    scale=p.scale, window_left=window_left),
                    dtype=np.float64).reshape(-1, p.num_q_heads, p.head_dim)


def check_brute_force(lib=None):
    for P in (1, 4):
        for p in edge_problems(page_size=P):
            kc, vc = stored_caches(p, lib)
            o, _ = run_oracle(p, lib, caches=(kc, vc))
            ob = _brute(p, kc, vc, lib)
            _assert_close(o, ob, 1e-12, f"brute force P={P}")


def check_equal_scores(lib=None):
    """q = 0: every visible score is 0, so O is the mean of the visible V."""
    p = W.small_problem(11, [5, 0, 9], [3, 4, 1], num_q_heads=4, num_kv_heads=2, head_dim=8,
                        page_size=4)
    p.q[:] = 0
    kc, vc = stored_caches(p, lib)
    o, lse = run_oracle(p, lib, caches=(kc, vc))
    cu_q, cu_k, _, _ = _meta(p, lib)
    V = oracle.bf16_to_f64(vc).reshape(-1, p.num_kv_heads, p.head_dim)
    g = p.num_q_heads // p.num_kv_heads
    for b in range(p.num_seqs):
        Lq = int(cu_q[b + 1] - cu_q[b])
        Lk = int(cu_k[b + 1] - cu_k[b])
        slots = p.token_table[b, :Lk]
        for i in range(Lq):
            n = Lk - Lq + i + 1
            for h in range(p.num_q_heads):
                want = V[slots[:n], h // g].mean(axis=0)
                _assert_close(o[cu_q[b] + i, h], want, 1e-13, "equal scores -> mean of V")
                _assert_close(lse[cu_q[b] + i, h], math.log(n), 1e-13, "equal scores lse = ln n")


def check_single_key(lib=None):
    """One visible key: O = V_0 exactly and lse = its score."""
    p = W.small_problem(12, [0, 0], [1, 1], num_q_heads=4, num_kv_heads=2, head_dim=8, page_size=4)
    kc, vc = stored_caches(p, lib)
    o, lse = run_oracle(p, lib, caches=(kc, vc))
    g = p.num_q_heads // p.num_kv_heads
    q = oracle.bf16_to_f64(p.q)
    for b in range(2):
        slot = p.token_table[b, 0]
        for h in range(p.num_q_heads):
            v0 = oracle.bf16_to_f64(vc.reshape(-1, p.num_kv_heads, p.head_dim)[slot, h // g])
            k0 = oracle.bf16_to_f64(kc.reshape(-1, p.num_kv_heads, p.head_dim)[slot, h // g])
            _assert_close(o[b, h], v0, 0.0, "single key -> V_0")
            _assert_close(lse[b, h], p.scale * float(np.dot(q[b, h], k0)), 1e-12, "single key lse")


def check_dominant_key(lib=None):
    """One key whose score exceeds every other by > 60 nats: O = that V to
    within e^-60 relative."""
    p = W.small_problem(13, [20], [1], num_q_heads=2, num_kv_heads=1, head_dim=8, page_size=4,
                        scale=1.0)
    q = np.zeros((1, 2, 8), np.float32)
    q[0, :, 0] = 8.0
    p.q = W.f32_to_bf16_bits(q)
    kcr = p.k_cache.reshape(-1, 1, 8)
    kcr[:] = 0
    target = 13
    slot = p.token_table[0, target]
    kcr[slot, 0, 0] = W.f32_to_bf16_bits(np.array([16.0], np.float32))[0]   # score 128
    kc, vc = stored_caches(p, lib)
    kc.reshape(-1, 1, 8)[p.slot_mapping[0], 0, :] = 0      # the new token: score 0
    o, lse = run_oracle(p, lib, caches=(kc, vc))
    v = oracle.bf16_to_f64(vc.reshape(-1, 1, 8)[slot, 0])
    for h in range(2):
        _assert_close(o[0, h], v, 1e-40, "dominant key")


def check_empty(lib=None):
    """No visible key: a decode row over an empty cache gives O = 0 and
    lse = -inf, and a request with Lq = Lk = 0 inside a batch has no rows and
    leaves its neighbours' results unchanged."""
    p = W.small_problem(14, [0, 3, 0], [0, 2, 0], num_q_heads=4, num_kv_heads=2, head_dim=8,
                        page_size=4)
    kc, vc = stored_caches(p, lib)
    cu_q, cu_k, _, pt = _meta(p, lib)
    o, l = oracle.attention(p.q, kc, vc, pt, cu_q, cu_k, num_q_heads=4, num_kv_heads=2,
                            head_dim=8, page_size=4, causal=True, scale=p.scale, lib=lib)
    o_alone, l_alone = oracle.attention(p.q, kc, vc, pt[1:2], np.array([0, 2], np.int32),
                                        np.array([0, 5], np.int32), num_q_heads=4,
                                        num_kv_heads=2, head_dim=8, page_size=4, causal=True,
                                        scale=p.scale, lib=lib)
    _assert_close(o, o_alone, 0.0, "empty neighbours change nothing")
    o1, l1 = oracle.decode(p.q[:1], kc, vc, pt[:1], np.array([0]), num_q_heads=4, num_kv_heads=2,
                           head_dim=8, page_size=4, scale=p.scale, lib=lib)
    assert np.all(o1 == 0.0) and np.all(np.isneginf(l1)), "empty KV must give O = 0, lse = -inf"


def check_sdpa_library(lib=None):
    """torch SDPA in float64 with an explicit end-aligned mask on gathered K/V."""
    import torch
    for P in (1, 4):
        for p in edge_problems(head_dim=16, page_size=P)[:3] + [
                W.small_problem(15, [37, 0, 12], [11, 23, 1], num_q_heads=6, num_kv_heads=2,
                                head_dim=16, page_size=P)]:
            kc, vc = stored_caches(p, lib)
            o, lse = run_oracle(p, lib, caches=(kc, vc))
            cu_q, cu_k, _, _ = _meta(p, lib)
            K = oracle.bf16_to_f64(kc).reshape(-1, p.num_kv_heads, p.head_dim)
            V = oracle.bf16_to_f64(vc).reshape(-1, p.num_kv_heads, p.head_dim)
            Q = oracle.bf16_to_f64(p.q)
            g = p.num_q_heads // p.num_kv_heads
            for b in range(p.num_seqs):
                Lq = int(cu_q[b + 1] - cu_q[b])
                Lk = int(cu_k[b + 1] - cu_k[b])
                if Lq == 0:
                    continue
                slots = p.token_table[b, :Lk]
                kb = torch.from_numpy(K[slots]).permute(1, 0, 2).repeat_interleave(g, dim=0)
                vb = torch.from_numpy(V[slots]).permute(1, 0, 2).repeat_interleave(g, dim=0)
                qb = torch.from_numpy(Q[cu_q[b]:cu_q[b + 1]]).permute(1, 0, 2)
                i = torch.arange(Lq)[:, None]
                j = torch.arange(Lk)[None, :]
                mask = j <= (Lk - Lq) + i
                ref = torch.nn.functional.scaled_dot_product_attention(
                    qb, kb, vb, attn_mask=mask, scale=p.scale).permute(1, 0, 2).numpy()
                _assert_close(o[cu_q[b]:cu_q[b + 1]], ref, 1e-12, f"SDPA library P={P}")
                s = torch.einsum("hqd,hkd->hqk", qb, kb) * p.scale
                s = s.masked_fill(~mask, float("-inf"))
                ref_lse = torch.logsumexp(s, dim=-1).permute(1, 0).numpy()
                _assert_close(lse[cu_q[b]:cu_q[b + 1]], ref_lse, 1e-12, "lse vs logsumexp")


def check_decode_is_last_prefill_row(lib=None):
    L = [9, 17, 33]
    pre = W.small_problem(16, [0, 0, 0], L, num_q_heads=4, num_kv_heads=2, head_dim=8, page_size=4)
    o_pre, l_pre = run_oracle(pre, lib)
    kc, vc = stored_caches(pre, lib)
    cu_q, cu_k, _, pt = _meta(pre, lib)
    last = cu_q[1:] - 1
    o_dec, l_dec = oracle.decode(pre.q[last], kc, vc, pt, np.array(L), num_q_heads=4,
                                 num_kv_heads=2, head_dim=8, page_size=4, scale=pre.scale, lib=lib)
    _assert_close(o_dec, o_pre[last], 0.0, "decode == last row of causal prefill")
    _assert_close(l_dec, l_pre[last], 0.0, "decode lse == last prefill lse")


def check_extend_is_prefill_tail(lib=None):
    """A request with C cached tokens and E extend tokens gives the last E rows
    of the causal prefill of all C + E tokens (same K/V, same queries)."""
    C, E = [13, 0, 5], [6, 4, 9]
    full = W.small_problem(17, [0, 0, 0], [c + e for c, e in zip(C, E)], num_q_heads=4,
                           num_kv_heads=2, head_dim=8, page_size=4)
    o_full, l_full = run_oracle(full, lib)
    kc, vc = stored_caches(full, lib)
    cu_qf, cu_kf, _, pt = _meta(full, lib)
    rows = np.concatenate([np.arange(cu_qf[b] + C[b], cu_qf[b + 1]) for b in range(3)])
    cu_q = np.concatenate([[0], np.cumsum(E)]).astype(np.int32)
    o_ext, l_ext = oracle.attention(full.q[rows], kc, vc, pt, cu_q, cu_kf, num_q_heads=4,
                                    num_kv_heads=2, head_dim=8, page_size=4, causal=True,
                                    scale=full.scale, lib=lib)
    _assert_close(o_ext, o_full[rows], 0.0, "extend == tail of full causal prefill")
    _assert_close(l_ext, l_full[rows], 0.0, "extend lse == tail lse")


def check_gqa_equals_repeated_mha(lib=None):
    p = W.small_problem(18, [7, 2], [5, 9], num_q_heads=6, num_kv_heads=2, head_dim=8, page_size=4)
    o, l = run_oracle(p, lib)
    kc, vc = stored_caches(p, lib)
    g = 3
    kr = np.repeat(kc.reshape(-1, 2, 8), g, axis=1).copy()
    vr = np.repeat(vc.reshape(-1, 2, 8), g, axis=1).copy()
    cu_q, cu_k, _, pt = _meta(p, lib)
    o2, l2 = oracle.attention(p.q, kr, vr, pt, cu_q, cu_k, num_q_heads=6, num_kv_heads=6,
                              head_dim=8, page_size=4, causal=True, scale=p.scale, lib=lib)
    _assert_close(o, o2, 0.0, "GQA == MHA with repeated KV heads")
    _assert_close(l, l2, 0.0, "GQA lse == MHA lse")


def check_page_size_equivalence(lib=None):
    """Same logical K/V under a page-16 table and under the token-granular
    (page size 1) table of the same slots."""
    p = W.small_problem(19, [40, 3, 0], [2, 30, 17], num_q_heads=4, num_kv_heads=2, head_dim=8,
                        page_size=16)
    o16, l16 = run_oracle(p, lib)
    kc, vc = stored_caches(p, lib)
    cu_q, cu_k, _, _ = _meta(p, lib)
    pt1 = oracle.page_table_from_token_table(p.token_table, p.table_idx, int(p.device_len.max()), 1,
                                             lib=lib)
    o1, l1 = oracle.attention(p.q, kc, vc, pt1, cu_q, cu_k, num_q_heads=4, num_kv_heads=2,
                              head_dim=8, page_size=1, causal=True, scale=p.scale, lib=lib)
    _assert_close(o16, o1, 0.0, "page size 16 == page size 1")
    _assert_close(l16, l1, 0.0, "page size lse")


def check_permutation_invariance(lib=None):
    """Re-pack the same logical K/V onto another seeded page permutation."""
    p = W.small_problem(20, [21, 6, 0], [3, 11, 9], num_q_heads=4, num_kv_heads=2, head_dim=8,
                        page_size=4)
    o, l = run_oracle(p, lib)
    kc, vc = stored_caches(p, lib)
    npg = p.num_pages
    perm = np.random.default_rng(99).permutation(npg - 1)
    perm = np.concatenate([perm, [npg - 1]])           # poison page stays put
    kc2 = np.empty_like(kc)
    vc2 = np.empty_like(vc)
    kc2[perm] = kc
    vc2[perm] = vc
    tt = p.token_table.astype(np.int64)
    tt2 = (perm[tt // 4] * 4 + tt % 4).astype(np.int32)
    cu_q, cu_k, _, _ = _meta(p, lib)
    pt2 = oracle.page_table_from_token_table(tt2, p.table_idx, int(p.device_len.max()), 4, lib=lib)
    o2, l2 = oracle.attention(p.q, kc2, vc2, pt2, cu_q, cu_k, num_q_heads=4, num_kv_heads=2,
                              head_dim=8, page_size=4, causal=True, scale=p.scale, lib=lib)
    _assert_close(o, o2, 0.0, "physical page permutation invariance")
    _assert_close(l, l2, 0.0, "permutation lse")


def check_threads_and_rows_invariance(lib=None):
    """The oracle computes every (token, head) row on its own, so neither the
    number of threads nor computing a sample of rows may change a value: one
    thread and every thread give the same bits, and the rows mode returns the
    same bits as the full call at those rows (the sampled parity tests and the
    bench's CPU baselines use it)."""
    p = W.small_problem(21, [0, 37, 130, 5], [19, 64, 150, 1], num_q_heads=8, num_kv_heads=2, head_dim=64,
                        page_size=16)
    full_o, full_l = run_oracle(p, lib)
    saved = oracle.num_threads()
    try:
        oracle.set_threads(1)
        one_o, one_l = run_oracle(p, lib)
    finally:
        oracle.set_threads(saved)
    assert np.array_equal(one_o, full_o) and np.array_equal(one_l, full_l), "thread count changed the oracle"
    rng = np.random.default_rng(5)
    tok = rng.integers(0, full_o.shape[0], size=40)
    head = rng.integers(0, p.num_q_heads, size=40)
    rows = np.stack([tok, head], axis=1).astype(np.int64)
    ro, rl = run_oracle(p, lib, rows=rows)
    assert np.array_equal(ro, full_o[tok, head]) and np.array_equal(rl, full_l[tok, head]), \
        "rows mode differs from the full call"


def check_shared_prefix(lib=None):
    """Two requests whose tables share physical prefix pages give the same
    result as two requests holding private copies of those pages."""
    P = 4
    sh = W.small_problem(21, [10, 10], [3, 3], num_q_heads=4, num_kv_heads=2, head_dim=8,
                         page_size=P, shared_prefix_pages={1: (0, 2)})
    kc, vc = stored_caches(sh, lib)
    o, l = run_oracle(sh, lib, caches=(kc, vc))
    # private copy: duplicate request 0's first two pages into fresh pages for request 1
    extra = 2
    kc2 = np.concatenate([kc[:-1], kc[[sh.meta['page_lists'][0][0], sh.meta['page_lists'][0][1]]],
                          kc[-1:]])
    vc2 = np.concatenate([vc[:-1], vc[[sh.meta['page_lists'][0][0], sh.meta['page_lists'][0][1]]],
                          vc[-1:]])
    npg = sh.num_pages + extra
    tt = sh.token_table.astype(np.int64).copy()
    tt[tt // P == sh.num_pages - 1] = (npg - 1) * P          # poison moved to the end
    new0, new1 = sh.num_pages - 1, sh.num_pages
    tt[1, 0:P] = new0 * P + np.arange(P)
    tt[1, P:2 * P] = new1 * P + np.arange(P)
    cu_q, cu_k, _, _ = _meta(sh, lib)
    pt2 = oracle.page_table_from_token_table(tt.astype(np.int32), sh.table_idx,
                                             int(sh.device_len.max()), P, lib=lib)
    o2, l2 = oracle.attention(sh.q, kc2, vc2, pt2, cu_q, cu_k, num_q_heads=4, num_kv_heads=2,
                              head_dim=8, page_size=P, causal=True, scale=sh.scale, lib=lib)
    _assert_close(o, o2, 0.0, "shared prefix == private copies")


def check_online_and_split_merge(lib=None):
    """Online block merge (section 12) with random blocks and the split merge
    (section 16) over random key splits both equal the two-pass result."""
    rng = np.random.default_rng(5)
    p = W.small_problem(22, [50, 0], [1, 40], num_q_heads=4, num_kv_heads=2, head_dim=8, page_size=4)
    kc, vc = stored_caches(p, lib)
    o, lse = run_oracle(p, lib, caches=(kc, vc))
    cu_q, cu_k, _, pt = _meta(p, lib)
    K = oracle.bf16_to_f64(kc).reshape(-1, 2, 8)
    V = oracle.bf16_to_f64(vc).reshape(-1, 2, 8)
    Q = oracle.bf16_to_f64(p.q)
    for b in range(2):
        Lq, Lk = int(cu_q[b + 1] - cu_q[b]), int(cu_k[b + 1] - cu_k[b])
        slots = p.token_table[b, :Lk]
        for i in range(Lq):
            n = Lk - Lq + i + 1
            for h in range(4):
                s = p.scale * (K[slots[:n], h // 2] @ Q[cu_q[b] + i, h])
                cuts = sorted(set(rng.integers(1, max(2, n), size=rng.integers(0, 6)).tolist()))
                edges = [0] + [c for c in cuts if 0 < c < n] + [n]
                oo, ll = online.online_softmax_row(s, V[slots[:n], h // 2], edges)
                _assert_close(oo, o[cu_q[b] + i, h], 1e-12, "online == two-pass")
                _assert_close(ll, lse[cu_q[b] + i, h], 1e-12, "online lse == two-pass lse")
    # split merge: decode of request 0 (51 keys) split at page edges into sub-requests
    Lk = int(p.device_len[0])
    for cuts in ([16], [8, 20, 44], [4, 8, 12, 16, 48]):
        edges = [0] + cuts + [Lk]
        parts_o, parts_l = [], []
        for a, e in zip(edges[:-1], edges[1:]):
            sub_pt = pt[0:1, a // 4:]
            oo, ll = oracle.decode(p.q[0:1], kc, vc, sub_pt, np.array([e - a]), num_q_heads=4,
                                   num_kv_heads=2, head_dim=8, page_size=4, scale=p.scale, lib=lib)
            parts_o.append(oo[0])
            parts_l.append(ll[0])
        # one empty split as well
        parts_o.append(np.zeros_like(parts_o[0]))
        parts_l.append(np.full_like(parts_l[0], -np.inf))
        mo, ml = online.merge_partials(np.stack(parts_o, axis=1), np.stack(parts_l, axis=1))
        _assert_close(mo, o[0], 1e-12, "split merge == whole")
        _assert_close(ml, lse[0], 1e-12, "split merge lse == whole")


def check_golden(lib=None):
    """Hand-worked cases in tests/golden/attention_cases.json."""
    with open(os.path.join(GOLDEN, "attention_cases.json")) as f:
        cases = json.load(f)["cases"]
    for c in cases:
        bf = lambda a: W.f32_to_bf16_bits(np.asarray(a, np.float32))
        q = bf(c["q"])
        kc, vc = bf(c["k_cache"]), bf(c["v_cache"])
        o, l = oracle.attention(q, kc, vc, np.asarray(c["page_table"], np.int32),
                                np.asarray(c["cu_seqlens_q"], np.int32),
                                np.asarray(c["cu_seqlens_k"], np.int32),
                                num_q_heads=c["num_q_heads"], num_kv_heads=c["num_kv_heads"],
                                head_dim=c["head_dim"], page_size=c["page_size"],
                                causal=c["causal"], scale=c["scale"], lib=lib)
        _assert_close(o, np.asarray(c["out"], np.float64), 1e-12, f"golden {c['name']}")
        _assert_close(l, np.asarray(c["lse"], np.float64), 1e-12, f"golden {c['name']} lse")


def check_store(lib=None):
    """Store is a bit copy into the listed slots, skipping negative slots and
    leaving every other row untouched (numpy fancy-index assignment as the
    library reference)."""
    rng = np.random.default_rng(3)
    slots_total, row = 40, 12
    kc = rng.integers(0, 1 << 16, size=(slots_total, row), dtype=np.uint16)
    vc = rng.integers(0, 1 << 16, size=(slots_total, row), dtype=np.uint16)
    sm = np.array([5, -1, 39, 0, 17, -7, 6], np.int32)
    k = rng.integers(0, 1 << 16, size=(7, row), dtype=np.uint16)
    v = rng.integers(0, 1 << 16, size=(7, row), dtype=np.uint16)
    ke, ve = kc.copy(), vc.copy()
    keep = sm >= 0
    ke[sm[keep]] = k[keep]
    ve[sm[keep]] = v[keep]
    oracle.store_kv(k, v, sm, kc, vc, lib=lib)
    assert np.array_equal(kc, ke) and np.array_equal(vc, ve), "store must be a bit copy"


def check_metadata(lib=None):
    """cu_seqlens are the prefix sums (numpy cumsum as the library reference)
    and the page table lists the pages the allocator handed out, in order."""
    p = W.small_problem(23, [0, 17, 5, 40], [3, 1, 12, 9], num_q_heads=4, num_kv_heads=2,
                        head_dim=8, page_size=16)
    cu_q, cu_k, cs, mq, mk = oracle.seqlens(p.cached_len, p.extend_len, lib=lib)
    assert np.array_equal(cu_q, np.concatenate([[0], np.cumsum(p.extend_len)]))
    assert np.array_equal(cu_k, np.concatenate([[0], np.cumsum(p.device_len)]))
    assert np.array_equal(cs, p.device_len) and mq == 12 and mk == 49
    for P in (16,):
        pt = oracle.page_table_from_token_table(p.token_table, p.table_idx, mk, P, lib=lib)
        for b in range(p.num_seqs):
            pl = p.meta["page_lists"][b]
            assert list(pt[b, :len(pl)]) == pl, "page table must list the allocated pages"
    pt1 = oracle.page_table_from_token_table(p.token_table, p.table_idx, mk, 1, lib=lib)
    assert np.array_equal(pt1, p.token_table[:, :mk])


def _e4m3_reference_round(x: np.ndarray) -> np.ndarray:
    """Nearest E4M3 value of float32 x, computed by binades: the quantum of
    the binade [2^e, 2^(e+1)) is 2^(e-3) (3 mantissa bits), subnormals share
    the quantum 2^-9 of the lowest normal binade (e = -6), numpy rounds half
    to even, and magnitudes of 448 and more saturate to 448."""
    a = np.abs(x.astype(np.float64))
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    e = np.maximum(e, -6.0)
    quantum = np.exp2(e - 3.0)
    val = np.round(a / quantum) * quantum
    val = np.where(a >= 448.0, 448.0, np.minimum(val, 448.0))
    return np.copysign(val, x.astype(np.float64))


def check_e4m3_codec(lib=None):
    """E4M3 decode against closed forms and encode against an independent
    rounding procedure."""
    v = oracle.e4m3_value(np.arange(256), lib=lib)
    closed = {0x00: 0.0, 0x01: 2.0 ** -9, 0x07: 7 * 2.0 ** -9, 0x08: 2.0 ** -6, 0x30: 0.5,
              0x38: 1.0, 0x39: 1.125, 0x3F: 1.875, 0x40: 2.0, 0x78: 256.0, 0x7E: 448.0,
              0xB8: -1.0, 0xFE: -448.0}
    for c, want in closed.items():
        assert v[c] == want, f"E4M3 code {c:#x} decodes to {v[c]}, not {want}"
    assert np.isnan(v[0x7F]) and np.isnan(v[0xFF])
    assert np.all(np.diff(v[:0x7F]) > 0), "positive codes must increase"
    assert np.array_equal(v[0x80:0xFF], -v[:0x7F]), "sign bit must negate"
    codes = np.arange(0x7F, dtype=np.uint8)
    assert np.array_equal(oracle.e4m3_encode(v[:0x7F].astype(np.float32), lib=lib), codes), \
        "every finite value must encode to its own code"
    rng = np.random.default_rng(11)
    x = np.concatenate([
        rng.standard_normal(4000) * 10.0 ** rng.uniform(-4, 3, 4000),
        (v[1:0x7E] + v[2:0x7F]) / 2.0,              # midpoints between neighbours: ties
        [0.0, 2.0 ** -10, 3 * 2.0 ** -11, 447.9, 448.0, 460.0, 464.0, 1e6, 2.0 ** -20]]).astype(np.float32)
    x = np.concatenate([x, -x])
    got = oracle.e4m3_value(oracle.e4m3_encode(x, lib=lib), lib=lib)
    want = _e4m3_reference_round(x)
    assert np.array_equal(np.abs(got), np.abs(want)), "E4M3 rounding differs from the binade rule"
    nz = want != 0
    assert np.array_equal(np.signbit(got[nz]), np.signbit(want[nz]))


def check_store_fp8(lib=None):
    """FP8 store: each element becomes E4M3(x / scale[head]) (the division in
    float32), rows of negative slots are skipped, other rows untouched."""
    rng = np.random.default_rng(5)
    slots, Hkv, d = 30, 3, 8
    kc = rng.integers(0, 256, size=(slots, Hkv, d), dtype=np.uint8)
    vc = rng.integers(0, 256, size=(slots, Hkv, d), dtype=np.uint8)
    sm = np.array([4, -1, 29, 0, 11], np.int32)
    kf = (rng.standard_normal((5, Hkv, d)) * 3).astype(np.float32)
    vf = (rng.standard_normal((5, Hkv, d)) * 3).astype(np.float32)
    k = W.f32_to_bf16_bits(kf)
    v = W.f32_to_bf16_bits(vf)
    ks = np.array([0.02, 0.5, 3.0], np.float32)
    vs = np.array([0.25, 0.0078125, 1.5], np.float32)
    ke, ve = kc.copy(), vc.copy()
    for t, s_ in enumerate(sm):
        if s_ < 0:
            continue
        kq = (W.bf16_bits_to_f32(k[t]) / ks[:, None]).astype(np.float32)
        vq = (W.bf16_bits_to_f32(v[t]) / vs[:, None]).astype(np.float32)
        ke[s_] = oracle.e4m3_encode(kq, lib=lib)
        ve[s_] = oracle.e4m3_encode(vq, lib=lib)
    oracle.store_kv_fp8(k, v, sm, kc, vc, ks, vs, lib=lib)
    assert np.array_equal(kc, ke) and np.array_equal(vc, ve), "FP8 store differs from E4M3(x / scale)"
    # the codec agrees with the binade rule on these quotients as well
    q = (W.bf16_bits_to_f32(k[0]) / ks[:, None]).astype(np.float32)
    assert np.array_equal(np.abs(oracle.e4m3_value(kc[4], lib=lib)), np.abs(_e4m3_reference_round(q)))


def check_attention_fp8_exact_values(lib=None):
    """Attention over E4M3 pools with per-head power-of-two scales equals,
    bit for bit, attention over bf16 pools holding code value * scale."""
    p = W.small_problem(31, [5, 0, 40], [3, 9, 1], num_q_heads=8, num_kv_heads=4, head_dim=16,
                        page_size=4)
    rng = np.random.default_rng(9)
    shape = p.k_cache.shape
    kc8 = rng.integers(0, 256, size=shape, dtype=np.uint8)
    vc8 = rng.integers(0, 256, size=shape, dtype=np.uint8)
    for c8 in (kc8, vc8):                       # no NaN codes
        c8[(c8 & 0x7F) == 0x7F] = 0x3A
    ks = np.array([0.125, 1.0, 4.0, 0.5], np.float32)
    vs = np.array([2.0, 0.25, 1.0, 8.0], np.float32)
    kval = oracle.e4m3_value(kc8, lib=lib) * ks[None, None, :, None]
    vval = oracle.e4m3_value(vc8, lib=lib) * vs[None, None, :, None]
    kb, vb = W.f32_to_bf16_bits(kval.astype(np.float32)), W.f32_to_bf16_bits(vval.astype(np.float32))
    assert np.array_equal(W.bf16_bits_to_f32(kb).astype(np.float64), kval), "values must be bf16-exact"
    cu_q, cu_k, _, pt = _meta(p, lib)
    kw = dict(num_q_heads=p.num_q_heads, num_kv_heads=p.num_kv_heads, head_dim=p.head_dim,
              page_size=p.page_size, causal=True, scale=p.scale, lib=lib)
    o8, l8 = oracle.attention(p.q, kc8, vc8, pt, cu_q, cu_k, k_scale=ks, v_scale=vs, **kw)
    ob, lb = oracle.attention(p.q, kb, vb, pt, cu_q, cu_k, **kw)
    assert np.array_equal(o8, ob) and np.array_equal(l8, lb), "FP8 attention differs from bf16 on equal values"


def check_rope_table(lib=None):
    """cos / sin table against numpy on the same angles."""
    for r, base in ((128, 10000.0), (64, 500000.0), (16, 10.0)):
        c, s_ = oracle.rope_table(300, r, base, lib=lib)
        p = np.arange(300, dtype=np.float64)[:, None]
        i = np.arange(r // 2, dtype=np.float64)[None, :]
        ang = p * np.power(base, -2.0 * i / r)
        assert np.allclose(c, np.cos(ang), rtol=0, atol=1e-13), "RoPE cos table"
        assert np.allclose(s_, np.sin(ang), rtol=0, atol=1e-13), "RoPE sin table"


def _rope_case(seed, T=6, H=3, d=32):
    rng = np.random.default_rng(seed)
    x = W.normal_bf16(rng, (T, H, d))
    pos = rng.integers(0, 200, size=T).astype(np.int32)
    return x, pos


def check_rope_complex(lib=None):
    """Each rotated pair equals (a + i b) * e^(i angle) by numpy complex
    multiplication, for both pairings and a partial rotated width."""
    x, pos = _rope_case(41)
    xf = W.bf16_bits_to_f32(x).astype(np.float64)
    for r, inter in ((32, False), (32, True), (16, False)):
        c, s_ = oracle.rope_table(200, r, 10000.0, lib=lib)
        got = oracle.rope_rotate(x, pos, c, s_, rot_dim=r, interleaved=inter, lib=lib)
        h = r // 2
        ia = np.arange(h) * 2 if inter else np.arange(h)
        ib = ia + 1 if inter else ia + h
        z = (xf[:, :, ia] + 1j * xf[:, :, ib]) * np.exp(1j * np.arctan2(s_[pos], c[pos]))[:, None, :]
        assert np.allclose(got[:, :, ia], z.real, rtol=0, atol=1e-12), "RoPE real part"
        assert np.allclose(got[:, :, ib], z.imag, rtol=0, atol=1e-12), "RoPE imaginary part"
        rest = np.setdiff1d(np.arange(xf.shape[2]), np.concatenate([ia, ib]))
        assert np.array_equal(got[:, :, rest], xf[:, :, rest]), "elements past the rotated width change"


def check_rope_relative_position(lib=None):
    """q(m) . k(n) depends only on m - n; position 0 is the identity."""
    rng = np.random.default_rng(43)
    q = W.normal_bf16(rng, (1, 1, 64))
    k = W.normal_bf16(rng, (1, 1, 64))
    c, s_ = oracle.rope_table(400, 64, 10000.0, lib=lib)
    dots = []
    for m, n in ((10, 3), (107, 100), (397, 390)):
        qm = oracle.rope_rotate(q, [m], c, s_, rot_dim=64, lib=lib)
        kn = oracle.rope_rotate(k, [n], c, s_, rot_dim=64, lib=lib)
        dots.append(float(np.sum(qm * kn)))
    assert max(dots) - min(dots) < 1e-10, f"RoPE dot products depend on absolute position: {dots}"
    q0 = oracle.rope_rotate(q, [0], c, s_, rot_dim=64, lib=lib)
    assert np.array_equal(q0, W.bf16_bits_to_f32(q).astype(np.float64))


def check_round_bf16(lib=None):
    """One-step bf16 rounding equals float32 -> bf16 rounding on float32
    inputs, including exact ties, signs and subnormals."""
    rng = np.random.default_rng(47)
    f = (rng.standard_normal(5000) * 10.0 ** rng.uniform(-30, 30, 5000)).astype(np.float32)
    ties = (W.bf16_bits_to_f32(W.f32_to_bf16_bits(f)).astype(np.float64) +
            np.ldexp(1.0, np.frexp(f.astype(np.float64))[1] - 9)).astype(np.float32)
    special = np.array([0.0, -0.0, 1.00390625, 1.01171875, 2.0 ** -130, 2.0 ** -133, 3 * 2.0 ** -134], np.float32)
    x = np.concatenate([f, ties, special])
    got = oracle.round_bf16(x.astype(np.float64), lib=lib)
    assert np.array_equal(got, W.f32_to_bf16_bits(x)), "bf16 rounding differs from float32 -> bf16"


def _oracle_window(p, kc, vc, window_left, causal=None, lib=None, rows=None):
    cu_q, cu_k, _, pt = _meta(p, lib)
    return oracle.attention(p.q, kc, vc, pt, cu_q, cu_k, num_q_heads=p.num_q_heads,
                            num_kv_heads=p.num_kv_heads, head_dim=p.head_dim, page_size=p.page_size,
                            causal=p.causal if causal is None else causal, scale=p.scale,
                            window_left=window_left, rows=rows, lib=lib)


def check_window_brute_force(lib=None):
    """Sliding windows of several widths, causal and not, against the brute
    force (which filters keys by p - j <= window_left)."""
    for P in (1, 4):
        for p in edge_problems(page_size=P):
            kc, vc = stored_caches(p, lib)
            for w in (0, 1, 3, 7):
                for causal in (True, False):
                    o, _ = _oracle_window(p, kc, vc, w, causal, lib)
                    ob = _brute(p, kc, vc, lib, window_left=w, causal=causal)
                    _assert_close(o, ob, 1e-12, f"window {w} causal {causal} P={P}")


def check_window_closed_forms(lib=None):
    """A window of 0 under the causal mask leaves each row its own key (O = V
    of its position, lse = its score); a window covering every key changes
    nothing."""
    p = W.small_problem(57, [5, 0, 9], [3, 4, 2], num_q_heads=4, num_kv_heads=2, head_dim=8, page_size=4)
    kc, vc = stored_caches(p, lib)
    o0, l0 = _oracle_window(p, kc, vc, 0, True, lib)
    cu_q, cu_k, _, pt = _meta(p, lib)
    g = p.num_q_heads // p.num_kv_heads
    for b in range(p.num_seqs):
        Lq, Lk = int(p.extend_len[b]), int(p.device_len[b])
        for i in range(Lq):
            t, pos = int(cu_q[b]) + i, Lk - Lq + i
            slot = int(pt[b, pos // p.page_size]) * p.page_size + pos % p.page_size
            for h in range(p.num_q_heads):
                kv = h // g
                vrow = W.bf16_bits_to_f32(vc.reshape(-1, p.num_kv_heads, p.head_dim)[slot, kv]).astype(np.float64)
                krow = W.bf16_bits_to_f32(kc.reshape(-1, p.num_kv_heads, p.head_dim)[slot, kv]).astype(np.float64)
                qrow = W.bf16_bits_to_f32(p.q[t, h]).astype(np.float64)
                assert np.array_equal(o0[t, h], vrow), "window 0 must return the own value"
                assert abs(l0[t, h] - p.scale * math.fsum(qrow * krow)) < 1e-12
    on, ln = _oracle_window(p, kc, vc, -1, True, lib)
    ow, lw = _oracle_window(p, kc, vc, int(p.device_len.max()), True, lib)
    assert np.array_equal(on, ow) and np.array_equal(ln, lw), "a window over every key must change nothing"


def check_window_is_truncated_cache(lib=None):
    """Decode with window w over a token-granular table equals decode without
    a window over the same table row with its first L - 1 - w entries cut."""
    p = W.small_problem(59, [30, 12, 50], [1, 1, 1], num_q_heads=4, num_kv_heads=2, head_dim=8, page_size=1)
    kc, vc = stored_caches(p, lib)
    _, _, cs, pt = _meta(p, lib)
    w = 9
    o, l = oracle.decode(p.q, kc, vc, pt, cs, num_q_heads=4, num_kv_heads=2, head_dim=8, page_size=1,
                         scale=p.scale, window_left=w, lib=lib)
    for b in range(p.num_seqs):
        L = int(cs[b])
        s0 = max(0, L - 1 - w)
        ob, lb = oracle.decode(p.q[b:b + 1], kc, vc, pt[b:b + 1, s0:L], [L - s0], num_q_heads=4,
                               num_kv_heads=2, head_dim=8, page_size=1, scale=p.scale, lib=lib)
        assert np.array_equal(o[b], ob[0]) and np.array_equal(l[b], lb[0]), "window != truncated cache"


# ------------------------------------------------------- block-sparse mask
def _mask_problems():
    """Requests longer than one 128-row / 128-key block: a long prompt, a
    cached prefix with an extend crossing a block edge, a short extend over a
    long prefix, and an empty request."""
    return [W.small_problem(71, [0, 40, 200, 0], [300, 130, 64, 0], num_q_heads=4, num_kv_heads=2,
                            head_dim=8, page_size=4),
            W.small_problem(72, [0, 129], [257, 128], num_q_heads=2, num_kv_heads=1, head_dim=8,
                            page_size=16)]


def _oracle_mask(p, kc, vc, mask, causal=None, lib=None, window_left=-1):
    cu_q, cu_k, _, pt = _meta(p, lib)
    return oracle.attention(p.q, kc, vc, pt, cu_q, cu_k, num_q_heads=p.num_q_heads,
                            num_kv_heads=p.num_kv_heads, head_dim=p.head_dim, page_size=p.page_size,
                            causal=p.causal if causal is None else causal, scale=p.scale,
                            window_left=window_left, block_mask=mask, lib=lib)


def check_block_mask_brute_force(lib=None):
    """Random 128 x 128 block masks, causal and not, with and without a
    window, against the brute force (which filters keys by the mask byte of
    the query's and the key's blocks)."""
    rng = np.random.default_rng(7)
    for p in _mask_problems():
        kc, vc = stored_caches(p, lib)
        cu_q, cu_k, _, pt = _meta(p, lib)
        kcr = kc.reshape(-1, p.num_kv_heads, p.head_dim)
        vcr = vc.reshape(-1, p.num_kv_heads, p.head_dim)
        for causal, w in ((True, -1), (False, -1), (True, 150)):
            m = W.block_mask(rng, p.extend_len, p.device_len, density=0.5, keep_diagonal=False)
            o, _ = _oracle_mask(p, kc, vc, m, causal, lib, window_left=w)
            ob = np.array(brute.attention(p.q, kcr, vcr, pt, cu_q, cu_k, num_q_heads=p.num_q_heads,
                                          num_kv_heads=p.num_kv_heads, head_dim=p.head_dim,
                                          page_size=p.page_size, causal=causal, scale=p.scale,
                                          window_left=w, block_mask=m),
                          dtype=np.float64).reshape(o.shape)
            _assert_close(o, ob, 1e-12, f"block mask causal={causal} window={w}")


def check_block_mask_closed_forms(lib=None):
    """An all-ones mask changes nothing; an all-zero mask leaves every row
    empty (O = 0, lse = -inf)."""
    for p in _mask_problems():
        kc, vc = stored_caches(p, lib)
        o, l = run_oracle(p, lib, caches=(kc, vc))
        nq = max(1, -(-int(p.extend_len.max()) // 128))
        nk = max(1, -(-int(p.device_len.max()) // 128))
        ones = np.ones((p.num_seqs, nq, nk), np.uint8)
        o1, l1 = _oracle_mask(p, kc, vc, ones, lib=lib)
        assert np.array_equal(o, o1) and np.array_equal(l, l1), "all-ones mask must change nothing"
        o0, l0 = _oracle_mask(p, kc, vc, np.zeros_like(ones), lib=lib)
        assert np.all(o0 == 0.0) and np.all(l0 == -np.inf), "all-zero mask must hide every key"


def check_block_mask_diagonal_is_split(lib=None):
    """Causal attention of a prompt with no cached prefix under a
    block-diagonal mask equals the same prompt cut into independent requests
    of 128 tokens (each block attends only within itself)."""
    L = 300
    p = W.small_problem(73, [0], [L], num_q_heads=4, num_kv_heads=2, head_dim=8, page_size=4)
    kc, vc = stored_caches(p, lib)
    nb = -(-L // 128)
    diag = np.zeros((1, nb, nb), np.uint8)
    for k in range(nb):
        diag[0, k, k] = 1
    o, l = _oracle_mask(p, kc, vc, diag, causal=True, lib=lib)
    _, _, _, pt = _meta(p, lib)
    lens = [min(128, L - 128 * k) for k in range(nb)]
    per = 128 // p.page_size
    pts = np.full((nb, per), pt[0, 0], np.int32)
    for k in range(nb):
        row = pt[0, k * per:k * per + -(-lens[k] // p.page_size)]
        pts[k, :row.shape[0]] = row
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    os_, ls_ = oracle.attention(p.q, kc, vc, pts, cu, cu, num_q_heads=4, num_kv_heads=2, head_dim=8,
                                page_size=p.page_size, causal=True, scale=p.scale, lib=lib)
    assert np.array_equal(o, os_) and np.array_equal(l, ls_), "block-diagonal mask != split requests"


def check_block_mask_hidden_prefix(lib=None):
    """Non-causal attention with key block 0 hidden for every query equals
    attention over the keys from 128 on (the page table shifted by 128
    keys)."""
    p = W.small_problem(74, [200, 140], [30, 9], num_q_heads=4, num_kv_heads=2, head_dim=8, page_size=4,
                        causal=False)
    kc, vc = stored_caches(p, lib)
    nk = -(-int(p.device_len.max()) // 128)
    m = np.ones((p.num_seqs, 1, nk), np.uint8)
    m[:, :, 0] = 0
    o, l = _oracle_mask(p, kc, vc, m, causal=False, lib=lib)
    cu_q, cu_k, _, pt = _meta(p, lib)
    shift = 128 // p.page_size
    Lk2 = (p.device_len - 128).astype(np.int64)
    cu_k2 = np.concatenate([[0], np.cumsum(Lk2)]).astype(np.int32)
    o2, l2 = oracle.attention(p.q, kc, vc, np.ascontiguousarray(pt[:, shift:]), cu_q, cu_k2,
                              num_q_heads=4, num_kv_heads=2, head_dim=8, page_size=p.page_size,
                              causal=False, scale=p.scale, lib=lib)
    assert np.array_equal(o, o2) and np.array_equal(l, l2), "hidden first key block != shifted table"


ALL_CHECKS = [check_block_mask_brute_force, check_block_mask_closed_forms,
              check_block_mask_diagonal_is_split, check_block_mask_hidden_prefix,
              check_window_brute_force, check_window_closed_forms, check_window_is_truncated_cache,
              check_rope_table, check_rope_complex, check_rope_relative_position, check_round_bf16,
              check_e4m3_codec, check_store_fp8, check_attention_fp8_exact_values, check_store, check_metadata, check_golden, check_brute_force, check_equal_scores,
              check_single_key, check_dominant_key, check_empty, check_sdpa_library,
              check_decode_is_last_prefill_row, check_extend_is_prefill_tail,
              check_gqa_equals_repeated_mha, check_page_size_equivalence,
              check_permutation_invariance, check_shared_prefix, check_online_and_split_merge,
              check_threads_and_rows_invariance]
