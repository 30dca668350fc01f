"""GPU parity of the FP8 (E4M3) KV path against the fp64 oracle: the FP8
store must equal the oracle's E4M3(x / scale) bit for bit, and decode over
FP8 pools must agree with the oracle's attention over the same codes and
scales within the bf16 contract (max abs <= 2e-2, mean abs <= 1e-3, lse
within 2e-3)."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from oracle_pins import _meta
from pa_harness import bf16_dev, compare

pytestmark = pytest.mark.gpu


def _u8(a, dev):
    return torch.from_numpy(np.ascontiguousarray(a)).to(dev)


def test_store_fp8_bit_exact(cuda_device):
    """Random bf16 bit patterns over 12 binades (about 1 in 16 is an exact
    E4M3 tie after a power-of-two scale), a head whose scale makes most
    quotients saturate, one whose quotients fall among the subnormals, and
    padding slots."""
    import paged_kv_flashattention_gb300 as pa
    rng = np.random.default_rng(401)
    T, Hkv, d, slots = 300, 4, 128, 512
    sign = rng.integers(0, 2, size=(T, Hkv, d), dtype=np.uint16) << 15
    expo = rng.integers(121, 133, size=(T, Hkv, d), dtype=np.uint16) << 7   # 2^-6 .. 2^5
    mant = rng.integers(0, 128, size=(T, Hkv, d), dtype=np.uint16)
    k = (sign | expo | mant).astype(np.uint16)
    v = W.normal_bf16(rng, (T, Hkv, d))
    ks = np.array([1.0, 0.0625, 0.001, 64.0], np.float32)     # exact, exact, saturating, subnormal
    vs = np.array([0.37, 0.011, 3.3, 0.5], np.float32)
    sm = rng.permutation(slots)[:T].astype(np.int32)
    sm[::17] = -1
    kc = W.e4m3_codes(rng, (slots, Hkv, d))
    vc = W.e4m3_codes(rng, (slots, Hkv, d))
    kd, vd = _u8(kc, cuda_device), _u8(vc, cuda_device)
    pa.store_kv_fp8(bf16_dev(k, cuda_device), bf16_dev(v, cuda_device), _u8(sm, cuda_device), kd, vd,
                    _u8(ks, cuda_device), _u8(vs, cuda_device))
    torch.cuda.synchronize()
    oracle.store_kv_fp8(k, v, sm, kc, vc, ks, vs)
    gk, gv = kd.cpu().numpy(), vd.cpu().numpy()
    bad = np.argwhere(gk != kc)
    assert bad.size == 0, f"{len(bad)} K codes differ, first at {bad[0]}: gpu {gk[tuple(bad[0])]:#x} oracle {kc[tuple(bad[0])]:#x}"
    assert np.array_equal(gv, vc), "V codes differ"
    # the saturating head really saturated, and subnormal codes were produced
    assert np.any((gk[:, 2] & 0x7F) == 0x7E) and np.any((gk[:, 3] & 0x78) == 0)


class FP8Problem:
    """A Problem's FP8 stand-in on the device: pools of random E4M3 codes
    (the poison page NaN), per-head scales, the new tokens stored by the FP8
    store on both sides."""

    def __init__(self, p: W.Problem, dev, seed: int):
        import paged_kv_flashattention_gb300 as pa
        self.p = p
        kc, vc, ks, vs = W.fp8_pools(p, seed)
        self.ks, self.vs = ks, vs
        self.k_cache, self.v_cache = _u8(kc, dev), _u8(vc, dev)
        self.k_scale, self.v_scale = _u8(ks, dev), _u8(vs, dev)
        self.q = bf16_dev(p.q, dev)
        pa.store_kv_fp8(bf16_dev(p.k_new, dev), bf16_dev(p.v_new, dev), _u8(p.slot_mapping, dev),
                        self.k_cache, self.v_cache, self.k_scale, self.v_scale)
        oracle.store_kv_fp8(p.k_new, p.v_new, p.slot_mapping, kc.reshape(-1, p.num_kv_heads, p.head_dim),
                            vc.reshape(-1, p.num_kv_heads, p.head_dim), ks, vs)
        self.kc, self.vc = kc, vc
        from paged_kv_flashattention_gb300 import metadata
        self.meta = metadata.prepare(p.cached_len, p.extend_len, _u8(p.token_table, dev),
                                     _u8(p.table_idx, dev), p.page_size)
        torch.cuda.synchronize()
        assert np.array_equal(self.k_cache.cpu().numpy(), kc), "FP8 store differs from the oracle"
        assert np.array_equal(self.v_cache.cpu().numpy(), vc), "FP8 store differs from the oracle"

    def decode(self, kv_chunk=0):
        import paged_kv_flashattention_gb300 as pa
        B, Hq = self.p.num_seqs, self.p.num_q_heads
        lse = torch.empty((B, Hq), dtype=torch.float32, device=self.q.device)
        out = pa.decode(self.q, self.k_cache, self.v_cache, self.meta.page_table, self.meta.cache_seqlens,
                        self.meta.max_seqlen_k, scale=self.p.scale, lse=lse, kv_chunk=kv_chunk,
                        k_scale=self.k_scale, v_scale=self.v_scale)
        return out, lse

    def prefill(self):
        import paged_kv_flashattention_gb300 as pa
        Tq, Hq = self.q.shape[0], self.p.num_q_heads
        lse = torch.empty((Hq, max(Tq, 1)), dtype=torch.float32, device=self.q.device)
        m = self.meta
        out = pa.prefill(self.q, self.k_cache, self.v_cache, m.page_table, m.cu_seqlens_q, m.cu_seqlens_k,
                         m.max_seqlen_q, m.max_seqlen_k, causal=self.p.causal, scale=self.p.scale,
                         page_size=self.p.page_size, lse=lse, k_scale=self.k_scale, v_scale=self.v_scale)
        return out, lse

    def oracle(self, rows=None):
        p = self.p
        cu_q, cu_k, _, pt = _meta(p)
        return oracle.attention(p.q, self.kc, self.vc, pt, cu_q, cu_k, num_q_heads=p.num_q_heads,
                                num_kv_heads=p.num_kv_heads, head_dim=p.head_dim,
                                page_size=p.page_size, causal=p.causal, scale=p.scale, rows=rows,
                                k_scale=self.ks, v_scale=self.vs)


def _decode_fp8_check(p, dev, seed, kv_chunk=0, what=""):
    f = FP8Problem(p, dev, seed)
    out, lse = f.decode(kv_chunk=kv_chunk)
    torch.cuda.synchronize()
    ref, ref_lse = f.oracle()
    return compare(out, ref.reshape(out.shape), what or p.name, lse_gpu=lse,
                   lse_ref=ref_lse.reshape(lse.shape))


def test_tiny_decode_fp8(cuda_device):
    for chunk in (0, 16, 48):
        _decode_fp8_check(W.config(1), cuda_device, 501, kv_chunk=chunk, what=f"tiny fp8 C{chunk}")


def test_llama32_1b_decode_fp8_full(cuda_device):
    """B=64, Hq 32 / Hkv 8, d 64, contexts U[128, 4096], every output row."""
    _decode_fp8_check(W.config(2), cuda_device, 502)


EDGE_LENGTHS = [1, 15, 16, 17, 33, 100, 257]


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("hq,hkv", [(4, 4), (8, 4), (16, 4), (32, 4), (12, 6), (8, 1)])
@pytest.mark.parametrize("page", [1, 16])
def test_decode_fp8_edge_matrix(cuda_device, d, hq, hkv, page):
    Lk = np.array(EDGE_LENGTHS, np.int32)
    p = W.small_problem(1500 + d + hq + page, Lk - 1, np.ones_like(Lk), num_q_heads=hq,
                        num_kv_heads=hkv, head_dim=d, page_size=page)
    for chunk in (0, 16, 64):
        _decode_fp8_check(p, cuda_device, 600 + chunk, kv_chunk=chunk,
                          what=f"fp8 d{d} g{hq // hkv} P{page} C{chunk}")


def test_decode_fp8_long_contexts(cuda_device):
    """Contexts up to 16K over the mixed batch's head shape (d 128, Hq 32 /
    Hkv 8), sampled rows of every sequence."""
    rng = np.random.default_rng(503)
    Lk = np.exp(rng.uniform(np.log(512), np.log(16384), size=24)).astype(np.int32)
    p = W.small_problem(503, Lk - 1, np.ones_like(Lk), num_q_heads=32, num_kv_heads=8,
                        head_dim=128, page_size=16)
    _decode_fp8_check(p, cuda_device, 504, what="fp8 long contexts")


def _sample_rows(p, frac, seed):
    """Every request's first and last 3 rows, plus a random fraction; all heads."""
    rng = np.random.default_rng(seed)
    cu = np.concatenate([[0], np.cumsum(p.extend_len)])
    toks = set()
    for b in range(p.num_seqs):
        toks.update(range(cu[b], min(cu[b] + 3, cu[b + 1])))
        toks.update(range(max(cu[b], cu[b + 1] - 3), cu[b + 1]))
    T = int(cu[-1])
    toks.update(int(t) for t in rng.choice(T, size=max(1, int(T * frac)), replace=False))
    toks = np.array(sorted(int(t) for t in toks), np.int64)
    heads = np.arange(p.num_q_heads, dtype=np.int64)
    return np.stack(np.meshgrid(toks, heads, indexing="ij"), axis=-1).reshape(-1, 2)


def _prefill_fp8_check(p, dev, seed, rows=None, what=""):
    f = FP8Problem(p, dev, seed)
    out, lse = f.prefill()
    torch.cuda.synchronize()
    if rows is None:
        ref, ref_lse = f.oracle()
        return compare(out, ref, what or p.name, lse_gpu=lse[:, :ref.shape[0]].T.contiguous(), lse_ref=ref_lse)
    ref, ref_lse = f.oracle(rows=rows)
    t = torch.from_numpy(rows[:, 0]).to(dev)
    h = torch.from_numpy(rows[:, 1]).to(dev)
    return compare(out[t, h], ref, what or p.name, lse_gpu=lse[h, t], lse_ref=ref_lse)


def test_varlen_prefill_fp8_16x512(cuda_device):
    """16 requests x 512 prompt tokens over FP8 pools, every output row."""
    _prefill_fp8_check(W.config(3), cuda_device, 701)


@pytest.mark.parametrize("variant", [None, "p1"])
def test_extend_partial_hit_fp8(cuda_device, variant):
    p = W.config(4, variant)
    _prefill_fp8_check(p, cuda_device, 702, rows=_sample_rows(p, 0.2, 7), what=f"{p.name} fp8")


PREFILL_EDGE = [
    ([0, 0, 0, 0, 0], [1, 15, 16, 17, 129]),
    ([3, 16, 127, 128, 1000], [1, 16, 1, 129, 255]),
    ([0, 7, 0], [300, 0, 128]),
]


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("hq,hkv", [(4, 4), (8, 4), (32, 4)])
@pytest.mark.parametrize("page", [1, 16])
def test_prefill_fp8_edge_matrix(cuda_device, d, hq, hkv, page):
    for n, (cached, ext) in enumerate(PREFILL_EDGE):
        p = W.small_problem(2500 + 7 * n + d + hq + page, cached, ext, num_q_heads=hq,
                            num_kv_heads=hkv, head_dim=d, page_size=page)
        _prefill_fp8_check(p, cuda_device, 800 + n, what=f"fp8 prefill d{d} g{hq // hkv} P{page} case{n}")
