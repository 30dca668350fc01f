"""GPU parity of the fused RoPE + K/V store against the fp64 oracle.

The kernel rotates in fp32 (each product and the sum rounded) from an fp32
table and rounds to bf16; the oracle rotates exactly in fp64 from its own
table and rounds once.  The fp32 path's absolute error on an output of pair
(a, b) is at most about 4 * 2^-24 * (|a| + |b|) (table entries within 2^-25,
two rounded products, one rounded sum), so the two bf16 results may differ
by one bf16 step plus that bound (the bound matters only for outputs near
zero, where cancellation makes the bf16 step tiny); at most 1 % of the
elements may differ at all.  The roundings can differ only where the exact
value lies within that bound of a bf16 rounding boundary, which for these
N(0, 1) inputs is at most about 0.08 % of the elements (the mean of
min(1, 2 * bound / bf16 step)); a systematic error such as truncation would
change about half of them.  Copies (v, elements past the rotated width) and
untouched pool rows must be bit-exact."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from pa_harness import bf16_dev, bf16_host

pytestmark = pytest.mark.gpu

MAX_POS = 4096


def _ulp_bf16(x: np.ndarray) -> np.ndarray:
    """One bf16 step at each value (float64)."""
    a = np.abs(x)
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    return np.exp2(np.maximum(e, -126.0) - 7.0)


def _pair_mag(x_bits, rot_dim, interleaved):
    """|a| + |b| of the pair each element belongs to (|x| past rot_dim)."""
    x = np.abs(W.bf16_bits_to_f32(x_bits).astype(np.float64))
    m = x.copy()
    h = rot_dim // 2
    if interleaved:
        s = x[..., 0:rot_dim:2] + x[..., 1:rot_dim:2]
        m[..., 0:rot_dim:2] = s
        m[..., 1:rot_dim:2] = s
    else:
        s = x[..., :h] + x[..., h:rot_dim]
        m[..., :h] = s
        m[..., h:rot_dim] = s
    return m


def _close_bf16(got_bits, want_f64, what, mag, max_frac=0.01):
    got = W.bf16_bits_to_f32(got_bits).astype(np.float64)
    want = W.bf16_bits_to_f32(oracle.round_bf16(want_f64)).astype(np.float64)
    diff = np.abs(got - want)
    bound = _ulp_bf16(want) * 1.0000001 + 4.0 * 2.0 ** -24 * mag
    bad = np.argwhere(diff > bound)
    assert bad.size == 0, (f"{what}: {len(bad)} elements beyond one bf16 step + the fp32 bound, first at "
                           f"{tuple(bad[0])}: gpu {got[tuple(bad[0])]!r} oracle {want_f64[tuple(bad[0])]!r}")
    frac = float(np.mean(diff > 0))
    assert frac <= max_frac, f"{what}: {frac:.4f} of the elements differ"
    return frac


def _setup(dev, seed, T=300, Hq=32, Hkv=8, d=128, slots=512):
    rng = np.random.default_rng(seed)
    q = W.normal_bf16(rng, (T, Hq, d))
    k = W.normal_bf16(rng, (T, Hkv, d))
    v = W.normal_bf16(rng, (T, Hkv, d))
    pos = rng.integers(0, MAX_POS, size=T).astype(np.int32)
    sm = rng.permutation(slots)[:T].astype(np.int32)
    sm[::13] = -1
    return rng, q, k, v, pos, sm


@pytest.mark.parametrize("rot_dim,interleaved", [(128, False), (128, True), (64, False), (64, True)])
def test_rope_store_bf16(cuda_device, rot_dim, interleaved):
    import paged_kv_flashattention_gb300 as pa
    dev = cuda_device
    rng, q, k, v, pos, sm = _setup(dev, 900 + rot_dim + interleaved)
    slots, Hkv, d = 512, 8, 128
    kc = W.normal_bf16(rng, (slots, Hkv, d))
    vc = W.normal_bf16(rng, (slots, Hkv, d))
    table = pa.rope_cos_sin_table(MAX_POS, rot_dim, 10000.0).to(dev)
    kcd, vcd = bf16_dev(kc, dev), bf16_dev(vc, dev)
    q_out = pa.rope_store_kv(bf16_dev(q, dev), bf16_dev(k, dev), bf16_dev(v, dev),
                             torch.from_numpy(pos).to(dev), table, torch.from_numpy(sm).to(dev), kcd, vcd,
                             interleaved=interleaved)
    torch.cuda.synchronize()
    c, s_ = oracle.rope_table(MAX_POS, rot_dim, 10000.0)
    _close_bf16(bf16_host(q_out), oracle.rope_rotate(q, pos, c, s_, rot_dim=rot_dim, interleaved=interleaved), "q",
                _pair_mag(q, rot_dim, interleaved))
    k_rot = oracle.rope_rotate(k, pos, c, s_, rot_dim=rot_dim, interleaved=interleaved)
    gk, gv = bf16_host(kcd), bf16_host(vcd)
    live = sm >= 0
    _close_bf16(gk[sm[live]], k_rot[live], "stored k", _pair_mag(k[live], rot_dim, interleaved))
    assert np.array_equal(gv[sm[live]], v[live]), "v rows must be copied bit for bit"
    untouched = np.setdiff1d(np.arange(slots), sm[live])
    assert np.array_equal(gk[untouched], kc[untouched]) and np.array_equal(gv[untouched], vc[untouched])


def test_rope_store_fp8(cuda_device):
    """FP8 pools: k is rotated, rounded to bf16 and quantised like
    pa_store_kv_fp8; v codes are bit-exact."""
    import paged_kv_flashattention_gb300 as pa
    dev = cuda_device
    rng, q, k, v, pos, sm = _setup(dev, 950)
    slots, Hkv, d = 512, 8, 128
    kc = W.e4m3_codes(rng, (slots, Hkv, d))
    vc = W.e4m3_codes(rng, (slots, Hkv, d))
    ks = rng.uniform(0.01, 0.05, Hkv).astype(np.float32)
    vs = rng.uniform(0.01, 0.05, Hkv).astype(np.float32)
    table = pa.rope_cos_sin_table(MAX_POS, d, 500000.0).to(dev)
    kcd, vcd = torch.from_numpy(kc).to(dev), torch.from_numpy(vc).to(dev)
    pa.rope_store_kv(bf16_dev(q, dev), bf16_dev(k, dev), bf16_dev(v, dev), torch.from_numpy(pos).to(dev), table,
                     torch.from_numpy(sm).to(dev), kcd, vcd, k_scale=torch.from_numpy(ks).to(dev),
                     v_scale=torch.from_numpy(vs).to(dev))
    torch.cuda.synchronize()
    c, s_ = oracle.rope_table(MAX_POS, d, 500000.0)
    k_rot_bits = oracle.round_bf16(oracle.rope_rotate(k, pos, c, s_, rot_dim=d))
    ke, ve = kc.copy(), vc.copy()
    oracle.store_kv_fp8(k_rot_bits, v, sm, ke, ve, ks, vs)
    gk, gv = kcd.cpu().numpy(), vcd.cpu().numpy()
    assert np.array_equal(gv, ve), "v codes differ from the oracle's FP8 store"
    # k codes: equal except where the bf16 rotated k differed by one step;
    # then the decoded values differ by at most one E4M3 step
    vg, vo = oracle.e4m3_value(gk), oracle.e4m3_value(ke)
    a = np.abs(vo)
    e = np.maximum(np.floor(np.log2(np.where(a > 0, a, 1.0))), -6.0)
    assert np.all(np.abs(vg - vo) <= np.exp2(e - 3.0) * 1.0000001), "k codes differ by more than one step"
    assert float(np.mean(gk != ke)) <= 0.01


def test_rope_custom_table(cuda_device):
    """A table of arbitrary unit vectors (a scaled-RoPE stand-in) drives the
    rotation the same way on both sides."""
    import paged_kv_flashattention_gb300 as pa
    dev = cuda_device
    rng, q, k, v, pos, sm = _setup(dev, 970, T=64)
    theta = rng.uniform(-np.pi, np.pi, size=(MAX_POS, 64))
    table = np.concatenate([np.cos(theta), np.sin(theta)], axis=1).astype(np.float32)
    kc = W.normal_bf16(rng, (512, 8, 128))
    vc = W.normal_bf16(rng, (512, 8, 128))
    q_out = pa.rope_store_kv(bf16_dev(q, dev), bf16_dev(k, dev), bf16_dev(v, dev), torch.from_numpy(pos).to(dev),
                             torch.from_numpy(table).to(dev), torch.from_numpy(sm).to(dev),
                             bf16_dev(kc, dev), bf16_dev(vc, dev))
    torch.cuda.synchronize()
    want = oracle.rope_rotate(q, pos, table[:, :64].astype(np.float64), table[:, 64:].astype(np.float64),
                              rot_dim=128)
    _close_bf16(bf16_host(q_out), want, "q with a custom table", _pair_mag(q, 128, False))


def test_rope_in_place_and_bad_position(cuda_device):
    """q_out may be q; a position outside the table writes nothing for that
    token and raises PA_DEVERR_POSITION."""
    import paged_kv_flashattention_gb300 as pa
    dev = cuda_device
    rng, q, k, v, pos, sm = _setup(dev, 980, T=16)
    pos[5] = MAX_POS + 3
    table = pa.rope_cos_sin_table(MAX_POS, 128, 10000.0).to(dev)
    qd = bf16_dev(q, dev)
    kc = W.normal_bf16(rng, (512, 8, 128))
    kcd, vcd = bf16_dev(kc, dev), bf16_dev(W.normal_bf16(rng, (512, 8, 128)), dev)
    pa.device_error()
    pa.rope_store_kv(qd, bf16_dev(k, dev), bf16_dev(v, dev), torch.from_numpy(pos).to(dev), table,
                     torch.from_numpy(sm).to(dev), kcd, vcd, q_out=qd)
    err = pa.device_error()
    assert err & 8, f"expected PA_DEVERR_POSITION, got {err}"
    got = bf16_host(qd)
    assert np.array_equal(got[5], q[5]), "the bad token's q must be left as it was"
    ok = np.arange(16) != 5
    c, s_ = oracle.rope_table(MAX_POS, 128, 10000.0)
    _close_bf16(got[ok], oracle.rope_rotate(q[ok], pos[ok], c, s_, rot_dim=128), "in-place q",
                _pair_mag(q[ok], 128, False))
    if sm[5] >= 0:
        assert np.array_equal(bf16_host(kcd)[sm[5]], kc[sm[5]]), "the bad token's k must not be stored"
