"""GPU parity of the KV store and the page-table metadata kernel: bit-exact
against the oracle on every workload and on the edge cases."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from pa_harness import DeviceProblem, bf16_dev, bf16_host

pytestmark = pytest.mark.gpu


PROBLEMS = {"cfg1": (1, None), "cfg2": (2, None), "cfg3": (3, None), "cfg4_p16": (4, None),
            "cfg4_p1": (4, "p1")}


def _problem(name, with_data=True):
    c, v = PROBLEMS[name]
    return W.config(c, v, with_data=with_data)


@pytest.mark.parametrize("name", list(PROBLEMS))
def test_store_bit_exact(cuda_device, name):
    import paged_kv_flashattention_gb300 as pa
    p = _problem(name)
    d = DeviceProblem(p, cuda_device)
    d.store()
    torch.cuda.synchronize()
    row = p.num_kv_heads * p.head_dim
    kc, vc = p.k_cache.copy(), p.v_cache.copy()
    oracle.store_kv(p.k_new.reshape(-1, row), p.v_new.reshape(-1, row), p.slot_mapping,
                    kc.reshape(-1, row), vc.reshape(-1, row))
    assert np.array_equal(bf16_host(d.k_cache), kc), f"{name}: K pool differs"
    assert np.array_equal(bf16_host(d.v_cache), vc), f"{name}: V pool differs"
    assert pa.device_error() == 0


def test_store_skips_padding_and_out_of_range(cuda_device):
    import paged_kv_flashattention_gb300 as pa
    rng = np.random.default_rng(7)
    slots, Hkv, d = 97, 2, 64
    kc0 = W.normal_bf16(rng, (slots, Hkv, d))
    vc0 = W.normal_bf16(rng, (slots, Hkv, d))
    sm = np.array([3, -1, 96, 0, -5, 50, 97, 1000], np.int32)  # 97 and 1000 are outside the pool
    k = W.normal_bf16(rng, (sm.size, Hkv, d))
    v = W.normal_bf16(rng, (sm.size, Hkv, d))
    kc_d, vc_d = bf16_dev(kc0, cuda_device), bf16_dev(vc0, cuda_device)
    pa.device_error()     # clear
    pa.store_kv(bf16_dev(k, cuda_device), bf16_dev(v, cuda_device), torch.from_numpy(sm).to(cuda_device),
                kc_d, vc_d)
    err = pa.device_error()
    assert err & 1, "an out-of-range slot must raise the page-range bit"
    kc, vc = kc0.copy(), vc0.copy()
    keep = (sm >= 0) & (sm < slots)
    kc[sm[keep]] = k[keep]
    vc[sm[keep]] = v[keep]
    assert np.array_equal(bf16_host(kc_d), kc)
    assert np.array_equal(bf16_host(vc_d), vc)


def test_store_empty(cuda_device):
    import paged_kv_flashattention_gb300 as pa
    kc = torch.zeros((4, 16, 2, 64), dtype=torch.bfloat16, device=cuda_device)
    vc = torch.zeros_like(kc)
    e = torch.empty((0, 2, 64), dtype=torch.bfloat16, device=cuda_device)
    pa.store_kv(e, e, torch.empty(0, dtype=torch.int32, device=cuda_device), kc, vc)
    torch.cuda.synchronize()
    assert int(kc.view(torch.int16).abs().sum()) == 0


@pytest.mark.parametrize("name", list(PROBLEMS))
def test_page_table_bit_exact(cuda_device, name):
    import paged_kv_flashattention_gb300 as pa
    p = _problem(name, with_data=False)
    tt = torch.from_numpy(p.token_table).to(cuda_device)
    ti = torch.from_numpy(p.table_idx).to(cuda_device)
    mk = int(p.device_len.max())
    ncols = -(-mk // p.page_size)
    out = torch.full((p.num_seqs, ncols + 3), -12345, dtype=torch.int32, device=cuda_device)
    pa.build_page_table(tt, ti, mk, p.page_size, out=out)
    got = out.cpu().numpy()
    want = oracle.page_table_from_token_table(p.token_table, p.table_idx, mk, p.page_size)
    assert np.array_equal(got[:, :ncols], want)
    assert np.all(got[:, ncols:] == -12345), "columns past the last page must not be written"


def test_page_table_row_selection(cuda_device):
    """table_idx picks arbitrary rows (a dummy row included) in any order."""
    import paged_kv_flashattention_gb300 as pa
    p = W.small_problem(31, [40, 3, 17, 0], [1, 1, 1, 1], page_size=16)
    ti = np.array([2, 0, 3, 0, 1], np.int32)
    mk = 41
    got = pa.build_page_table(torch.from_numpy(p.token_table).to(cuda_device),
                              torch.from_numpy(ti).to(cuda_device), mk, 16).cpu().numpy()
    want = oracle.page_table_from_token_table(p.token_table, ti, mk, 16)
    assert np.array_equal(got, want)


def test_page_table_index_out_of_range(cuda_device):
    """A table_idx entry outside the token table's rows (device data) reads
    nothing: its row becomes -1 (a page the attention kernels skip) and
    PA_DEVERR_TABLE_INDEX is raised; the other rows are still exact."""
    import paged_kv_flashattention_gb300 as pa
    p = W.small_problem(32, [40, 3, 17], [1, 1, 1], page_size=16)
    rows = p.token_table.shape[0]
    ti = np.array([1, rows, 0, -1, 2], np.int32)
    mk = 41
    pa.device_error()                                   # clear earlier bits
    got = pa.build_page_table(torch.from_numpy(p.token_table).to(cuda_device),
                              torch.from_numpy(ti).to(cuda_device), mk, 16).cpu().numpy()
    assert pa.device_error() & 16
    ok = [0, 2, 4]
    want = oracle.page_table_from_token_table(p.token_table, ti[ok], mk, 16)
    assert np.array_equal(got[ok], want)
    assert np.all(got[[1, 3]] == -1)
