"""Shared helpers for the GPU parity tests: move a workloads.Problem to the
device, run the product path through the C ABI, run the oracle on the same
inputs, and compare with the contract's tolerances."""
from __future__ import annotations

import numpy as np
import torch

import oracle
import workloads as W
from oracle_pins import run_oracle, stored_caches

# Tolerances for bf16 outputs with fp32 accumulation against the fp64 oracle.
TOL_MAX_ABS = 2e-2
TOL_MEAN_ABS = 1e-3
TOL_LSE_ABS = 2e-3


def bf16_dev(a: np.ndarray, dev) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.bfloat16)


def bf16_host(t: torch.Tensor) -> np.ndarray:
    return t.detach().view(torch.int16).cpu().numpy().view(np.uint16)


def to_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


class DeviceProblem:
    """Device copies of a Problem's inputs (pool, q, new K/V, token table)."""

    def __init__(self, p: W.Problem, dev):
        self.p = p
        self.dev = dev
        self.k_cache = bf16_dev(p.k_cache, dev)
        self.v_cache = bf16_dev(p.v_cache, dev)
        self.q = bf16_dev(p.q, dev)
        self.k_new = bf16_dev(p.k_new, dev)
        self.v_new = bf16_dev(p.v_new, dev)
        self.slot_mapping = torch.from_numpy(p.slot_mapping).to(dev)
        self.token_table = torch.from_numpy(p.token_table).to(dev)
        self.table_idx = torch.from_numpy(p.table_idx).to(dev)

    def store(self):
        import paged_kv_flashattention_gb300 as pa
        pa.store_kv(self.k_new, self.v_new, self.slot_mapping, self.k_cache, self.v_cache)

    def metadata(self):
        from paged_kv_flashattention_gb300 import metadata
        return metadata.prepare(self.p.cached_len, self.p.extend_len, self.token_table,
                                self.table_idx, self.p.page_size)

    def decode(self, kv_chunk=0, with_lse=True):
        import paged_kv_flashattention_gb300 as pa
        m = self.metadata()
        B, Hq = self.p.num_seqs, self.p.num_q_heads
        lse = torch.empty((B, Hq), dtype=torch.float32, device=self.dev) if with_lse else None
        out = pa.decode(self.q, self.k_cache, self.v_cache, m.page_table, m.cache_seqlens,
                        m.max_seqlen_k, scale=self.p.scale, lse=lse, kv_chunk=kv_chunk)
        return out, lse

    def prefill(self, with_lse=True):
        import paged_kv_flashattention_gb300 as pa
        m = self.metadata()
        Tq, Hq = self.q.shape[0], self.p.num_q_heads
        lse = torch.empty((Hq, max(Tq, 1)), dtype=torch.float32, device=self.dev) if with_lse else None
        out = pa.prefill(self.q, self.k_cache, self.v_cache, m.page_table, m.cu_seqlens_q,
                         m.cu_seqlens_k, m.max_seqlen_q, m.max_seqlen_k, causal=self.p.causal,
                         scale=self.p.scale, lse=lse)
        return out, lse


def compare(out_gpu: torch.Tensor, ref: np.ndarray, what: str, *, lse_gpu=None, lse_ref=None,
            tol_max=TOL_MAX_ABS, tol_mean=TOL_MEAN_ABS):
    """Assert bf16 GPU output is within tolerance of the fp64 oracle.  Returns
    the statistics (max/mean abs, max rel, cosine)."""
    g = to_f64(out_gpu).reshape(ref.shape)
    assert np.all(np.isfinite(g)), f"{what}: NaN/Inf in GPU output"
    err = np.abs(g - ref)
    stats = {"max_abs": float(err.max()) if err.size else 0.0,
             "mean_abs": float(err.mean()) if err.size else 0.0}
    if err.size:
        denom = np.linalg.norm(g.ravel()) * np.linalg.norm(ref.ravel())
        stats["cosine"] = float(np.dot(g.ravel(), ref.ravel()) / denom) if denom > 0 else 1.0
    assert stats["max_abs"] <= tol_max, f"{what}: max abs err {stats['max_abs']:.4g} > {tol_max}"
    assert stats["mean_abs"] <= tol_mean, f"{what}: mean abs err {stats['mean_abs']:.4g} > {tol_mean}"
    if lse_gpu is not None:
        lg = lse_gpu.detach().cpu().numpy().astype(np.float64).reshape(lse_ref.shape)
        fin = np.isfinite(lse_ref)
        assert np.array_equal(np.isfinite(lg), fin), f"{what}: lse finiteness differs"
        if fin.any():
            le = float(np.max(np.abs(lg[fin] - lse_ref[fin])))
            stats["lse_max_abs"] = le
            assert le <= TOL_LSE_ABS, f"{what}: lse max abs err {le:.4g} > {TOL_LSE_ABS}"
        assert np.all(lg[~fin] == -np.inf), f"{what}: empty rows must have lse = -inf"
    return stats


def oracle_decode_ref(p: W.Problem, rows=None):
    """Oracle result for a decode Problem (store first): out [B, Hq, d], lse [B, Hq]."""
    return run_oracle(p, rows=rows)


def oracle_ref(p: W.Problem, rows=None):
    return run_oracle(p, rows=rows)


__all__ = ["DeviceProblem", "compare", "oracle_ref", "oracle_decode_ref", "bf16_dev", "bf16_host",
           "to_f64", "stored_caches", "oracle", "W"]
