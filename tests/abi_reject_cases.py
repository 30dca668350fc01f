"""Malformed C-ABI calls that libpa must reject on the host, before any launch.

The pointers in these calls are made-up addresses, so a call that slipped
past its checks would launch a kernel on memory that does not exist.
tests/test_abi_cpu.py therefore runs this file as a child process with
CUDA_VISIBLE_DEVICES='' (no GPU visible): a regressed check then fails with a
CUDA error status instead of touching a GPU.  Run as a script, it prints one
JSON object {case id: [status, last error]}.
"""
from __future__ import annotations

import ctypes
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

OK, INVALID, UNSUPPORTED = 0, 1, 2

PREFILL_BASE = dict(q=0x1000, k_cache=0x2000, v_cache=0x3000, page_table=0x4000, page_table_stride=64,
                    total_q=64, cu_seqlens_q=0x5000, cu_seqlens_k=0x6000, num_seqs=2, max_seqlen_q=16,
                    max_seqlen_k=32, num_q_heads=8, num_kv_heads=2, head_dim=128, page_size=16,
                    num_pages=100, causal=1, scale=0.1, out=0x7000, lse=None, lse_stride=0,
                    scheduler=0x9000)

DECODE_BASE = dict(q=0x1000, k_cache=0x2000, v_cache=0x3000, page_table=0x4000, page_table_stride=64,
                   cache_seqlens=0x5000, num_seqs=2, max_seqlen_k=4096, num_q_heads=8,
                   num_kv_heads=2, head_dim=128, page_size=16, num_pages=1000, scale=0.1,
                   out=0x7000, lse=None, workspace=0x8000, workspace_bytes=16, kv_chunk=0)

ROPE_BASE = dict(q=0x1000, q_out=0x1000, k=0x2000, v=0x3000, positions=0x4000, cos_sin=0x5000, max_pos=64,
                 rot_dim=128, interleaved=0, slot_mapping=0x6000, num_tokens=4, num_q_heads=8,
                 num_kv_heads=2, head_dim=128, k_cache=0x7000, v_cache=0x8000, num_slots=64, kv_dtype=0)

# (id, changed fields, expected status)
PREFILL_CASES = [
    ("head_dim96", dict(head_dim=96), UNSUPPORTED),
    ("page8", dict(page_size=8), UNSUPPORTED),
    ("heads6_4", dict(num_q_heads=6, num_kv_heads=4), INVALID),
    ("group16", dict(num_q_heads=32, num_kv_heads=2), UNSUPPORTED),
    ("misaligned_q", dict(q=0x1001), INVALID),
    ("null_out", dict(out=0), INVALID),
    ("q_longer_than_k", dict(max_seqlen_q=64, max_seqlen_k=32), INVALID),
    ("causal2", dict(causal=2), INVALID),
    ("table_stride", dict(page_table_stride=1), INVALID),
    ("scale_nan", dict(scale=float("nan")), INVALID),
    ("scale_zero", dict(scale=0.0), INVALID),
    ("scale_negative", dict(scale=-0.1), INVALID),
    ("scale_inf", dict(scale=float("inf")), INVALID),
    ("window_negative", dict(sliding_window=-3), INVALID),
    ("no_scheduler", dict(scheduler=0), INVALID),
    ("misaligned_scheduler", dict(scheduler=0x9004), INVALID),
]

DECODE_CASES = [
    ("head_dim80", dict(head_dim=80), UNSUPPORTED),
    ("chunk24", dict(kv_chunk=24), INVALID),
    ("chunk_negative", dict(kv_chunk=-16), INVALID),
    ("no_workspace", dict(workspace=0), INVALID),
    ("small_workspace", dict(workspace_bytes=16), INVALID),     # far too small for 4096 keys
    ("misaligned_pool", dict(k_cache=0x2008), INVALID),
    ("table_stride", dict(page_table_stride=8), INVALID),
    ("too_many_seqs", dict(num_seqs=20000), UNSUPPORTED),
    ("kv_dtype2", dict(kv_dtype=2), INVALID),
    ("fp8_no_scales", dict(kv_dtype=1), INVALID),
    ("window_negative", dict(sliding_window=-1), INVALID),
    ("scale_negative", dict(scale=-0.125), INVALID),
    ("scale_inf", dict(scale=float("inf")), INVALID),
    # 16384 sequences x 2^17 keys x 8 KV heads: the key-range arithmetic of the
    # split layout would leave int32 (shared prefixes make such lengths legal)
    ("keys_overflow_int32", dict(num_seqs=16384, max_seqlen_k=1 << 17, num_q_heads=32, num_kv_heads=8,
                                 page_table_stride=1 << 13, num_pages=1 << 20, kv_chunk=1 << 16), UNSUPPORTED),
]

# pa_decode_noalloc with sizes whose split scratch exceeds its fixed 32 MiB
NOALLOC_CASES = [
    ("oversized_scratch", dict(num_seqs=4096, max_seqlen_k=32768, num_q_heads=32, num_kv_heads=8,
                               page_table_stride=2048, num_pages=1 << 20, kv_chunk=128, workspace=None,
                               workspace_bytes=0), UNSUPPORTED),
]

# pa_mixed_batch: a prefill half and a decode half that cannot share one launch
MIXED_PREFILL = dict(PREFILL_BASE, num_q_heads=32, num_kv_heads=8, max_seqlen_k=4096, page_table_stride=256,
                     num_pages=1000)
MIXED_DECODE = dict(DECODE_BASE, num_q_heads=32, num_kv_heads=8, page_table_stride=256, workspace_bytes=1 << 30)
MIXED_CASES = [
    ("other_pools", dict(k_cache=0x9100), {}, INVALID),
    ("other_head_dim", {}, dict(head_dim=64), INVALID),
    ("fp8_other_scales", dict(kv_dtype=1, k_scale=0xA000, v_scale=0xA100), dict(kv_dtype=1, k_scale=0xA200, v_scale=0xA100),
     INVALID),
    ("mixed_pool_types", dict(kv_dtype=1, k_scale=0xA000, v_scale=0xA100), {}, INVALID),
    ("prefill_window", dict(sliding_window=64), {}, UNSUPPORTED),
    ("odd_group", dict(num_q_heads=8, num_kv_heads=8), dict(num_q_heads=8, num_kv_heads=8), UNSUPPORTED),
    ("kv_heads_not_4", dict(num_q_heads=12, num_kv_heads=6), dict(num_q_heads=12, num_kv_heads=6), UNSUPPORTED),
    ("overlap_previous", {}, dict(overlap_previous=1), INVALID),
    ("no_scheduler", dict(scheduler=0), {}, INVALID),
    # FP8 at d = 64: the standalone decode groups 8 KV heads (2^30 rows pass its
    # check), the mixed launch groups 4 (2^31 rows do not)
    ("decode_rows_overflow", dict(kv_dtype=1, k_scale=0xA000, v_scale=0xA100, head_dim=64, num_pages=1 << 20),
     dict(kv_dtype=1, k_scale=0xA000, v_scale=0xA100, head_dim=64, num_seqs=16384, max_seqlen_k=1 << 16,
          page_table_stride=1 << 12, num_pages=1 << 20, kv_chunk=1 << 15, workspace_bytes=1 << 50), UNSUPPORTED),
]

ROPE_CASES = [
    ("rot72", dict(rot_dim=72), UNSUPPORTED),
    ("rot256", dict(rot_dim=256), UNSUPPORTED),
    ("interleaved2", dict(interleaved=2), INVALID),
    ("fp8_no_scales", dict(kv_dtype=1), INVALID),
    ("misaligned_q", dict(q=0x1008), INVALID),
    ("head_dim72", dict(head_dim=72), UNSUPPORTED),
]

# positional pa_store_kv / pa_store_kv_fp8 calls
STORE_CASES = [
    ("misaligned_k", "pa_store_kv", (0x1001, 0x2000, 0x3000, 4, 0x4000, 0x5000, 64, 2, 64, None), INVALID),
    ("negative_tokens", "pa_store_kv", (0x1000, 0x2000, 0x3000, -1, 0x4000, 0x5000, 64, 2, 64, None), INVALID),
    ("row_not_16b", "pa_store_kv", (0x1000, 0x2000, 0x3000, 4, 0x4000, 0x5000, 64, 1, 4, None), UNSUPPORTED),
    ("zero_tokens", "pa_store_kv", (0, 0, 0, 0, 0, 0, 0, 2, 64, None), OK),
    ("fp8_no_k_scale", "pa_store_kv_fp8",
     (0x1000, 0x2000, 0x3000, 4, 0x4000, 0x5000, 64, 2, 64, None, 0x6000, None), INVALID),
    ("fp8_head_dim72", "pa_store_kv_fp8",
     (0x1000, 0x2000, 0x3000, 4, 0x4000, 0x5000, 64, 2, 72, 0x6000, 0x7000, None), UNSUPPORTED),
    ("fp8_misaligned_k", "pa_store_kv_fp8",
     (0x1008, 0x2000, 0x3000, 4, 0x4000, 0x5000, 64, 2, 64, 0x6000, 0x7000, None), INVALID),
    ("fp8_zero_tokens", "pa_store_kv_fp8", (0, 0, 0, 0, 0, 0, 0, 2, 64, None, None, None), OK),
]


def all_case_ids():
    ids = [f"prefill/{c[0]}" for c in PREFILL_CASES] + [f"decode/{c[0]}" for c in DECODE_CASES]
    ids += [f"noalloc/{c[0]}" for c in NOALLOC_CASES] + [f"rope/{c[0]}" for c in ROPE_CASES]
    ids += [f"mixed/{c[0]}" for c in MIXED_CASES]
    return ids + [f"store/{c[0]}" for c in STORE_CASES]


def expected():
    out = {f"prefill/{i}": s for i, _, s in PREFILL_CASES}
    out.update({f"decode/{i}": s for i, _, s in DECODE_CASES})
    out.update({f"noalloc/{i}": s for i, _, s in NOALLOC_CASES})
    out.update({f"rope/{i}": s for i, _, s in ROPE_CASES})
    out.update({f"store/{i}": s for i, _, _, s in STORE_CASES})
    out.update({f"mixed/{i}": s for i, _, _, s in MIXED_CASES})
    return out


def run_all() -> dict:
    from paged_kv_flashattention_gb300 import _lib
    lib = _lib.load()
    res = {}

    def rec(key, status):
        res[key] = [int(status), lib.pa_last_error().decode(errors="replace")]

    for i, kw, _ in PREFILL_CASES:
        p = _lib.PrefillParams(**{**PREFILL_BASE, **kw})
        rec(f"prefill/{i}", lib.pa_prefill(ctypes.byref(p), None))
    for i, kw, _ in DECODE_CASES:
        p = _lib.DecodeParams(**{**DECODE_BASE, **kw})
        rec(f"decode/{i}", lib.pa_decode(ctypes.byref(p), None))
    for i, kw, _ in NOALLOC_CASES:
        p = _lib.DecodeParams(**{**DECODE_BASE, **kw})
        rec(f"noalloc/{i}", lib.pa_decode_noalloc(ctypes.byref(p), None))
    for i, kw, _ in ROPE_CASES:
        p = _lib.RopeStoreParams(**{**ROPE_BASE, **kw})
        rec(f"rope/{i}", lib.pa_rope_store_kv(ctypes.byref(p), None))
    for i, fn, args, _ in STORE_CASES:
        rec(f"store/{i}", getattr(lib, fn)(*args))
    for i, kp, kd, _ in MIXED_CASES:
        p = _lib.PrefillParams(**{**MIXED_PREFILL, **kp})
        d = _lib.DecodeParams(**{**MIXED_DECODE, **kd})
        rec(f"mixed/{i}", lib.pa_mixed_batch(ctypes.byref(p), ctypes.byref(d), None))
    return res


if __name__ == "__main__":
    print(json.dumps(run_all()))
