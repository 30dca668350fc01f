"""Benchmark of the paged-KV attention path on one mixed continuous batch.

One STEP is one pass of the whole path over one batch: the KV store of every
new token (256 decode tokens + 2 x 2048 prefill tokens), the metadata of both
sub-batches (host seqlens -> pinned, non-blocking H2D; page tables sliced on
the device), causal prefill of the two 2048-token chunks, and split-KV decode
(+ LSE combine) of 256 sequences with contexts log-uniform in [512, 32768]
over a ~40 GB bf16 KV pool (Hq 32 / Hkv 8, d 128, page 16).

value    = algorithmic bytes of the step (decode K/V + q/o, prefill Q/K/V/O,
           store read+write) / device step time, in GB/s.  Inputs are resident
           in HBM; the step's decode reads ~8 GB, far larger than L2.
e2e      = the same bytes / step time through the public API with HOST
           buffers: q, new K/V and slot mapping copied H2D from pinned memory
           (double-buffered on a copy stream, overlapping the neighbouring
           steps' kernels)
           and both outputs copied back D2H inside the timed region.
roofline = the decode pass (split kernel + combine) against measured HBM
           bandwidth; prefill TFLOP/s against the measured bf16 peak is
           reported beside it.

--impl reference times the fp64 CPU oracle on a bounded sample of the same
workload (the benchmark's reference arm).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import workloads as W  # noqa: E402

METRIC = "paged-attn decode HBM GB/s; prefill TFLOP/s; fraction of GB300 roofline"
WORKLOAD = ("mixed_batch_llama3_8b: 256 decode seqs (context log-uniform [512, 32768]) + "
            "2 prefill chunks x 2048 (no cache hit), Hq 32 / Hkv 8, head_dim 128, page 16, "
            "bf16 KV pool 2 x 20 GB, seeded permuted page tables")
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in FALLBACK_PEAKS}, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


def source_sha256(kernel_files) -> str:
    """sha256 of the kernel's source files (csrc/, in the order given)."""
    h = hashlib.sha256()
    for f in kernel_files:
        h.update(open(os.path.join(ROOT, "paged_kv_flashattention_gb300", "csrc", f), "rb").read())
    return h.hexdigest()


def ncu_traffic(kernel_files, summary: str):
    """DRAM bytes per launch from a committed ncu summary, or None when the
    kernel's sources changed since the capture (the summary records their
    hash, source_sha256(kernel_files))."""
    try:
        text = open(os.path.join(ROOT, "profiles", summary)).read()
        want = re.search(r"source_sha256:\s*([0-9a-f]{64})", text).group(1)
        bytes_ = float(re.search(r"traffic_bytes_per_full_launch:\s*([0-9.eE+]+)", text).group(1))
        return bytes_ if source_sha256(kernel_files) == want else None
    except Exception:
        return None


# the sources of the two attention passes the roofline names
MIXED_SOURCES = ("mixed.cu", "prefill_impl.cuh", "decode_impl.cuh", "pa_device.cuh", "decode.cu")
DECODE_SOURCES = ("decode.cu", "decode_impl.cuh", "pa_device.cuh")


# --------------------------------------------------------------------------
class ClockSampler:
    """nvidia-smi sampling during the timed region."""

    FIELDS = ("clocks.sm,clocks.max.sm,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()
                out = ""
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        sm, mx, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in getattr(self, "lines", []):
            parts = [p.strip() for p in l.split(",")]
            if len(parts) < 6:
                continue
            try:
                sm.append(float(parts[0]))
                mx = max(mx, float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[2:6]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx or None,
                "reasons": sorted(reasons), "samples": len(sm)}


# --------------------------------------------------------------------------
class MixedBatch:
    """Device state of the mixed-batch workload (pool, inputs, buffers)."""

    def __init__(self, dev, seed_offset: int = 0):
        import torch
        import paged_kv_flashattention_gb300 as pa
        self.torch, self.pa, self.dev = torch, pa, dev
        cfg = W.config(5, with_data=False)
        self.dec, self.pre = cfg["decode"], cfg["prefill"]
        d, p = self.dec, self.pre
        self.Hq, self.Hkv, self.D, self.P = d.num_q_heads, d.num_kv_heads, d.head_dim, d.page_size
        shape = (d.num_pages, self.P, self.Hkv, self.D)
        self.k_cache = torch.empty(shape, dtype=torch.bfloat16, device=dev)
        self.v_cache = torch.empty(shape, dtype=torch.bfloat16, device=dev)
        W.fill_normal_device(self.k_cache, W.SEED_BASE + 50 + seed_offset)
        W.fill_normal_device(self.v_cache, W.SEED_BASE + 51 + seed_offset)
        # never-written slots past each sequence's end in its last page: NaN
        W.poison_tails_device(d, self.k_cache, self.v_cache)
        W.poison_tails_device(p, self.k_cache, self.v_cache)
        g = torch.Generator(device=dev)
        g.manual_seed(W.SEED_BASE + 52 + seed_offset)
        Tn = d.num_new_tokens + p.num_new_tokens
        self.q_dec = torch.randn((d.num_seqs, self.Hq, self.D), generator=g, device=dev).to(torch.bfloat16)
        self.q_pre = torch.randn((p.num_new_tokens, self.Hq, self.D), generator=g, device=dev).to(torch.bfloat16)
        self.k_new = torch.randn((Tn, self.Hkv, self.D), generator=g, device=dev).to(torch.bfloat16)
        self.v_new = torch.randn((Tn, self.Hkv, self.D), generator=g, device=dev).to(torch.bfloat16)
        self.slot_mapping = torch.from_numpy(np.concatenate([d.slot_mapping, p.slot_mapping])).to(dev)
        # global token-granular table: decode requests, then the prefill chunks
        width = max(d.token_table.shape[1], p.token_table.shape[1])
        tt = np.full((d.num_seqs + p.num_seqs, width), (d.num_pages - 1) * self.P, np.int32)
        tt[:d.num_seqs, :d.token_table.shape[1]] = d.token_table
        tt[d.num_seqs:, :p.token_table.shape[1]] = p.token_table
        self.token_table = torch.from_numpy(tt).to(dev)
        # rows of the token table: the decode requests, then the prefill chunks
        self.idx_all = torch.arange(d.num_seqs + p.num_seqs, dtype=torch.int32, device=dev)
        self.max_dec = int(d.device_len.max())
        self.out_dec = torch.empty_like(self.q_dec)
        self.out_pre = torch.empty_like(self.q_pre)
        ws = pa.decode_workspace_size(self.q_dec.shape, self.k_cache, self.max_dec, kv_chunk=256)
        self.workspace = torch.empty(max(ws, 16), dtype=torch.uint8, device=dev)
        width = -(-max(self.max_dec, int(p.device_len.max())) // self.P)
        self.pt_all = torch.empty((d.num_seqs + p.num_seqs, width), dtype=torch.int32, device=dev)
        # algorithmic work of one step
        ctx = d.device_len.astype(np.int64)
        self.decode_bytes = int(ctx.sum()) * self.Hkv * self.D * 2 * 2 + 2 * self.q_dec.numel() * 2
        pairs = sum(int(L) * (int(L) + 1) // 2 for L in p.extend_len)
        self.prefill_flops = 4 * self.D * self.Hq * pairs
        self.prefill_bytes = 2 * self.q_pre.numel() * 2 + 2 * p.num_new_tokens * self.Hkv * self.D * 2
        self.store_bytes = 2 * 2 * Tn * self.Hkv * self.D * 2
        self.step_bytes = self.decode_bytes + self.prefill_bytes + self.store_bytes
        self.launches_per_step = 5   # store, page table, prefill, decode split + combine
        self.num_sms = torch.cuda.get_device_properties(dev).multi_processor_count
        self.prefill_sms = 12        # overlapped schedule (0: phases in sequence)
        # "overlap": prefill on prefill_sms SMs, decode as its programmatic
        # dependent on the rest; "fused": both halves in one persistent launch
        # (pa_mixed_batch); "sequential": one phase after the other
        self.schedule = "fused"
        self.mixed_sched = torch.zeros(4, dtype=torch.int32, device=dev)
        self.fused_prefill_ctas = 12   # fused schedule: CTAs that take prefill tiles first (0 = automatic)
        self.fused_kv_chunk = 256      # fused schedule: the decode split layout's unit
        from paged_kv_flashattention_gb300.metadata import MixedMetadataBuilder
        # both halves' lengths in one copy, both page tables in one launch
        self.meta = MixedMetadataBuilder(dev, p.num_seqs, d.num_seqs)

    def step(self, timing: bool = False, concurrent: bool | None = None):
        """One pass of the path.  concurrent (the default unless timing):
        prefill runs on ``prefill_sms`` SMs and decode, launched as its
        programmatic dependent, on the others at the same time (prefill is
        tensor-bound, decode HBM-bound).  timing: the phases one after the
        other, with events between them."""
        torch, pa = self.torch, self.pa
        if concurrent is None:
            concurrent = not timing and self.prefill_sms > 0 and self.schedule == "overlap"
        fused = not timing and self.schedule == "fused"
        ev = None
        if timing:
            ev = [torch.cuda.Event(enable_timing=True) for _ in range(5)]
            ev[0].record()
        pa.store_kv(self.k_new, self.v_new, self.slot_mapping, self.k_cache, self.v_cache)
        mp, md = self.meta.prepare(self.pre.cached_len, self.pre.extend_len, self.dec.cached_len,
                                   self.dec.extend_len, self.token_table, self.idx_all, self.P,
                                   page_table_out=self.pt_all)
        if timing:
            ev[1].record()
        if fused:
            self._keep = (md, mp)
            self.fused_pass()
            return ev
        pa.prefill(self.q_pre, self.k_cache, self.v_cache, mp.page_table, mp.cu_seqlens_q, mp.cu_seqlens_k,
                   mp.max_seqlen_q, mp.max_seqlen_k, causal=True, out=self.out_pre,
                   max_ctas=self.prefill_sms if concurrent else 0)
        if timing:
            ev[2].record()
        pa.decode(self.q_dec, self.k_cache, self.v_cache, md.page_table, md.cache_seqlens, md.max_seqlen_k,
                  out=self.out_dec, workspace=self.workspace,
                  max_ctas=2 * (self.num_sms - self.prefill_sms) if concurrent else 0,
                  overlap_previous=concurrent)
        if timing:
            ev[3].record()
        self._keep = (md, mp)
        return ev


def _fused_pass(self):
    """The attention of one step in one launch (pa_mixed_batch: prefill and
    split-KV decode, then the combine) on the last step's metadata."""
    md, mp = self._keep
    self.pa.mixed_batch(self.q_pre, self.q_dec, self.k_cache, self.v_cache, mp.page_table, mp.cu_seqlens_q,
                        mp.cu_seqlens_k, mp.max_seqlen_q, mp.max_seqlen_k, md.page_table, md.cache_seqlens,
                        md.max_seqlen_k, causal=True, out_prefill=self.out_pre, out_decode=self.out_dec,
                        workspace=self.workspace, scheduler=self.mixed_sched,
                        prefill_ctas=self.fused_prefill_ctas, kv_chunk=self.fused_kv_chunk)


MixedBatch.fused_pass = _fused_pass


def schedule_text(mb) -> str:
    if mb.schedule == "fused":
        n = mb.fused_prefill_ctas or "automatically chosen"
        return (f"prefill and decode in one persistent launch: {n} CTAs take the prefill tiles first, the "
                f"others start on decode key ranges at once (T-ranges of {mb.fused_kv_chunk} keys), then "
                f"the LSE combine")
    if mb.schedule == "overlap" and mb.prefill_sms > 0:
        return f"prefill on {mb.prefill_sms} SMs overlapped with decode on the other {mb.num_sms - mb.prefill_sms}"
    return "phases in sequence"


def schedule_compare(mb, steps: int) -> dict:
    """Median step time of every schedule of the same step (events around
    every step, back to back), the chosen one restored afterwards."""
    import torch
    keep = mb.schedule, mb.prefill_sms, mb.fused_prefill_ctas, mb.fused_kv_chunk
    out = {}
    runs = [("overlap", "overlap", keep[1] or 12, 0, 0), ("sequential", "sequential", 0, 0, 0),
            ("fused", "fused", 0, keep[2], keep[3]), ("fused_prefill_share_automatic", "fused", 0, 0, keep[3]),
            ("fused_prefill_on_all_ctas", "fused", 0, mb.num_sms, keep[3]),
            ("fused_ranges_1024", "fused", 0, keep[2], 1024)]
    for name, sched, sms, fpc, kc in runs:
        mb.schedule, mb.prefill_sms, mb.fused_prefill_ctas, mb.fused_kv_chunk = sched, sms, fpc, kc
        for _ in range(3):
            mb.step()
        pairs = []
        for _ in range(steps):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            mb.step()
            b.record()
            pairs.append((a, b))
        torch.cuda.synchronize()
        t = sorted(a.elapsed_time(b) for a, b in pairs)
        out[name] = {"ms_median": round(_pct(t, 50), 4), "ms_p95": round(_pct(t, 95), 4),
                     "gbs": round(mb.step_bytes / (_pct(t, 50) * 1e-3) / 1e9, 1)}
    mb.schedule, mb.prefill_sms, mb.fused_prefill_ctas, mb.fused_kv_chunk = keep
    return out



def roofline_block(mb, fused_ms, dec_gbs, peaks, peak_src) -> dict:
    """The dominant kernel of the timed step against the measured HBM copy
    peak: the mixed-batch launch (with its combine) under the fused schedule,
    else the decode pass (split kernel + combine)."""
    if fused_ms:
        ms = _pct(fused_ms, 50)
        nbytes = mb.decode_bytes + mb.prefill_bytes
        gbs = nbytes / (ms * 1e-3) / 1e9
        return {"bound": "hbm", "kernel": "mixed-batch launch (prefill tiles and split-KV decode in one "
                "persistent kernel) + LSE combine", "achieved": round(gbs, 1), "peak": peaks["hbm_gbs"],
                "unit": "GB/s", "frac": round(gbs / peaks["hbm_gbs"], 4), "peak_source": peak_src,
                "bytes_per_launch": nbytes, "ms_median": round(ms, 4), "ms_p95": round(_pct(fused_ms, 95), 4),
                "traffic": ncu_traffic(MIXED_SOURCES, "mixed_batch_launch.md")}
    return {"bound": "hbm", "kernel": "decode pass (split-KV kernel + LSE combine)",
            "achieved": round(dec_gbs, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
            "frac": round(dec_gbs / peaks["hbm_gbs"], 4), "peak_source": peak_src,
            "bytes_per_launch": mb.decode_bytes,
            "traffic": ncu_traffic(DECODE_SOURCES, "decode_mixed_batch.md")}


def _pct(sorted_vals, q):
    """q-th percentile (nearest rank) of an ascending list."""
    if not sorted_vals:
        return float("nan")
    i = min(len(sorted_vals) - 1, max(0, int(math.ceil(q / 100.0 * len(sorted_vals))) - 1))
    return float(sorted_vals[i])


# The other workloads of the path, each timed on its own in the default run
# (config name -> microbenchmark cases): tiny decode, Llama-3.2-1B-shaped
# decode, varlen causal prefill 16 x 512, extend with a partial prefix hit at
# page size 16 and 1, the store of the 16 x 512 batch, a smaller mixed batch
# in one launch, and the FP8 variants.
CONFIG_CASES = {
    "tiny_decode": ["tiny_decode"],
    "llama32_1b_decode": ["llama32_1b_decode", "llama32_1b_decode_fp8"],
    "varlen_prefill_16x512": ["varlen_prefill_16x512", "varlen_prefill_16x512_fp8", "store_16x512",
                              "rope_store_16x512"],
    "extend_partial_hit": ["extend_partial_hit_p16", "extend_partial_hit_p1", "extend_partial_hit_p16_fp8",
                           "extend_partial_hit_p1_fp8", "extend_partial_hit_p16_mask50"],
    "decode_64seq_logu": ["decode_64seq_logu", "decode_64seq_logu_fp8"],
    "mixed_64seq_logu": ["mixed_64seq_logu", "mixed_64seq_logu_fp8"],
}


def config_block(dev, peaks, args):
    """Median / p95 time, rate and fraction of the measured peak of every
    case in CONFIG_CASES (prefill also against its attainable roofline
    max(FLOP / peak, bytes / HBM))."""
    import torch
    out = {}
    for cfg, cases in CONFIG_CASES.items():
        out[cfg] = {}
        for name in cases:
            r = time_case(name, dev, args.config_steps, 5)
            if r["unit"] == "TFLOP/s":
                r["frac_bf16"] = round(r["rate"] / peaks["bf16_tflops"], 4)
                t_att = max(r["work"] / (peaks["bf16_tflops"] * 1e12), r["bytes"] / (peaks["hbm_gbs"] * 1e9))
                r["attainable_us"] = round(t_att * 1e6, 2)
                r["frac_attainable"] = round(t_att * 1e6 / r["us_median"], 4)
            else:
                r["frac_hbm"] = round(r["rate"] / peaks["hbm_gbs"], 4)
            out[cfg][name] = r
            torch.cuda.empty_cache()
    return out


def max_over_ranks(value: float, world: int, device=None) -> float:
    """The slowest rank's time: every rank contributes its own measurement and
    all receive the maximum (a plain all-reduce; nothing of the attention
    path is exchanged between ranks)."""
    if world <= 1:
        return float(value)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def run_gpu(args):
    import torch
    import torch.distributed as dist
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    peaks, peak_src = load_peaks()

    mb = MixedBatch(dev)
    mb.prefill_sms = args.prefill_sms
    mb.schedule = args.schedule
    mb.fused_prefill_ctas = args.fused_prefill_ctas
    mb.fused_kv_chunk = args.fused_kv_chunk
    if mb.schedule == "fused":
        mb.launches_per_step = 4     # store, page table, mixed prefill+decode, combine
    elif mb.schedule == "sequential":
        mb.prefill_sms = 0
    torch.cuda.synchronize()

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()

    for _ in range(args.warmup):
        mb.step()
    barrier()
    # ---- timed device steps: the headline (prefill and decode overlapped)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        start.record()
        for _ in range(args.steps):
            mb.step()
        end.record()
        torch.cuda.synchronize()
    barrier()
    total_ms = start.elapsed_time(end)
    # ---- per-step times: events around every step, back to back (median,
    # p95), then the same with L2 flushed before every step (a 512 MiB
    # write, outside the events)
    def per_step(flush=None):
        pairs = []
        for _ in range(args.steps):
            if flush is not None:
                flush.zero_()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            mb.step()
            b.record()
            pairs.append((a, b))
        torch.cuda.synchronize()
        return sorted(a.elapsed_time(b) for a, b in pairs)
    step_ms = per_step()
    flush_buf = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    step_ms_flushed = per_step(flush_buf)
    del flush_buf
    barrier()
    # ---- the same steps with the phases in sequence, for the per-kernel
    # numbers (events recorded between the launches on the same stream)
    phase = {"store_meta": [], "prefill": [], "decode": []}
    evs = []
    for _ in range(args.steps):
        evs.append(mb.step(timing=True))
    torch.cuda.synchronize()
    barrier()
    for e in evs:
        phase["store_meta"].append(e[0].elapsed_time(e[1]))
        phase["prefill"].append(e[1].elapsed_time(e[2]))
        phase["decode"].append(e[2].elapsed_time(e[3]))
    # ---- the attention of the timed step on its own (fused schedule): one
    # pa_mixed_batch per iteration (mixed kernel + combine), events around each
    fused_ms = []
    if mb.schedule == "fused":
        pairs = []
        for _ in range(args.steps):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            mb.fused_pass()
            b.record()
            pairs.append((a, b))
        torch.cuda.synchronize()
        fused_ms = sorted(a.elapsed_time(b) for a, b in pairs)
    barrier()
    ms_step = max_over_ranks(total_ms, world, dev) / args.steps
    from paged_kv_flashattention_gb300 import device_error
    dev_err = device_error()

    # ---- end-to-end through the public API with host buffers
    pin = lambda x: torch.empty(x.shape, dtype=x.dtype, pin_memory=True).copy_(x.cpu())
    h_qd, h_qp, h_k, h_v, h_sm = pin(mb.q_dec), pin(mb.q_pre), pin(mb.k_new), pin(mb.v_new), pin(mb.slot_mapping)
    h_od = torch.empty(mb.out_dec.shape, dtype=mb.out_dec.dtype, pin_memory=True)
    h_op = torch.empty(mb.out_pre.shape, dtype=mb.out_pre.dtype, pin_memory=True)
    h2d = sum(x.numel() * x.element_size() for x in (h_qd, h_qp, h_k, h_v, h_sm))
    d2h = h_od.numel() * h_od.element_size() + h_op.numel() * h_op.element_size()

    # Two sets of device inputs / outputs: while step i runs on the compute
    # stream, the copy stream uploads step i+1's inputs into the other set and
    # downloads step i-1's results, so every step still moves its own bytes
    # but the copies overlap the neighbouring steps' kernels (as a serving
    # loop would).  Events order each set's reuse.
    names_in = ("q_dec", "q_pre", "k_new", "v_new", "slot_mapping")
    names_out = ("out_dec", "out_pre")
    sets = [{n: getattr(mb, n) for n in names_in + names_out},
            {n: torch.empty_like(getattr(mb, n)) for n in names_in + names_out}]
    host_in = dict(zip(names_in, (h_qd, h_qp, h_k, h_v, h_sm)))
    host_out = [(h_od, h_op), (torch.empty_like(h_od).pin_memory(), torch.empty_like(h_op).pin_memory())]
    comp = torch.cuda.current_stream(dev)
    cstream = torch.cuda.Stream(dev)
    ev = lambda: torch.cuda.Event()
    uploaded, computed, downloaded = [ev(), ev()], [ev(), ev()], [ev(), ev()]
    used = [False, False]

    def upload(k):
        with torch.cuda.stream(cstream):
            if used[k]:
                cstream.wait_event(computed[k])            # the last step on set k has read its inputs
            for n in names_in:
                sets[k][n].copy_(host_in[n], non_blocking=True)
            uploaded[k].record(cstream)

    def compute(k):
        comp.wait_event(uploaded[k])
        if used[k]:
            comp.wait_event(downloaded[k])                 # set k's previous results are on the host
        for n in names_in + names_out:
            setattr(mb, n, sets[k][n])
        mb.step()
        computed[k].record(comp)
        used[k] = True

    def download(k):
        with torch.cuda.stream(cstream):
            cstream.wait_event(computed[k])
            host_out[k][0].copy_(sets[k]["out_dec"], non_blocking=True)
            host_out[k][1].copy_(sets[k]["out_pre"], non_blocking=True)
            downloaded[k].record(cstream)

    def e2e_run(n_steps, start=None, end=None):
        if start is not None:
            start.record(comp)
            cstream.wait_event(start)
        upload(0)
        for i in range(n_steps):
            compute(i % 2)
            if i + 1 < n_steps:
                upload((i + 1) % 2)
            download(i % 2)
        if end is not None:
            end.record(cstream)
        comp.wait_stream(cstream)

    e2e_run(max(2, args.warmup // 2))
    barrier()
    s2, e2 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e2e_run(args.steps, s2, e2)
    torch.cuda.synchronize()
    for n in names_in + names_out:                         # back to the first set
        setattr(mb, n, sets[0][n])
    ms_e2e = max_over_ranks(s2.elapsed_time(e2), world, dev) / args.steps
    h2d += mb._keep[0].h2d_bytes + mb._keep[1].h2d_bytes          # the metadata copy of both halves

    dec_ms = statistics.mean(phase["decode"])
    pre_ms = statistics.mean(phase["prefill"])
    dec_gbs = mb.decode_bytes / (dec_ms * 1e-3) / 1e9
    pre_tflops = mb.prefill_flops / (pre_ms * 1e-3) / 1e12
    value = world * mb.step_bytes / (ms_step * 1e-3) / 1e9

    line = {
        "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": WORKLOAD, "l2": "inputs larger than L2 (decode reads "
                   f"{mb.decode_bytes / 1e9:.2f} GB per step; no flush)",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "step": "store_kv + metadata of both halves (one copy, one page-table launch) + prefill "
                           "+ decode (split + combine)",
                   "schedule": schedule_text(mb),
                   "step_bytes": mb.step_bytes},
        "roofline": roofline_block(mb, fused_ms, dec_gbs, peaks, peak_src),
        "decode": {"ms": round(dec_ms, 4), "gbs": round(dec_gbs, 1),
                   "frac_hbm": round(dec_gbs / peaks["hbm_gbs"], 4),
                   "frac_hbm_spec_8tbs": round(dec_gbs / 8000.0, 4),
                   "seqs_per_s": round(mb.dec.num_seqs / (dec_ms * 1e-3), 1)},
        "prefill": {"ms": round(pre_ms, 4), "tflops": round(pre_tflops, 1),
                    "frac_bf16": round(pre_tflops / peaks["bf16_tflops"], 4),
                    "frac_bf16_sustained": round(pre_tflops / peaks["bf16_tflops_sustained"], 4),
                    "frac_bf16_spec_2250": round(pre_tflops / 2250.0, 4),
                    "tokens_per_s": round(mb.pre.num_new_tokens / (pre_ms * 1e-3), 1)},
        "store_meta_ms": round(statistics.mean(phase["store_meta"]), 4),
        "e2e": {"value": round(world * mb.step_bytes / (ms_e2e * 1e-3) / 1e9, 1), "unit": "GB/s",
                "ms_per_step": round(ms_e2e, 4), "h2d_bytes_per_step": int(h2d),
                "d2h_bytes_per_step": int(d2h)},
        "step_ms": {"median": round(_pct(step_ms, 50), 4), "p95": round(_pct(step_ms, 95), 4),
                    "note": "events around every step, back to back"},
        "l2_flushed": {"ms_median": round(_pct(step_ms_flushed, 50), 4),
                       "ms_p95": round(_pct(step_ms_flushed, 95), 4),
                       "value": round(world * mb.step_bytes / (_pct(step_ms_flushed, 50) * 1e-3) / 1e9, 1),
                       "unit": "GB/s", "flush": "512 MiB device write before every step, outside the events"},
        "gpu_launches": mb.launches_per_step * args.steps,
        "clocks": clk.summary(),
        "device_error": dev_err,
    }
    if rank == 0:
        line["schedules"] = schedule_compare(mb, args.steps)
        line["device_error"] |= device_error()
    if rank == 0 and not args.no_configs:
        line["configs"] = config_block(dev, peaks, args)
        line["device_error"] |= device_error()
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(mb, args.cpu_seconds)
        if "configs" in line:
            for cfg, r in config_cpu_baselines(args.config_cpu_seconds).items():
                line["configs"][cfg]["cpu_baseline"] = r
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()


# --------------------------------------------------------------------------
def oracle_decode_sample(dec: W.Problem, seqs, fetch_pages, q_rows):
    """Run the oracle on decode sequences `seqs` of the mixed batch.  The
    pages those sequences use are packed into a compact host pool (the
    oracle's result does not depend on physical placement) and the K/V rows
    of the new tokens are already in them.  Returns (seconds, bytes)."""
    import oracle
    pages = sorted(set(p for b in seqs for p in dec.meta["page_lists"][b]))
    remap = {p: i for i, p in enumerate(pages)}
    kc, vc = fetch_pages(pages)
    L = dec.device_len[seqs].astype(np.int64)
    width = max(1, int(max(len(dec.meta["page_lists"][b]) for b in seqs)))
    pt = np.zeros((len(seqs), width), np.int32)
    for i, b in enumerate(seqs):
        pl = [remap[p] for p in dec.meta["page_lists"][b]]
        pt[i, :len(pl)] = pl
    t0 = time.perf_counter()
    oracle.decode(q_rows, kc, vc, pt, L, num_q_heads=dec.num_q_heads, num_kv_heads=dec.num_kv_heads,
                  head_dim=dec.head_dim, page_size=dec.page_size, scale=dec.scale)
    dt = time.perf_counter() - t0
    return dt, int(L.sum()) * dec.num_kv_heads * dec.head_dim * 2 * 2


def decode_sample(dec: W.Problem, cap_bytes: float = 2e9):
    """The fixed sample of the mixed batch's decode sequences that both CPU
    timings use (the cpu_baseline leg and the reference arm): a seeded
    permutation of the 256 sequences, taken in order until about cap_bytes
    of K/V."""
    order = np.random.default_rng(5).permutation(dec.num_seqs)
    seqs, acc = [], 0
    for b in order:
        nb = int(dec.device_len[b]) * dec.num_kv_heads * dec.head_dim * 4
        if seqs and acc + nb > cap_bytes:
            break
        seqs.append(int(b))
        acc += nb
    return seqs


def cpu_baseline(mb: MixedBatch, target_s: float):
    """The fp64 oracle on the host cores, on a bounded sample of the decode
    batch (the step's dominant work), in the same unit (GB/s of K/V)."""
    import oracle
    torch = mb.torch
    dec = mb.dec

    def fetch(pages):
        idx = torch.tensor(pages, dtype=torch.long, device=mb.dev)
        k = mb.k_cache.index_select(0, idx).view(torch.int16).cpu().numpy().view(np.uint16)
        v = mb.v_cache.index_select(0, idx).view(torch.int16).cpu().numpy().view(np.uint16)
        return k, v

    qh = mb.q_dec.view(torch.int16).cpu().numpy().view(np.uint16)
    # the sample (~2 GB of K/V), run repeatedly until about target_s seconds
    # of oracle time have been spent
    seqs = decode_sample(dec)
    total_t, total_b, reps = 0.0, 0, 0
    while total_t < target_s and reps < 100:
        dt, by = oracle_decode_sample(dec, seqs, fetch, qh[seqs])
        total_t += dt
        total_b += by
        reps += 1
    return {"value": round(total_b / total_t / 1e9, 4), "unit": "GB/s", "cores": oracle.num_threads(),
            "kind": "oracle",
            "sample": f"fp64 oracle decode of {len(seqs)} of the 256 decode sequences "
                      f"({total_b / reps / 1e9:.2f} GB of K/V) x {reps} repetitions, {total_t:.1f} s"}


# The oracle on the other workloads, each in the unit of its GPU case: the
# config name, the config number and the case it stands beside.
CONFIG_CPU_CASES = {"tiny_decode": 1, "llama32_1b_decode": 2, "varlen_prefill_16x512": 3,
                    "extend_partial_hit": 4}


def oracle_config_rate(p: W.Problem, budget_s: float, threads: int | None = None):
    """The fp64 oracle on host workload p (its new K/V stored first): whole
    requests in a seeded order, one oracle call each (the oracle computes
    only the requested rows), cycling through them until about budget_s
    seconds are spent (at least one request).  Decode workloads are rated in
    GB/s of the K/V the sampled sequences read, prefill workloads in TFLOP/s
    of 4 d Hq per visible (query, key) pair; both also in query tokens per
    second."""
    import oracle
    row = p.num_kv_heads * p.head_dim
    kc, vc = p.k_cache.copy(), p.v_cache.copy()
    oracle.store_kv(p.k_new.reshape(-1, row), p.v_new.reshape(-1, row), p.slot_mapping,
                    kc.reshape(-1, row), vc.reshape(-1, row))
    cu_q, cu_k, _, mq, mk = oracle.seqlens(p.cached_len, p.extend_len)
    pt = oracle.page_table_from_token_table(p.token_table, p.table_idx, max(mk, 1), p.page_size)
    decode = bool(np.all(p.extend_len == 1))
    saved = oracle.num_threads()
    if threads is not None:
        oracle.set_threads(threads)
    try:
        spent, tokens, work, calls = 0.0, 0, 0, 0
        order = [int(b) for b in np.random.default_rng(11).permutation(p.num_seqs) if cu_q[b + 1] > cu_q[b]]
        seen = set()
        for n in range(1000 * len(order)):
            b = order[n % len(order)]
            q0, q1 = int(cu_q[b]), int(cu_q[b + 1])
            Lk = int(cu_k[b + 1] - cu_k[b])
            tok = np.arange(q0, q1, dtype=np.int64)
            rows = np.stack([np.repeat(tok, p.num_q_heads),
                             np.tile(np.arange(p.num_q_heads, dtype=np.int64), q1 - q0)], axis=1)
            t0 = time.perf_counter()
            oracle.attention(p.q, kc, vc, pt, cu_q, cu_k, num_q_heads=p.num_q_heads,
                             num_kv_heads=p.num_kv_heads, head_dim=p.head_dim, page_size=p.page_size,
                             causal=p.causal, scale=p.scale, rows=rows)
            spent += time.perf_counter() - t0
            tokens += q1 - q0
            calls += 1
            seen.add(b)
            if decode:
                work += Lk * row * 2 * 2
            else:                    # visible pairs of the end-aligned causal rows
                off = Lk - (q1 - q0)
                work += 4 * p.head_dim * p.num_q_heads * sum(min(Lk, off + i + 1) for i in range(q1 - q0))
            if spent >= budget_s:
                break
        cores = oracle.num_threads()
    finally:
        oracle.set_threads(saved)
    value = work / spent / (1e9 if decode else 1e12)
    return {"value": round(value, 4), "unit": "GB/s" if decode else "TFLOP/s",
            "tokens_per_s": round(tokens / spent, 1), "cores": cores, "kind": "oracle",
            "sample": f"fp64 oracle on {len(seen)} of {p.num_seqs} requests, {calls} request calls "
                      f"({tokens} query tokens), {spent:.2f} s"}


def config_cpu_baselines(budget_s: float):
    """The oracle on each workload of CONFIG_CPU_CASES with every host
    thread, and with one thread on the two decode workloads."""
    out = {}
    for name, cfg in CONFIG_CPU_CASES.items():
        p = W.config(cfg)
        r = oracle_config_rate(p, budget_s)
        if cfg in (1, 2):
            r["single_thread"] = oracle_config_rate(p, budget_s, threads=1)
        out[name] = r
    return out


def run_reference(args):
    """Reference arm: the fp64 CPU oracle, each step the same decode sample
    as the cpu_baseline leg (rank 0 only)."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import oracle
    cfg = W.config(5, with_data=False)
    dec = cfg["decode"]
    rng = np.random.default_rng(W.SEED_BASE + 60)
    # host pool holding only the sampled sequences' pages (seeded N(0,1) values)
    seqs = decode_sample(dec, args.ref_cap_gb * 1e9)
    pages = sorted(set(p for b in seqs for p in dec.meta["page_lists"][b]))
    shape = (len(pages), dec.page_size, dec.num_kv_heads, dec.head_dim)
    kc, vc = W.normal_bf16(rng, shape), W.normal_bf16(rng, shape)
    q = W.normal_bf16(rng, (len(seqs), dec.num_q_heads, dec.head_dim))

    def fetch(_pages):
        return kc, vc

    for _ in range(args.warmup):
        oracle_decode_sample(dec, seqs, fetch, q)
    times, nbytes = [], 0
    for _ in range(args.steps):
        dt, nbytes = oracle_decode_sample(dec, seqs, fetch, q)
        times.append(dt)
    ms = 1e3 * sum(times) / len(times)
    value = nbytes / (ms * 1e-3) / 1e9
    sample = (f"fp64 oracle decode of {len(seqs)} of the 256 decode sequences, the cpu_baseline sample "
              f"({nbytes / 1e9:.3f} GB of K/V per step)")
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
            "n_gpus": int(os.environ.get("WORLD_SIZE", "1")), "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(ms, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": WORKLOAD, "sample": sample},
            "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": oracle.num_threads(),
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


MICRO_CASES = {
    # name: (config, variant, kernel)
    "tiny_decode": (1, None, "decode"),
    "llama32_1b_decode": (2, None, "decode"),
    "varlen_prefill_16x512": (3, None, "prefill"),
    "extend_partial_hit_p16": (4, None, "prefill"),
    "extend_partial_hit_p1": (4, "p1", "prefill"),
    "store_16x512": (3, None, "store"),
    # fused RoPE + store of the same 8192 tokens (q rotated in place)
    "rope_store_16x512": (3, None, "rope"),
    # a smaller mixed-batch decode: 64 sequences, contexts log-uniform
    # [512, 32768], ~2 GB pool (inputs still far larger than L2)
    "decode_64seq_logu": (None, None, "decode"),
    # the same decode workloads over FP8 (E4M3) pools with per-head scales
    "llama32_1b_decode_fp8": (2, None, "decode"),
    "decode_64seq_logu_fp8": (None, None, "decode"),
    "varlen_prefill_16x512_fp8": (3, None, "prefill"),
    "extend_partial_hit_p16_fp8": (4, None, "prefill"),
    "extend_partial_hit_p1_fp8": (4, "p1", "prefill"),
    # the extend batch under a block-sparse mask keeping half of the 128 x
    # 128 blocks (and every diagonal block): the skipped blocks cost nothing
    "extend_partial_hit_p16_mask50": (4, None, "prefill"),
    # decode_64seq_logu's sequences and two 2048-token prefill chunks over one
    # pool, in one mixed-batch launch (automatic prefill share, 256-key T-ranges)
    "mixed_64seq_logu": (None, None, "mixed"),
    "mixed_64seq_logu_fp8": (None, None, "mixed"),
}


def masked_causal_pairs(p, mask) -> int:
    """(query, key) pairs a causal prefill attends to under a 128 x 128
    block mask: per request and query row, the visible keys of the kept key
    blocks (work accounting for the bench only)."""
    total = 0
    kb = np.arange(mask.shape[2], dtype=np.int64)
    for b in range(p.num_seqs):
        Lq, Lk = int(p.extend_len[b]), int(p.device_len[b])
        if Lq == 0:
            continue
        i = np.arange(Lq, dtype=np.int64)
        last = (Lk - Lq) + i                                   # last visible key of row i
        per_block = np.clip(last[:, None] + 1 - 128 * kb[None, :], 0, 128)
        per_block = np.minimum(per_block, np.clip(Lk - 128 * kb[None, :], 0, 128))
        total += int((per_block * mask[b][i // 128]).sum())
    return total


def micro_problem(name):
    cfg, variant, kernel = MICRO_CASES[name]
    if cfg is not None:
        return W.config(cfg, variant), kernel
    rng = np.random.default_rng(W.SEED_BASE + 70)
    Lk = np.exp(rng.uniform(math.log(512), math.log(32768), size=64)).astype(np.int32)
    cached, ext = Lk - 1, np.ones(64, np.int32)
    if kernel == "mixed":          # then the two prefill chunks, no cached prefix
        cached = np.concatenate([cached, [0, 0]]).astype(np.int32)
        ext = np.concatenate([ext, [2048, 2048]]).astype(np.int32)
    p = W.build(name.replace("_fp8", ""), cached_len=cached, extend_len=ext, num_q_heads=32,
                num_kv_heads=8, head_dim=128, page_size=16, seed=W.SEED_BASE + 71, pool_factor=1.1)
    return p, kernel


def prepare_case(name, dev):
    """Device inputs of one microbenchmark case.  Returns (fn, work, unit,
    extra): fn() launches the kernel(s) once, work is the algorithmic bytes
    or FLOPs of one launch, extra holds derived facts of the case."""
    import torch
    import paged_kv_flashattention_gb300 as pa
    from paged_kv_flashattention_gb300 import metadata
    p, kernel = micro_problem(name)
    fp8 = name.endswith("_fp8")
    to = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.bfloat16)
    q = to(p.q)
    kn, vn = to(p.k_new), to(p.v_new)
    sm = torch.from_numpy(p.slot_mapping).to(dev)
    scales = {}
    if fp8:
        kc8, vc8, ks, vs = W.fp8_pools(p, W.SEED_BASE + 72)
        kc, vc = torch.from_numpy(kc8).to(dev), torch.from_numpy(vc8).to(dev)
        scales = dict(k_scale=torch.from_numpy(ks).to(dev), v_scale=torch.from_numpy(vs).to(dev))
        pa.store_kv_fp8(kn, vn, sm, kc, vc, **scales)
    else:
        kc, vc = to(p.k_cache), to(p.v_cache)
        pa.store_kv(kn, vn, sm, kc, vc)
    m = metadata.prepare(p.cached_len, p.extend_len, torch.from_numpy(p.token_table).to(dev),
                         torch.from_numpy(p.table_idx).to(dev), p.page_size)
    Hkv, D, Hq = p.num_kv_heads, p.head_dim, p.num_q_heads
    out = torch.empty_like(q)
    extra = {"kernel": kernel, "page_size": p.page_size, "kv": "fp8_e4m3" if fp8 else "bf16"}
    if kernel == "decode":
        ws = torch.empty(max(16, pa.decode_workspace_size(q.shape, kc, m.max_seqlen_k)),
                         dtype=torch.uint8, device=dev)
        fn = lambda: pa.decode(q, kc, vc, m.page_table, m.cache_seqlens, m.max_seqlen_k,
                               scale=p.scale, out=out, workspace=ws, **scales)
        work = int(p.device_len.astype(np.int64).sum()) * Hkv * D * 2 * kc.element_size() + 2 * q.numel() * 2
        unit = "GB/s"
        extra["seqs"] = p.num_seqs
    elif kernel == "prefill":
        sched = torch.zeros(2, dtype=torch.int32, device=dev)
        off = p.cached_len.astype(np.int64)
        E = p.extend_len.astype(np.int64)
        work = 4 * D * Hq * int(np.sum(E * off + E * (E + 1) // 2))
        if "_mask" in name:
            mask = W.block_mask(np.random.default_rng(W.SEED_BASE + 73), p.extend_len, p.device_len, 0.5)
            scales["block_mask"] = torch.from_numpy(mask).to(dev)
            work = 4 * D * Hq * masked_causal_pairs(p, mask)
            extra["kept_blocks"] = round(float(mask.mean()), 3)
        fn = lambda: pa.prefill(q, kc, vc, m.page_table, m.cu_seqlens_q, m.cu_seqlens_k,
                                m.max_seqlen_q, m.max_seqlen_k, causal=p.causal, scale=p.scale, out=out,
                                scheduler=sched, **scales)
        unit = "TFLOP/s"
        # bytes a perfect kernel moves: Q read, O written, each request's K/V read once
        extra["bytes"] = 2 * q.numel() * 2 + int(p.device_len.astype(np.int64).sum()) * Hkv * D * 2 * kc.element_size()
        extra["tokens"] = int(E.sum())
    elif kernel == "mixed":
        nd = p.num_seqs - 2
        tt, idx = torch.from_numpy(p.token_table).to(dev), torch.from_numpy(p.table_idx).to(dev)
        md = metadata.prepare(p.cached_len[:nd], p.extend_len[:nd], tt, idx[:nd], p.page_size)
        mp = metadata.prepare(p.cached_len[nd:], p.extend_len[nd:], tt, idx[nd:], p.page_size)
        qd, qp = q[:nd], q[nd:]
        od, op = torch.empty_like(qd), torch.empty_like(qp)
        ws = torch.empty(pa.decode_workspace_size(qd.shape, kc, md.max_seqlen_k, kv_chunk=256),
                         dtype=torch.uint8, device=dev)
        sched = torch.zeros(4, dtype=torch.int32, device=dev)
        fn = lambda: pa.mixed_batch(qp, qd, kc, vc, mp.page_table, mp.cu_seqlens_q, mp.cu_seqlens_k,
                                    mp.max_seqlen_q, mp.max_seqlen_k, md.page_table, md.cache_seqlens,
                                    md.max_seqlen_k, scale=p.scale, out_prefill=op, out_decode=od, workspace=ws,
                                    scheduler=sched, kv_chunk=256, **scales)
        kv_row = Hkv * D * 2 * kc.element_size()
        work = (int(p.device_len[:nd].astype(np.int64).sum()) * kv_row + 2 * qd.numel() * 2 +
                int(p.device_len[nd:].astype(np.int64).sum()) * kv_row + 2 * qp.numel() * 2)
        unit = "GB/s"
        extra["seqs"] = nd
        extra["tokens"] = int(p.extend_len[nd:].sum())
    elif kernel == "rope":
        table = pa.rope_cos_sin_table(int(p.device_len.max()) + 1, D, 10000.0).to(dev)
        pos = torch.from_numpy(np.concatenate([np.arange(c, c + e) for c, e in zip(p.cached_len, p.extend_len)])
                               .astype(np.int32)).to(dev)
        fn = lambda: pa.rope_store_kv(q, kn, vn, pos, table, sm, kc, vc, q_out=q)
        # q read + written, k and v read, two pool rows written
        work = 2 * q.numel() * 2 + 2 * 2 * kn.numel() * 2
        unit = "GB/s"
    else:
        fn = lambda: pa.store_kv(kn, vn, sm, kc, vc)
        work = 2 * 2 * kn.numel() * 2
        unit = "GB/s"
    return fn, work, unit, extra


def time_case(name, dev, steps, warmup):
    """One kernel on one workload, as in a microbenchmark manifest: warm-up,
    then replays of a captured CUDA graph of the call (so host launch gaps do
    not sit between the events), timed in groups of 10 back-to-back replays;
    median and p95 over the groups."""
    import torch
    fn, work, unit, extra = prepare_case(name, dev)
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        fn()
        torch.cuda.synchronize()
        with torch.cuda.graph(graph, stream=side):
            fn()
    torch.cuda.current_stream().wait_stream(side)
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()
    groups = max(1, steps // 10)
    ts = []
    for _ in range(groups):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(10):
            graph.replay()
        b.record()
        ts.append((a, b))
    torch.cuda.synchronize()
    us = sorted(a.elapsed_time(b) * 1e3 / 10 for a, b in ts)
    med = us[len(us) // 2]
    p95 = us[min(len(us) - 1, int(0.95 * len(us)))]
    rate = work / (med * 1e-6) / (1e12 if unit == "TFLOP/s" else 1e9)
    res = {"kernel": extra["kernel"], "us_median": round(med, 2), "us_p95": round(p95, 2), "rate": round(rate, 1),
           "unit": unit, "work": work, "iters": groups * 10}
    for k in ("page_size", "kv", "seqs", "tokens", "bytes", "kept_blocks"):
        if k in extra:
            res[k] = extra[k]
    del graph
    torch.cuda.synchronize()
    return res


def run_micro(args):
    import torch
    dev = torch.device("cuda", 0)
    r = time_case(args.micro, dev, args.steps, args.warmup)
    print(json.dumps({"micro": args.micro, **r, "warmup": args.warmup}), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cpu-seconds", type=float, default=10.0,
                    help="target wall time of the CPU-oracle baseline sample")
    ap.add_argument("--config-cpu-seconds", type=float, default=2.0,
                    help="oracle time per workload of the configs block's CPU baselines")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--prefill-sms", type=int, default=12,
                    help="SMs the prefill gets while decode runs beside it (0 = one after the other)")
    ap.add_argument("--schedule", choices=["overlap", "fused", "sequential"], default="fused",
                    help="how one step runs its prefill and decode halves")
    ap.add_argument("--fused-prefill-ctas", type=int, default=12,
                    help="fused schedule: CTAs that take prefill tiles before decode ranges "
                         "(0 = chosen by the kernel from the work)")
    ap.add_argument("--fused-kv-chunk", type=int, default=256,
                    help="fused schedule: keys per T-range of the decode split layout")
    ap.add_argument("--ref-cap-gb", type=float, default=2.0,
                    help="K/V bytes of the decode sample the reference arm times per step (the "
                         "cpu_baseline leg's sample at the default)")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the per-config block (configs 1-4 and FP8 variants timed one by one)")
    ap.add_argument("--config-steps", type=int, default=100, help="timed launches per config case")
    ap.add_argument("--micro", choices=sorted(MICRO_CASES), default=None,
                    help="time one kernel on one workload instead of the full step")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.micro:
        run_micro(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
