"""Batch metadata preparation: the scheduler's per-request lengths become the
kernel arguments ("code-series sgl-project mini-sglang 07", "from ledger to
tensors").

The host part (cu_seqlens_q / cu_seqlens_k / cache_seqlens and the maxima)
is computed by ``pa_build_seqlens`` into pinned host buffers and copied to the
device with non-blocking copies; the page table is sliced out of the
device-resident token-granular global table by the ``pa_build_page_table``
kernel.  Nothing here waits on the GPU except a ``MetadataBuilder`` that is
about to overwrite a pinned staging buffer whose previous copy is still in
flight.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np
import torch

from . import api


@dataclass
class BatchMetadata:
    num_seqs: int
    max_seqlen_q: int
    max_seqlen_k: int
    page_size: int
    cu_seqlens_q: torch.Tensor     # int32 [B+1] (device)
    cu_seqlens_k: torch.Tensor     # int32 [B+1] (device)
    cache_seqlens: torch.Tensor    # int32 [B]   (device)
    page_table: torch.Tensor       # int32 [B, >= ceil(max_seqlen_k / page_size)] (device)
    h2d_bytes: int


class MetadataBuilder:
    """Reusable pinned staging + device buffers for batches of up to
    ``max_seqs`` requests on one device."""

    def __init__(self, device, max_seqs: int):
        self.device = torch.device(device)
        self.max_seqs = int(max_seqs)
        n = self.max_seqs + 1
        # one pinned buffer: [cu_q (n) | cu_k (n) | cache_seqlens (n)]
        self.host = torch.empty(3 * n, dtype=torch.int32, pin_memory=True)
        self.dev = torch.empty(3 * n, dtype=torch.int32, device=self.device)
        self.copied = None   # event recorded after the last H2D from self.host

    def prepare(self, cached_len, extend_len, token_table: torch.Tensor, table_idx: torch.Tensor,
                page_size: int, *, page_table_out: torch.Tensor | None = None) -> BatchMetadata:
        cu_q, cu_k, cs, mq, mk = api.build_seqlens(cached_len, extend_len)
        B = len(cs)
        if B > self.max_seqs:
            raise ValueError(f"batch of {B} requests > builder capacity {self.max_seqs}")
        n = self.max_seqs + 1
        if self.copied is not None:
            self.copied.synchronize()        # the staging buffer is about to be rewritten
        h = self.host.numpy()
        h[0:B + 1] = cu_q
        h[n:n + B + 1] = cu_k
        h[2 * n:2 * n + B] = cs
        stream = torch.cuda.current_stream(self.device)
        self.dev.copy_(self.host, non_blocking=True)
        self.copied = torch.cuda.Event()
        self.copied.record(stream)
        pt = api.build_page_table(token_table, table_idx, max(mk, 1), page_size, out=page_table_out)
        return BatchMetadata(num_seqs=B, max_seqlen_q=mq, max_seqlen_k=mk, page_size=page_size,
                             cu_seqlens_q=self.dev[0:B + 1], cu_seqlens_k=self.dev[n:n + B + 1],
                             cache_seqlens=self.dev[2 * n:2 * n + B], page_table=pt,
                             h2d_bytes=3 * n * 4)


def prepare(cached_len, extend_len, token_table: torch.Tensor, table_idx: torch.Tensor,
            page_size: int, *, page_table_out: torch.Tensor | None = None) -> BatchMetadata:
    """One-off metadata preparation (allocates its own staging buffers)."""
    B = len(np.asarray(cached_len))
    builder = MetadataBuilder(token_table.device, max(B, 1))
    return builder.prepare(cached_len, extend_len, token_table, table_idx, page_size,
                           page_table_out=page_table_out)


class MixedMetadataBuilder:
    """Metadata of a mixed continuous batch for ``mixed_batch`` (prefill /
    extend requests and decode sequences over one pool).

    Both halves' lengths go to the device in ONE copy from one pinned staging
    buffer, and both halves' page-table rows are built by ONE launch (decode
    rows first, then the prefill rows, all ``ceil(max key length / page)``
    wide).  The copy runs on the builder's own stream into one of two device
    buffer sets used in turn, so it overlaps the kernels issued before the
    attention (the KV store, the page table); ``prepare`` makes the current
    stream wait for it before returning, so everything the caller launches
    afterwards sees the lengths.  A set is rewritten only after the work
    issued before the previous ``prepare`` (the attention that read it) is
    done, and its pinned staging buffer only after its last copy finished.
    """

    def __init__(self, device, max_prefill_seqs: int, max_decode_seqs: int):
        self.device = torch.device(device)
        self.np = int(max_prefill_seqs) + 1
        self.nd = int(max_decode_seqs) + 1
        n = 3 * (self.np + self.nd)
        # per set: [pre cu_q | pre cu_k | pre cache_seqlens (np each) | dec cu_q | dec cu_k | dec cache_seqlens]
        self.host = [torch.empty(n, dtype=torch.int32, pin_memory=True) for _ in range(2)]
        self.dev = [torch.empty(n, dtype=torch.int32, device=self.device) for _ in range(2)]
        self.copied = [None, None]       # last copy out of host[k]
        self.issued = None               # the current stream before the previous prepare
        self.copy_stream = torch.cuda.Stream(self.device)
        self.k = 0

    def prepare(self, pre_cached, pre_extend, dec_cached, dec_extend, token_table: torch.Tensor,
                table_idx: torch.Tensor, page_size: int, *, page_table_out: torch.Tensor | None = None):
        """Returns (prefill BatchMetadata, decode BatchMetadata).  table_idx
        holds the decode rows' indices into token_table, then the prefill
        rows'."""
        cq_p, ck_p, cs_p, mq_p, mk_p = api.build_seqlens(pre_cached, pre_extend)
        cq_d, ck_d, cs_d, mq_d, mk_d = api.build_seqlens(dec_cached, dec_extend)
        Bp, Bd = len(cs_p), len(cs_d)
        if Bp + 1 > self.np or Bd + 1 > self.nd:
            raise ValueError("batch larger than the builder's capacity")
        if table_idx.numel() != Bd + Bp:
            raise ValueError("table_idx must hold the decode rows then the prefill rows")
        k, npp, nd = self.k, self.np, self.nd
        self.k ^= 1
        if self.copied[k] is not None:
            self.copied[k].synchronize()         # host[k] is about to be rewritten
        h = self.host[k].numpy()
        h[0:Bp + 1] = cq_p
        h[npp:npp + Bp + 1] = ck_p
        h[2 * npp:2 * npp + Bp] = cs_p
        o = 3 * npp
        h[o:o + Bd + 1] = cq_d
        h[o + nd:o + nd + Bd + 1] = ck_d
        h[o + 2 * nd:o + 2 * nd + Bd] = cs_d
        stream = torch.cuda.current_stream(self.device)
        now = torch.cuda.Event()
        now.record(stream)
        with torch.cuda.stream(self.copy_stream):
            if self.issued is not None:
                # dev[k] was last read by work issued before the previous prepare
                self.copy_stream.wait_event(self.issued)
            self.dev[k].copy_(self.host[k], non_blocking=True)
            done = torch.cuda.Event()
            done.record(self.copy_stream)
        self.copied[k] = done
        self.issued = now
        mk = max(mk_p, mk_d, 1)
        pt = api.build_page_table(token_table, table_idx, mk, page_size, out=page_table_out)
        stream.wait_event(done)
        d = self.dev[k]
        mp = BatchMetadata(num_seqs=Bp, max_seqlen_q=mq_p, max_seqlen_k=mk_p, page_size=page_size,
                           cu_seqlens_q=d[0:Bp + 1], cu_seqlens_k=d[npp:npp + Bp + 1],
                           cache_seqlens=d[2 * npp:2 * npp + Bp], page_table=pt[Bd:], h2d_bytes=3 * npp * 4)
        md = BatchMetadata(num_seqs=Bd, max_seqlen_q=mq_d, max_seqlen_k=mk_d, page_size=page_size,
                           cu_seqlens_q=d[o:o + Bd + 1], cu_seqlens_k=d[o + nd:o + nd + Bd + 1],
                           cache_seqlens=d[o + 2 * nd:o + 2 * nd + Bd], page_table=pt[:Bd], h2d_bytes=3 * nd * 4)
        return mp, md
