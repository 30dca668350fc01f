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
