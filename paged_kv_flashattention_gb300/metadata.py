"""Batch metadata preparation: the scheduler's per-request lengths become the
kernel arguments ("code-series sgl-project mini-sglang 07", "from ledger to
tensors").

The host part (cu_seqlens_q / cu_seqlens_k / cache_seqlens and the maxima)
is computed by ``pa_build_seqlens`` into pinned host buffers and copied to the
device with non-blocking copies; the page table is sliced out of the
device-resident token-granular global table by the ``pa_build_page_table``
kernel.  Nothing here waits on the GPU.
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
    page_table: torch.Tensor       # int32 [B, ceil(max_seqlen_k / page_size)] (device)
    host: dict                     # pinned host copies (keep alive until the copies ran)

    @property
    def h2d_bytes(self) -> int:
        return sum(int(t.numel() * t.element_size()) for t in self.host.values())


def prepare(cached_len, extend_len, token_table: torch.Tensor, table_idx: torch.Tensor,
            page_size: int, *, pin: bool = True, page_table_out: torch.Tensor | None = None
            ) -> BatchMetadata:
    """Build the kernel arguments of one batch.

    cached_len / extend_len: host int arrays (one entry per request);
    token_table: device int32 [rows, max_len] global table (slot per position);
    table_idx: device int32 [B] row of each request.
    """
    cu_q, cu_k, cs, mq, mk = api.build_seqlens(cached_len, extend_len)
    dev = token_table.device
    host = {}
    devs = {}
    for name, arr in (("cu_seqlens_q", cu_q), ("cu_seqlens_k", cu_k), ("cache_seqlens", cs)):
        h = torch.from_numpy(np.ascontiguousarray(arr))
        if pin:
            h = h.pin_memory()
        host[name] = h
        devs[name] = h.to(dev, non_blocking=pin)
    pt = api.build_page_table(token_table, table_idx, max(mk, 1), page_size, out=page_table_out)
    return BatchMetadata(num_seqs=len(cs), max_seqlen_q=mq, max_seqlen_k=mk, page_size=page_size,
                         cu_seqlens_q=devs["cu_seqlens_q"], cu_seqlens_k=devs["cu_seqlens_k"],
                         cache_seqlens=devs["cache_seqlens"], page_table=pt, host=host)
