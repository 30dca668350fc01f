"""CUDA-graph replay of decode for a fixed set of batch sizes.

"Transformer inference kernels (3/10)", section 21: a CUDA graph removes the
launch overhead of a step whose shapes do not change.  "code-series
sgl-project mini-sglang 07", "the graph fixes the shape": decode batches are
padded to the first captured size that holds them, the missing rows are dummy
requests whose KV lies on a page nobody owns, and a replay only refreshes the
values in fixed buffers.  Here a dummy row has an empty KV range
(cache_seqlens = 0), so the kernels read no page for it and write O = 0,
lse = -inf; its page-table row may hold anything.

The decode kernels read the lengths on the device and size their work from
them, so one captured graph serves every length mix up to ``max_seqlen_k``.
Refreshing the inputs is plain copies: the lengths from pinned host memory,
q and the page table device to device (or written in place by the caller, e.g.
``rope_store_kv(q_out=runner.q[:B])`` and ``build_page_table(out=...)``).
"""
from __future__ import annotations

import math

import numpy as np
import torch

from . import api


def bucket_for(buckets, batch: int) -> int:
    """The smallest captured size that holds ``batch`` requests."""
    for b in sorted(buckets):
        if b >= batch:
            return b
    raise ValueError(f"batch of {batch} exceeds the largest captured size {max(buckets)}")


class DecodeGraphRunner:
    """Captured decode graphs over one paged pool for batch sizes ``buckets``.

    Fixed device buffers: ``q`` [max_B, Hq, d] bf16, ``page_table`` [max_B,
    ncols] int32, ``cache_seqlens`` [max_B] int32, ``out`` and ``lse``, and one
    workspace sized for the largest bucket.  ``run(lengths)`` pads to the
    bucket, uploads the lengths and replays; rows past the batch are dummies."""

    def __init__(self, k_cache: torch.Tensor, v_cache: torch.Tensor, *, num_q_heads: int,
                 max_seqlen_k: int, buckets=(1, 2, 4, 8, 16, 32, 64, 128, 256),
                 page_size: int | None = None, scale: float | None = None, kv_chunk: int = 0,
                 k_scale: torch.Tensor | None = None, v_scale: torch.Tensor | None = None,
                 sliding_window: int = 0):
        self.k_cache, self.v_cache = k_cache, v_cache
        self.k_scale, self.v_scale = k_scale, v_scale
        self.device = k_cache.device
        num_pages, P, Hkv, d = api._pool_geometry(k_cache, v_cache, page_size)
        self.page_size, self.head_dim, self.num_q_heads = P, d, int(num_q_heads)
        self.max_seqlen_k = int(max_seqlen_k)
        self.scale = float(1.0 / math.sqrt(d) if scale is None else scale)
        self.kv_chunk = int(kv_chunk)
        self.sliding_window = int(sliding_window)
        self.buckets = tuple(sorted(set(int(b) for b in buckets)))
        max_b = self.buckets[-1]
        ncols = max(1, -(-self.max_seqlen_k // P))
        dev = self.device
        self.q = torch.zeros((max_b, self.num_q_heads, d), dtype=torch.bfloat16, device=dev)
        self.page_table = torch.zeros((max_b, ncols), dtype=torch.int32, device=dev)
        self.cache_seqlens = torch.zeros(max_b, dtype=torch.int32, device=dev)
        self.out = torch.zeros((max_b, self.num_q_heads, d), dtype=torch.bfloat16, device=dev)
        self.lse = torch.zeros((max_b, self.num_q_heads), dtype=torch.float32, device=dev)
        need = api.decode_workspace_size((max_b, self.num_q_heads, d), k_cache, self.max_seqlen_k,
                                         page_size=page_size, kv_chunk=self.kv_chunk)
        self.workspace = torch.empty(max(16, need), dtype=torch.uint8, device=dev)
        self.lengths_host = torch.zeros(max_b, dtype=torch.int32, pin_memory=True)
        self.graphs: dict[int, torch.cuda.CUDAGraph] = {}
        self._uploaded = None

    def _decode(self, b: int):
        api.decode(self.q[:b], self.k_cache, self.v_cache, self.page_table[:b], self.cache_seqlens[:b],
                   self.max_seqlen_k, scale=self.scale, page_size=self.page_size, out=self.out[:b],
                   lse=self.lse[:b], workspace=self.workspace, kv_chunk=self.kv_chunk,
                   k_scale=self.k_scale, v_scale=self.v_scale, sliding_window=self.sliding_window)

    def capture(self) -> None:
        """Capture one graph per bucket (the buffers hold empty requests, so
        the warm-up launches read no page)."""
        self.cache_seqlens.zero_()
        side = torch.cuda.Stream(self.device)
        side.wait_stream(torch.cuda.current_stream(self.device))
        with torch.cuda.stream(side):
            for b in self.buckets:
                self._decode(b)                       # warm-up outside the capture
                torch.cuda.synchronize(self.device)
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=side):
                    self._decode(b)
                self.graphs[b] = g
        torch.cuda.current_stream(self.device).wait_stream(side)
        torch.cuda.synchronize(self.device)

    def run(self, lengths, q: torch.Tensor | None = None, page_table: torch.Tensor | None = None):
        """Decode ``len(lengths)`` requests: pad to the bucket, upload the
        lengths (zeros for the dummies), copy q / page-table rows when given
        (else they are expected in ``self.q`` / ``self.page_table``), replay.
        Returns (out[:B], lse[:B]) views of the fixed buffers."""
        lengths = np.asarray(lengths, dtype=np.int32)
        batch = int(lengths.shape[0])
        b = bucket_for(self.buckets, batch)
        if lengths.size and (lengths.min() < 0 or lengths.max() > self.max_seqlen_k):
            raise ValueError("lengths must lie in [0, max_seqlen_k]")
        stream = torch.cuda.current_stream(self.device)
        if self._uploaded is not None:
            self._uploaded.synchronize()              # the pinned buffer is about to be rewritten
        h = self.lengths_host.numpy()
        h[:batch] = lengths
        h[batch:b] = 0
        self.cache_seqlens[:b].copy_(self.lengths_host[:b], non_blocking=True)
        self._uploaded = torch.cuda.Event()
        self._uploaded.record(stream)
        if q is not None:
            self.q[:batch].copy_(q)
        if page_table is not None:
            self.page_table[:batch, :page_table.shape[1]].copy_(page_table)
        self.graphs[b].replay()
        return self.out[:batch], self.lse[:batch]
