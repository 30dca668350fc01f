"""Tiny pure-Python brute force for paged attention (oracle side).

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

A second, deliberately different derivation of scaled dot-product attention
("Transformer inference kernels ... (3/10)", section 10) for inputs of a few
dozen keys: the request's keys and values are first gathered into contiguous
Python lists by walking its page-table row page by page (section 14's logical
block -> physical block mapping, read in the other direction), then the
textbook softmax exp(s_j) / sum_k exp(s_k) is taken without the max shift, and
every sum is an exactly rounded ``math.fsum``.  Only for small, well-scaled
inputs (|s| < 700).
"""
from __future__ import annotations

import math
import struct


def _bf16(bits: int) -> float:
    return struct.unpack("<f", struct.pack("<I", (int(bits) & 0xFFFF) << 16))[0]


def gather_request(cache_rows, page_row, length: int, page_size: int, kv_head: int):
    """Contiguous list of the request's ``length`` rows for one KV head.

    cache_rows(slot, kv_head) -> list of d bf16 bit patterns."""
    out = []
    for logical_page, phys in enumerate(page_row):
        for offset in range(page_size):
            pos = logical_page * page_size + offset
            if pos >= length:
                return out
            out.append([_bf16(x) for x in cache_rows(int(phys) * page_size + offset, kv_head)])
    return out


def attention(q, k_cache, v_cache, page_table, cu_q, cu_k, *, num_q_heads, num_kv_heads,
              head_dim, page_size, causal, scale, window_left=-1, block_mask=None):
    """q: nested [Tq][Hq][d] bf16 bits (or a numpy array); caches indexable as
    cache[slot][kv_head] -> d bits; block_mask: optional [B][nq][nk] bytes over
    blocks of 128 query rows x 128 keys (0 = the keys of that block are not
    attended to).  Returns nested lists O[Tq][Hq][d]."""
    group = num_q_heads // num_kv_heads
    Tq = int(cu_q[-1])
    out = [[[0.0] * head_dim for _ in range(num_q_heads)] for _ in range(Tq)]
    for b in range(len(cu_q) - 1):
        q0, q1 = int(cu_q[b]), int(cu_q[b + 1])
        Lq, Lk = q1 - q0, int(cu_k[b + 1]) - int(cu_k[b])
        for kvh in range(num_kv_heads):
            K = gather_request(lambda s, h: k_cache[s][h], page_table[b], Lk, page_size, kvh)
            V = gather_request(lambda s, h: v_cache[s][h], page_table[b], Lk, page_size, kvh)
            for h in range(kvh * group, (kvh + 1) * group):
                for i in range(Lq):
                    qv = [_bf16(x) for x in q[q0 + i][h]]
                    # absolute position of this query among the request's keys
                    pos = (Lk - Lq) + i
                    keys = [j for j in range(Lk) if ((not causal) or j <= pos)
                            and (window_left < 0 or pos - j <= window_left)
                            and (block_mask is None or block_mask[b][i // 128][j // 128] != 0)]
                    if not keys:
                        continue            # empty: output stays 0
                    e = [math.exp(scale * math.fsum(a * c for a, c in zip(qv, K[j]))) for j in keys]
                    z = math.fsum(e)
                    for c in range(head_dim):
                        out[q0 + i][h][c] = math.fsum(e[n] * V[j][c] for n, j in enumerate(keys)) / z
    return out
