"""Online-softmax block merge and split-KV merge, fp64 (oracle side).

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

Written from "Transformer inference kernels: GEMM·Attention·FlashAttention·
Fusion (3/10)":

* section 12 (online softmax): with running statistics (m, l) over the blocks
  seen so far and a new block's maximum and exponential sum (m_b, l_b),
  m_new = max(m, m_b) and l_new = e^(m - m_new) l + e^(m_b - m_new) l_b; the
  output accumulator is rescaled by the same factors;
* section 16 (split-KV): each split of the key range yields a partial
  (m_s, l_s, O_s); a numerically stable merge combines them.

These are a second algorithm for the same exact result as the two-pass
softmax in ``oracle.c``; the tests use them to pin that path, and the split
merge is also the definition the GPU combine pass is checked against.
"""
from __future__ import annotations

import numpy as np


def online_softmax_row(scores: np.ndarray, values: np.ndarray, boundaries) -> tuple[np.ndarray, float]:
    """One attention row by the block-by-block online softmax.

    scores: float64 [L] (already scaled and masked to the visible keys);
    values: float64 [L, d]; boundaries: increasing block edges from 0 to L.
    Returns (O, lse).  Follows the steps of section 12: per block take its
    maximum m_b and its unnormalised sum l_b and partial output, then fold
    them into the running (m, l, acc) with the two rescale factors.
    """
    L, d = values.shape
    m = -np.inf
    l = 0.0
    acc = np.zeros(d, dtype=np.float64)
    edges = list(boundaries)
    assert edges[0] == 0 and edges[-1] == L
    for a, b in zip(edges[:-1], edges[1:]):
        if b <= a:
            continue
        s_blk = scores[a:b]
        m_b = float(np.max(s_blk))
        p_blk = np.exp(s_blk - m_b)
        l_b = float(np.sum(p_blk))
        o_b = p_blk @ values[a:b]           # unnormalised block output
        m_new = max(m, m_b)
        alpha = np.exp(m - m_new) if m != -np.inf else 0.0
        beta = np.exp(m_b - m_new)
        l = alpha * l + beta * l_b
        acc = alpha * acc + beta * o_b
        m = m_new
    if l == 0.0:
        return np.zeros(d, dtype=np.float64), -np.inf
    return acc / l, m + np.log(l)


def merge_partials(o_parts: np.ndarray, lse_parts: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
    """Merge split-KV partial results (section 16).

    o_parts: [..., S, d] normalised partial outputs O_s (each over its own key
    range); lse_parts: [..., S] with lse_s = m_s + ln l_s (-inf for an empty
    split).  The merged softmax weight of split s is
    e^(lse_s - M) / sum_s' e^(lse_s' - M) with M = max_s lse_s, which is the
    section-12 rescale written for normalised partials.  Returns (O, lse);
    when every split is empty, O = 0 and lse = -inf.
    """
    o_parts = np.asarray(o_parts, dtype=np.float64)
    lse_parts = np.asarray(lse_parts, dtype=np.float64)
    M = np.max(lse_parts, axis=-1, keepdims=True)
    empty = ~np.isfinite(M)
    Msafe = np.where(empty, 0.0, M)
    w = np.where(np.isfinite(lse_parts), np.exp(lse_parts - Msafe), 0.0)
    den = np.sum(w, axis=-1, keepdims=True)
    den_safe = np.where(den > 0, den, 1.0)
    o = np.sum(w[..., None] * o_parts, axis=-2) / den_safe
    o = np.where(empty, 0.0, o)
    lse = np.where(empty[..., 0], -np.inf, Msafe[..., 0] + np.log(den_safe[..., 0]))
    return o, lse
