"""Seeded synthetic inputs for the paged-KV attention path.

This module is shared by the tests, the smoke check and the benchmark.  It
holds none of the attention arithmetic: it only draws request lengths, hands
out physical pages the way a paged KV allocator does (a seeded permutation of
the pool), and draws bf16 N(0, 1) values.  Both the CUDA path and the oracle
consume what it returns; neither is imported here.

Shapes follow the workloads of "Transformer inference kernels: GEMM·
Attention·FlashAttention·Fusion (3/10)" (32 q heads on 8 KV heads, head_dim
128, page size 16, decode contexts up to tens of thousands of tokens, prompt
blocks of 16 x 512 = 8192 tokens) and the three per-request lengths of
"code-series sgl-project mini-sglang 07" (cached_len, extend_len,
device_len = cached_len + extend_len).

Conventions
-----------
* bf16 tensors are numpy ``uint16`` bit patterns on the host.
* The KV pool is [num_pages, page_size, Hkv, d] for K and for V.  The last
  page of every pool is a POISON page filled with bf16 NaN; every unused
  page-table entry and the padding of the token table point at it, so a
  kernel that reads an entry it should not shows NaN in its output instead of
  touching memory outside the pool.
* Slots past a request's last key inside its last page were never written by
  the store (a serving engine's pool holds whatever was there before): they
  are filled with NaN too (``tail_slots``), so a kernel that lets any value
  of an unwritten slot reach an output fails the parity tests.
* ``token_table`` is the allocator's record at token granularity (one slot per
  position, slot = page * page_size + offset), one row per request
  (``table_idx = arange(B)``).  ``slot_mapping`` lists the slots of the new
  tokens (positions cached_len .. device_len-1), in request order.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

SEED_BASE = 20261202
BF16_NAN = np.uint16(0x7FC0)

CONFIG_NAMES = {
    1: "tiny_decode",
    2: "llama32_1b_decode",
    3: "varlen_prefill_16x512",
    4: "extend_partial_hit",
    5: "mixed_batch_llama3_8b",
}


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bf16 (nearest, ties to even); returns uint16 bits."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    rounding = ((u >> 16) & 1) + np.uint32(0x7FFF)
    return ((u + rounding) >> 16).astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Exact float32 values of bf16 bit patterns."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def normal_bf16(rng: np.random.Generator, shape) -> np.ndarray:
    """bf16 bits of N(0, 1) float32 draws, in chunks to bound memory."""
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.uint16)
    chunk = 1 << 24
    for s in range(0, n, chunk):
        e = min(n, s + chunk)
        out[s:e] = f32_to_bf16_bits(rng.standard_normal(e - s, dtype=np.float32))
    return out.reshape(shape)


E4M3_NAN = np.uint8(0x7F)


def e4m3_codes(rng: np.random.Generator, shape, exp_lo: int = 4, exp_hi: int = 9) -> np.ndarray:
    """Random E4M3 codes (uint8) for an FP8 pool: random sign, exponent field
    uniform in [exp_lo, exp_hi] (magnitudes 2^(e-7) .. 1.875 * 2^(e-7)), random
    mantissa; never a NaN code.  The default spans 0.125 .. 7.5, the spread
    of quantised N(0, 1)-like data."""
    sign = (rng.integers(0, 2, size=shape, dtype=np.uint8) << 7).astype(np.uint8)
    e = (rng.integers(exp_lo, exp_hi + 1, size=shape, dtype=np.uint8) << 3).astype(np.uint8)
    m = rng.integers(0, 8, size=shape, dtype=np.uint8)
    return (sign | e | m).astype(np.uint8)


def fp8_pools(p: "Problem", seed: int, scale_lo: float = 0.1, scale_hi: float = 0.5):
    """FP8 stand-ins for a Problem's pools: (k_codes, v_codes, k_scale,
    v_scale) with the pool's shape, the last (poison) page holding NaN codes,
    and one float32 scale per KV head drawn from U[scale_lo, scale_hi]."""
    rng = np.random.default_rng(seed)
    kc = e4m3_codes(rng, p.k_cache.shape)
    vc = e4m3_codes(rng, p.v_cache.shape)
    kc[p.num_pages - 1] = E4M3_NAN
    vc[p.num_pages - 1] = E4M3_NAN
    poison_tails(p, kc, vc, E4M3_NAN)
    ks = rng.uniform(scale_lo, scale_hi, size=p.num_kv_heads).astype(np.float32)
    vs = rng.uniform(scale_lo, scale_hi, size=p.num_kv_heads).astype(np.float32)
    return kc, vc, ks, vs


def tail_slots(page_lists, device_len, token_table, page_size: int) -> np.ndarray:
    """Flat slot indices (page * page_size + offset) of the slots of used
    pages that no request reads: the unwritten tail of each request's last
    page.  A slot that some request reads (shared prefix pages) is excluded."""
    used = sorted(set(int(p) for pl in page_lists for p in pl))
    if not used or page_size == 1:
        return np.zeros(0, np.int64)
    every = (np.asarray(used, np.int64)[:, None] * page_size + np.arange(page_size)).ravel()
    read = [token_table[b, :int(L)].astype(np.int64) for b, L in enumerate(device_len) if int(L) > 0]
    read = np.concatenate(read) if read else np.zeros(0, np.int64)
    return np.setdiff1d(every, read)


def poison_tails(p: "Problem", k_pool: np.ndarray, v_pool: np.ndarray, value) -> None:
    """Write `value` (NaN bits) into every unwritten tail slot of p's pools
    (shape [num_pages, page_size, Hkv, d], modified in place)."""
    s = tail_slots(p.meta["page_lists"], p.device_len, p.token_table, p.page_size)
    if s.size:
        k_pool.reshape(p.num_pages * p.page_size, -1)[s] = value
        v_pool.reshape(p.num_pages * p.page_size, -1)[s] = value


@dataclass
class Problem:
    """One batch of requests over one paged KV pool.

    Lengths are per request; device_len = cached_len + extend_len.  For a
    decode batch extend_len is 1 everywhere and the new token is the last
    position.  Data arrays are None when generated without host data.
    """
    name: str
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    page_size: int
    num_pages: int            # including the poison page (the last one)
    causal: bool
    scale: float
    cached_len: np.ndarray    # int32 [B]
    extend_len: np.ndarray    # int32 [B]
    token_table: np.ndarray   # int32 [B, max(1, max device_len)]
    table_idx: np.ndarray     # int32 [B]
    slot_mapping: np.ndarray  # int32 [sum extend_len]
    seed: int
    q: np.ndarray | None = None        # uint16 [sum extend_len, Hq, d]
    k_new: np.ndarray | None = None    # uint16 [sum extend_len, Hkv, d]
    v_new: np.ndarray | None = None
    k_cache: np.ndarray | None = None  # uint16 [num_pages, P, Hkv, d]
    v_cache: np.ndarray | None = None
    meta: dict = field(default_factory=dict)

    @property
    def num_seqs(self) -> int:
        return int(self.cached_len.shape[0])

    @property
    def device_len(self) -> np.ndarray:
        return (self.cached_len.astype(np.int64) + self.extend_len).astype(np.int32)

    @property
    def poison_page(self) -> int:
        return self.num_pages - 1

    @property
    def num_new_tokens(self) -> int:
        return int(self.extend_len.sum())

    @property
    def is_decode(self) -> bool:
        return bool(np.all(self.extend_len == 1))

    def row_elems(self) -> int:
        return self.num_kv_heads * self.head_dim


def allocate(rng: np.random.Generator, device_len: np.ndarray, page_size: int,
             num_pages: int, *, shared_prefix_pages: dict | None = None):
    """Hand out physical pages like a paged allocator: a seeded permutation of
    the pool (minus the poison page) consumed in request order.

    shared_prefix_pages maps request b -> (donor request a, n): request b's
    first n pages are request a's first n pages (prefix sharing).
    Returns the token table (poison-padded) and per-request page lists.
    """
    B = device_len.shape[0]
    poison = num_pages - 1
    pages_needed = [(-(-int(L) // page_size)) for L in device_len]
    perm = rng.permutation(poison).astype(np.int64)
    cursor = 0
    page_lists = []
    for b in range(B):
        own = []
        if shared_prefix_pages and b in shared_prefix_pages:
            a, n = shared_prefix_pages[b]
            own = list(page_lists[a][:n])
        fresh = pages_needed[b] - len(own)
        if cursor + fresh > perm.shape[0]:
            raise ValueError("KV pool too small for the requested lengths")
        own += [int(p) for p in perm[cursor:cursor + fresh]]
        cursor += fresh
        page_lists.append(own)
    width = max(1, int(device_len.max()) if B else 1)
    token_table = np.full((B, width), poison * page_size, dtype=np.int64)
    for b in range(B):
        L = int(device_len[b])
        if L == 0:
            continue
        pos = np.arange(L, dtype=np.int64)
        pg = np.asarray(page_lists[b], dtype=np.int64)[pos // page_size]
        token_table[b, :L] = pg * page_size + pos % page_size
    return token_table.astype(np.int32), page_lists


def build(name: str, *, cached_len, extend_len, num_q_heads: int, num_kv_heads: int,
          head_dim: int, page_size: int, seed: int, num_pages: int | None = None,
          pool_factor: float = 1.25, causal: bool = True, scale: float | None = None,
          with_data: bool = True, shared_prefix_pages: dict | None = None) -> Problem:
    """Generate one Problem.  ``num_pages`` includes the poison page; by
    default the pool holds the pages needed times ``pool_factor`` plus it."""
    rng = np.random.default_rng(seed)
    cached = np.asarray(cached_len, dtype=np.int32).reshape(-1)
    extend = np.asarray(extend_len, dtype=np.int32).reshape(-1)
    assert cached.shape == extend.shape
    device_len = cached.astype(np.int64) + extend
    needed = int(sum(-(-int(L) // page_size) for L in device_len))
    if num_pages is None:
        num_pages = max(2, int(math.ceil(needed * pool_factor)) + 1)
    token_table, page_lists = allocate(rng, device_len, page_size, num_pages,
                                       shared_prefix_pages=shared_prefix_pages)
    slots = [token_table[b, int(cached[b]):int(device_len[b])] for b in range(cached.shape[0])]
    slot_mapping = (np.concatenate(slots) if slots else np.zeros(0, np.int32)).astype(np.int32)
    if scale is None:
        scale = 1.0 / math.sqrt(head_dim)
    p = Problem(name=name, num_q_heads=num_q_heads, num_kv_heads=num_kv_heads,
                head_dim=head_dim, page_size=page_size, num_pages=int(num_pages),
                causal=causal, scale=float(scale), cached_len=cached, extend_len=extend,
                token_table=token_table, table_idx=np.arange(cached.shape[0], dtype=np.int32),
                slot_mapping=slot_mapping, seed=int(seed))
    p.meta["page_lists"] = page_lists
    if with_data:
        T = int(extend.sum())
        p.q = normal_bf16(rng, (T, num_q_heads, head_dim))
        p.k_new = normal_bf16(rng, (T, num_kv_heads, head_dim))
        p.v_new = normal_bf16(rng, (T, num_kv_heads, head_dim))
        shape = (num_pages, page_size, num_kv_heads, head_dim)
        p.k_cache = normal_bf16(rng, shape)
        p.v_cache = normal_bf16(rng, shape)
        p.k_cache[num_pages - 1] = BF16_NAN
        p.v_cache[num_pages - 1] = BF16_NAN
        poison_tails(p, p.k_cache, p.v_cache, BF16_NAN)
    return p


def config(cfg: int, variant: str | None = None, *, with_data: bool = True) -> Problem | dict:
    """The five workloads.  Config 5 returns {"decode": Problem, "prefill":
    Problem} sharing one pool (no host data: its ~40 GB pool is filled on the
    device, see ``fill_pool_device``)."""
    seed = SEED_BASE + cfg
    rng = np.random.default_rng(seed + 1000)
    if cfg == 1:
        Lk = np.array([7, 16, 33, 50], dtype=np.int32)
        return build(CONFIG_NAMES[1], cached_len=Lk - 1, extend_len=np.ones(4, np.int32),
                     num_q_heads=4, num_kv_heads=2, head_dim=64, page_size=16, seed=seed,
                     num_pages=33, causal=True, with_data=with_data)
    if cfg == 2:
        Lk = rng.integers(128, 4096, size=64, endpoint=True).astype(np.int32)
        return build(CONFIG_NAMES[2], cached_len=Lk - 1, extend_len=np.ones(64, np.int32),
                     num_q_heads=32, num_kv_heads=8, head_dim=64, page_size=16, seed=seed,
                     causal=True, with_data=with_data)
    if cfg == 3:
        return build(CONFIG_NAMES[3], cached_len=np.zeros(16, np.int32),
                     extend_len=np.full(16, 512, np.int32), num_q_heads=32, num_kv_heads=8,
                     head_dim=128, page_size=16, seed=seed, causal=True, with_data=with_data)
    if cfg == 4:
        cached = rng.integers(0, 4096, size=8, endpoint=True).astype(np.int32)
        extend = rng.integers(64, 1024, size=8, endpoint=True).astype(np.int32)
        page = 1 if variant in ("p1", "p1_shuffled") else 16
        name = CONFIG_NAMES[4] + ("_p1" if page == 1 else "_p16")
        return build(name, cached_len=cached, extend_len=extend, num_q_heads=32,
                     num_kv_heads=8, head_dim=128, page_size=page, seed=seed,
                     causal=True, with_data=with_data)
    if cfg == 5:
        lo, hi = math.log(512), math.log(32768)
        Lk = np.exp(rng.uniform(lo, hi, size=256)).astype(np.int64).clip(512, 32768).astype(np.int32)
        # ~40 GB of K+V: 610,352 pages of 16 x 8 x 128 bf16 (32 KiB) per cache
        num_pages = 610352
        dec = build(CONFIG_NAMES[5] + "_decode", cached_len=Lk - 1,
                    extend_len=np.ones(256, np.int32), num_q_heads=32, num_kv_heads=8,
                    head_dim=128, page_size=16, seed=seed, num_pages=num_pages,
                    causal=True, with_data=False)
        # the two prefill chunks take pages the decode batch did not use
        used = set(p for pl in dec.meta["page_lists"] for p in pl)
        free = np.array([p for p in np.random.default_rng(seed + 7).permutation(num_pages - 1)[:400000]
                         if p not in used][:2 * 2048 // 16], dtype=np.int64)
        pre = build(CONFIG_NAMES[5] + "_prefill", cached_len=np.zeros(2, np.int32),
                    extend_len=np.full(2, 2048, np.int32), num_q_heads=32, num_kv_heads=8,
                    head_dim=128, page_size=16, seed=seed + 1, num_pages=num_pages,
                    causal=True, with_data=False)
        pos = np.arange(2048, dtype=np.int64)
        for b in range(2):
            pg = free[b * 128:(b + 1) * 128][pos // 16]
            pre.token_table[b, :2048] = (pg * 16 + pos % 16).astype(np.int32)
            pre.meta["page_lists"][b] = [int(x) for x in free[b * 128:(b + 1) * 128]]
        pre.slot_mapping = np.concatenate([pre.token_table[b, :2048] for b in range(2)]).astype(np.int32)
        return {"decode": dec, "prefill": pre}
    raise ValueError(f"unknown config {cfg}")


def add_host_data(p: Problem, rng_seed: int | None = None) -> Problem:
    """Draw q / new K,V / pool values for a Problem made with with_data=False."""
    rng = np.random.default_rng(p.seed if rng_seed is None else rng_seed)
    T = p.num_new_tokens
    p.q = normal_bf16(rng, (T, p.num_q_heads, p.head_dim))
    p.k_new = normal_bf16(rng, (T, p.num_kv_heads, p.head_dim))
    p.v_new = normal_bf16(rng, (T, p.num_kv_heads, p.head_dim))
    shape = (p.num_pages, p.page_size, p.num_kv_heads, p.head_dim)
    p.k_cache = normal_bf16(rng, shape)
    p.v_cache = normal_bf16(rng, shape)
    p.k_cache[-1] = BF16_NAN
    p.v_cache[-1] = BF16_NAN
    poison_tails(p, p.k_cache, p.v_cache, BF16_NAN)
    return p


MASK_BLOCK = 128


def block_mask(rng: np.random.Generator, extend_len, device_len, density: float = 0.6,
               keep_diagonal: bool = True) -> np.ndarray:
    """A random block-sparse mask for a batch: uint8 [B, nq, nk] over blocks of
    128 query rows (of each request's own rows) x 128 keys, each block kept
    with probability ``density``; with ``keep_diagonal`` the block holding a
    query block's own positions at the end of its keys is always kept (the
    usual shape of a sparse causal pattern).  Blocks outside a request's
    lengths are set too (never read)."""
    ext = np.asarray(extend_len, np.int64)
    dev = np.asarray(device_len, np.int64)
    B = ext.shape[0]
    nq = max(1, int(-(-ext.max() // MASK_BLOCK)) if B else 1)
    nk = max(1, int(-(-dev.max() // MASK_BLOCK)) if B else 1)
    m = (rng.random((B, nq, nk)) < density).astype(np.uint8)
    if keep_diagonal:
        for b in range(B):
            off = int(dev[b] - ext[b])
            for qb in range(nq):
                last = off + min(int(ext[b]), (qb + 1) * MASK_BLOCK) - 1    # last row's position
                if last >= 0:
                    m[b, qb, last // MASK_BLOCK] = 1
    return m


def poison_tails_device(p: Problem, k_pool, v_pool) -> int:
    """Device-pool version of ``poison_tails``: write bf16 NaN into p's
    unwritten tail slots of two torch CUDA pools [num_pages, P, Hkv, d].
    Returns the number of slots poisoned."""
    import torch
    s = tail_slots(p.meta["page_lists"], p.device_len, p.token_table, p.page_size)
    if s.size:
        idx = torch.from_numpy(s).to(k_pool.device)
        for t in (k_pool, v_pool):
            t.view(-1, t.shape[-2] * t.shape[-1]).index_fill_(0, idx, float("nan"))
    return int(s.size)


def fill_normal_device(t, seed: int) -> None:
    """Fill a bf16 torch CUDA tensor with seeded N(0, 1) draws (torch's own
    generator; used for pools too large to draw on the host)."""
    import torch
    g = torch.Generator(device=t.device)
    g.manual_seed(int(seed))
    flat = t.view(-1)
    chunk = 1 << 28
    for s in range(0, flat.numel(), chunk):
        e = min(flat.numel(), s + chunk)
        flat[s:e].normal_(0.0, 1.0, generator=g)


def small_problem(seed: int, cached_len, extend_len, *, num_q_heads=4, num_kv_heads=2,
                  head_dim=64, page_size=16, causal=True, pool_factor=1.5,
                  shared_prefix_pages=None, scale=None) -> Problem:
    """Arbitrary small shapes for edge-case tests."""
    return build("custom", cached_len=cached_len, extend_len=extend_len,
                 num_q_heads=num_q_heads, num_kv_heads=num_kv_heads, head_dim=head_dim,
                 page_size=page_size, seed=seed, pool_factor=pool_factor, causal=causal,
                 scale=scale, shared_prefix_pages=shared_prefix_pages)
