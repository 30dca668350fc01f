// Varlen causal prefill / extend attention over a paged KV cache on the
// 5th-generation tensor cores (tcgen05 + TMEM): the device code (shared by
// the prefill kernel and the mixed-batch kernel) and the host-side argument
// setup.
//
// "Transformer inference kernels: GEMM·Attention·FlashAttention·Fusion
// (3/10)": attention is computed tile by tile so the score matrix never
// reaches HBM (section 11), with the online softmax merge of section 12; keys
// are read through the page table (section 14), several query heads share a
// KV head (section 15), and the causal window of a request with a cached
// prefix is aligned to the end of its keys ("code-series sgl-project
// mini-sglang 07": seqlens_q = extend_len, seqlens_k = device_len).
//
// GB300 design (the pages' prior art is Ampere/Hopper; this is not it).
// Persistent: one CTA per SM.  A work item is one 128-row query tile of T
// query heads that share a KV head (T = 2 when the GQA group allows it), so
// every K/V tile feeds 2T MMAs.  Items are ordered last tile first (the k-th
// tile from the end of every request before any (k+1)-th) and handed out by a
// device counter; the producer publishes each item index to the other roles
// through a small ring of mbarriers, and TMEM, barriers and the K/V ring
// carry over from one item to the next.
//   warp 4T (producer): takes the next item, TMA-loads its T Q tiles
//     (64-column halves, 128-byte swizzle, K-major) once the previous item's
//     last score MMA is done, then per 128-key step the K and V tiles:
//     page size 16 -> one 3-D TMA box of 16 tokens per page and half;
//     page size 1  -> cp.async 16-byte pieces of key rows placed in the same
//     swizzled layout, shared round robin with warps 4T+2 and 4T+3.  K and V
//     tiles go to separate slots of one ring (5 slots of 32 KiB for d = 128
//     next to 64 KiB of Q), so loads run several tiles ahead; pages past the
//     visible keys are filled with zeros by out-of-range TMA coordinates.
//   warp 4T+1 (MMA): one thread issues tcgen05.mma.  Order per step j:
//     PV_0(j), S_0(j+1), PV_1(j), S_1(j+1), ...: S_k(j+1) overwrites the TMEM
//     columns that PV_k(j) reads P from, which relies on tcgen05.mma ops of
//     one thread executing in issue order; and because a tcgen05.commit
//     tracks every earlier MMA of the thread, the arrival of S_k(j+1) also
//     tells the softmax that PV_k(j) has finished (O_k may be rescaled).
//   warps 4k..4k+3 (softmax of tile k): thread r owns query row r = TMEM
//     lane r.  It loads its S row with tcgen05.ld, masks only on tiles that
//     reach the causal diagonal or the end of the keys, takes the row maximum
//     with a tree of independent maxima, updates the running maximum lazily
//     (only when the tile maximum exceeds it by more than 8 in log2 units;
//     then O_k in TMEM is rescaled), computes p = 2^(s*scale*log2 e - m) with
//     packed f32x2 FMAs and the MUFU unit, writes P as bf16 over its S
//     columns with tcgen05.st, and at the end normalises O and writes bf16
//     output and the natural-log LSE.
// TMEM (512 columns): S_k at [128k, 128k+128), O_k at [256 + 128k, +d).
//
// FP8 pools (E4M3 codes with a scale per KV head; the first page lists FP8 /
// quantized KV as a dispatch axis, section 19): tcgen05 kind::f16 needs 16-bit
// operands on both sides, so the E4M3 tiles are loaded one byte per element
// without swizzle (at d = 128 into the upper half of the f16 slot they are
// widened into, in place; at d = 64 into a separate landing ring) and the two
// otherwise idle warps of the control warpgroup widen them exactly to f16 in
// the swizzled layout the MMA reads, and turn each item's Q tiles in place
// into f16 q * k_scale.
// The MMAs then run with f16 operands (P is written to TMEM as f16) and the
// epilogue multiplies by v_scale.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>

#include <mutex>

#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {
namespace {

constexpr int kBM = 128;          // query rows per tile
constexpr int kBN = 128;          // keys per step
constexpr float kLazy = 8.0f;

__device__ __forceinline__ float2 add2(float2 a, float2 b) {
    uint64_t ai = *reinterpret_cast<uint64_t *>(&a), bi = *reinterpret_cast<uint64_t *>(&b), r;
    asm("add.f32x2 %0, %1, %2;" : "=l"(r) : "l"(ai), "l"(bi));
    return *reinterpret_cast<float2 *>(&r);
}

__device__ __forceinline__ float max3(float a, float b, float c) {
    float r;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}

struct PrefillArgs {
    CUtensorMap qmap;             // bf16 (d, Hq, total_q), box (64, 1, 128)
    CUtensorMap kmap;             // bf16 (d, Hkv, num_slots), box (64, 1, 16)
    CUtensorMap vmap;
    const uint8_t *k_cache;       // for page size 1 (row gathers)
    const uint8_t *v_cache;
    const int32_t *page_table;
    int64_t pt_stride;
    const int32_t *cu_q;
    const int32_t *cu_k;
    __nv_bfloat16 *out;
    float *lse;
    int64_t lse_stride;
    int32_t num_seqs;
    int32_t total_q;
    int32_t num_q_heads;
    int32_t num_kv_heads;
    int32_t page_size;
    int32_t num_slots;
    int32_t causal;
    float scale_log2;
    int32_t num_virtual;          // max_tiles * num_seqs * (Hq / T) work-item slots
    const float *k_scale;         // FP8 pools: per-KV-head scales
    const float *v_scale;
    int32_t *sched;               // caller's [0] next item, [1] CTAs finished; 0 between launches
    int32_t window;               // sliding window W (0 = none): keys >= position - (W - 1)
    const uint8_t *bmask;         // block-sparse mask [num_seqs][bm_q][bm_k] over 128 x 128 blocks, or null
    int32_t bm_q, bm_k;
    int32_t max_q, max_k;         // the call's max_seqlen_q / max_seqlen_k (bounds of the device lengths)
    int32_t num_ctas;             // CTAs that run the work loop (the last of them resets sched);
                                  // 0: the count passed to prefill_body
};

// One work item: a 128-row query tile of T query heads of one request.
struct PrefillItem {
    int b, tile, h0, kvh, q0, Lk, off, rows_here, kv_end, min_vis;
    int n_all;    // 128-key steps from j0 up to the last key the tile sees
    int n_kv;     // of those, the steps the block mask keeps (all of them without one)
    int j0;       // first 128-key step (a sliding window skips the ones before)
    int lo_max;   // keys below this are outside some row's window: mask there
};

// With a block-sparse mask an item's steps are the kept ones only: every
// role walks them by ordinal 0 .. n_kv - 1 (barrier phases, first and last
// step, load counts) and maps an ordinal to its step with a cursor, which
// advances through the mask row of the item's query block.  Ordinals are
// visited in increasing order.  Without a mask the map is the identity.
struct StepCursor {
    int idx = -1, step = -1;      // the idx-th kept step is `step` (relative to j0)
    template <bool EXT>
    __device__ __forceinline__ int at(const PrefillArgs &a, const PrefillItem &it, int i) {
        if (!EXT || a.bmask == nullptr) return i;
        if (i < idx) idx = step = -1;
        const uint8_t *row = a.bmask + ((int64_t)it.b * a.bm_q + it.tile) * a.bm_k + it.j0;
        while (idx < i) {
            ++step;
            while (row[step] == 0) ++step;   // the i-th kept step exists: i < n_kv
            ++idx;
        }
        return step;
    }
};

// Item v of the virtual list (k-th tile from the end of request b, head group
// hp), k-major: every request's later, longer tiles come before its earlier
// ones, so persistent CTAs taking items round robin start with the longest
// work.  Returns false for a hole (request b has fewer than k + 1 tiles).
template <int T, bool EXT = false>
__device__ __forceinline__ bool prefill_item(const PrefillArgs &a, int v, PrefillItem &it) {
    const int groups = a.num_q_heads / T;
    const int hp = v % groups;
    const int rest = v / groups;
    const int b = rest % a.num_seqs;
    const int k = rest / a.num_seqs;
    const int q0 = a.cu_q[b];
    const int Lq = a.cu_q[b + 1] - q0;
    const int Lk = a.cu_k[b + 1] - a.cu_k[b];
    // device lengths outside the call's bounds: the request is skipped (its
    // rows are not written) rather than read or written out of bounds
    if (q0 < 0 || Lq < 0 || q0 + Lq > a.total_q || Lq > a.max_q || Lk < 0 || Lk > a.max_k ||
        (Lk > 0 && Lq > Lk)) {
        raise_error(PA_DEVERR_SEQLENS);
        return false;
    }
    const int tiles = (Lq + kBM - 1) / kBM;
    if (k >= tiles) return false;
    it.b = b;
    it.tile = tiles - 1 - k;
    it.h0 = hp * T;
    it.kvh = it.h0 / (a.num_q_heads / a.num_kv_heads);
    it.q0 = q0;
    it.Lk = Lk;
    it.off = it.Lk - Lq;                                  // cached prefix length
    it.rows_here = min(kBM, Lq - it.tile * kBM);
    int kv_end = it.Lk;                                   // keys the tile's last row sees
    if (a.causal) kv_end = min(it.Lk, it.off + it.tile * kBM + it.rows_here);
    it.kv_end = kv_end < 0 ? 0 : kv_end;
    it.n_kv = (it.kv_end + kBN - 1) / kBN;
    // keys every row of the tile sees: steps entirely below this need no mask
    const int mv = a.causal ? min(it.Lk, it.off + it.tile * kBM + 1) : it.Lk;
    it.min_vis = mv < 0 ? 0 : mv;
    // sliding window: row i sees keys >= off + i - (W - 1); the first row's
    // bound fixes the first step, the last row's where masking stops
    it.j0 = 0;
    it.lo_max = 0;
    if (EXT && a.window > 0) {
        const int lo_first = it.off + it.tile * kBM - (a.window - 1);
        it.j0 = lo_first > 0 ? lo_first / kBN : 0;
        it.lo_max = lo_first + it.rows_here - 1;
        it.n_kv -= it.j0;
        if (it.n_kv < 0) it.n_kv = 0;
    }
    it.n_all = it.n_kv;
    if (EXT && a.bmask != nullptr) {        // count the steps the block mask keeps
        const uint8_t *row = a.bmask + ((int64_t)b * a.bm_q + it.tile) * a.bm_k + it.j0;
        int kept = 0;
        for (int j = 0; j < it.n_all; ++j) kept += row[j] != 0;
        it.n_kv = kept;
    }
    return true;
}

// Next item for this CTA (producer lane 0), or -1 when none is left.  Items
// are handed out by one counter in the order above, so CTAs that finish early
// take more.  A hole means the whole row (k, b) is a hole, and the rows after
// it often are too (short requests have few tiles): the counter is moved past
// every hole row up to the next row with work before taking another number.
template <int T>
__device__ int prefill_fetch(const PrefillArgs &a) {
    const int groups = a.num_q_heads / T;
    const int rows = a.num_virtual / groups;
    for (;;) {
        const int v = atomicAdd(&a.sched[0], 1);
        if (v >= a.num_virtual) return -1;
        PrefillItem it;
        if (prefill_item<T>(a, v, it)) return v;
        int row = v / groups + 1;
        for (; row < rows; ++row)
            if (prefill_item<T>(a, row * groups, it)) break;
        atomicMax(&a.sched[0], row * groups);
    }
}

// Called once per CTA after its last fetch: the last CTA to finish resets the
// counters (in the caller's scheduler array) for the next launch that uses
// them.
__device__ void prefill_sched_done(const PrefillArgs &a, int num_ctas) {
    __threadfence();
    if (atomicAdd(&a.sched[1], 1) == num_ctas - 1) {
        atomicExch(&a.sched[0], 0);
        atomicExch(&a.sched[1], 0);
    }
}

// Shared memory: T query tiles, then a ring of K-or-V tile slots (as many as
// fit in 227 KiB next to Q and the output staging, at most 8), then 4 KiB of
// output staging per softmax warp, then the barriers.  K_j goes to slot
// (2j) mod n and V_j to slot (2j+1) mod n, so the producer can run several
// tiles ahead of the MMAs: with one CTA per SM the loads from L2 are latency
// bound, and bytes in flight set the rate (at d = 128 with two heads, 4
// slots measured as fast as 5).
template <int D, int T, bool F8>
struct PrefillSmem {
    static constexpr int kHalves = D / 64;                 // 64-column (128-byte) halves
    static constexpr int kTileBytes = kHalves * 128 * 128; // 128 rows x D, 16-bit elements
    static constexpr int kLTile = F8 ? kTileBytes / 2 : kTileBytes;   // a tile as loaded
    static constexpr int kQ = 0;                           // T query tiles
    static constexpr int kRing = T * kTileBytes;           // ring of loaded tiles
    static constexpr int kStageBytes = 4 * T * 4096;      // 32 rows x 64 columns bf16 per warp
    static constexpr int kAvail = 232448 - 1024 - kRing - kStageBytes - 512;
    // FP8, d = 128 (in place): an E4M3 tile lands in the upper half of its f16
    // slot (row r's 128 codes where the f16 row r of the upper 64 columns
    // goes) and is widened where it lies, so the slots serve both rings.
    // FP8, d = 64: a ring of widened f16 tiles (2..4 slots) and a separate
    // ring of loaded tiles from the rest.
    static constexpr bool kInPlace = F8 && D == 128;
    static constexpr int kFitTiles = kAvail / kTileBytes;
    static constexpr int kCSlotsFit = (kAvail / 2) / kTileBytes;
    static constexpr int kCSlots = !F8 ? 0
                                 : kInPlace ? (kFitTiles > 8 ? 8 : kFitTiles)
                                            : (kCSlotsFit > 4 ? 4 : (kCSlotsFit < 2 ? 2 : kCSlotsFit));
    static constexpr int kSlotsFit = kInPlace ? kCSlots : (kAvail - kCSlots * kTileBytes) / kLTile;
    static constexpr int kSlots = kSlotsFit > 8 ? 8 : kSlotsFit;
    static constexpr int kLStride = kInPlace ? kTileBytes : kLTile;       // landing slot stride
    static constexpr int kLOff = kInPlace ? kTileBytes - kLTile : 0;      // landing offset in a slot
    static constexpr int kConv = kInPlace ? kRing : kRing + kSlots * kLTile;
    static constexpr int kStage = kInPlace ? kRing + kCSlots * kTileBytes : kConv + kCSlots * kTileBytes;
    static constexpr int kBars = kStage + kStageBytes;
    static constexpr int kTotal = kBars + 512;
};

// Eight bf16 (one 16-byte piece of a Q tile) to eight f16 of x * s.
__device__ __forceinline__ uint4 bf16x8_to_f16x8_scaled(uint4 x, float s) {
    const uint32_t w[4] = {x.x, x.y, x.z, x.w};
    uint32_t o[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const __half2 h = __floats2half2_rn(__uint_as_float(w[i] << 16) * s, __uint_as_float(w[i] & 0xffff0000u) * s);
        o[i] = *reinterpret_cast<const uint32_t *>(&h);
    }
    return make_uint4(o[0], o[1], o[2], o[3]);
}


__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
    const __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&h);
}

__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }
// The mbarrier counts one more pending arrival until every cp.async this
// thread issued so far has landed (a regular arrive must follow).
__device__ __forceinline__ void cp_async_mbar_arrive(uint64_t *bar) {
    asm volatile("cp.async.mbarrier.arrive.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}
// Page size 1: warps that gather K/V rows (the producer and the two warps of
// the control warpgroup that have no other role, fewer if the ring is
// shorter), loads dealt out round robin.  bf16: each warp waits for its
// copies, fences and signals the load.  FP8 (the producer gathers alone): a
// load's barrier completes when its copies have landed and the warp goes on
// to its next load at once (410 us against 446 on the FP8 extend workload;
// with three bf16 gather warps the same measured no gain, and the proxy fence
// it moves into the MMA thread cost page size 16 about 2 %).
// Measured on the extend workload with page size 1 (5 ring slots): 1 warp
// 698 us, 2 warps 393 us, 3 warps 282 us.
constexpr int kGatherWarpsMax = 3;

// Register split (T = 2): 384 threads launch with kLaunchRegs = 168
// registers each (64,512 in all); the softmax warpgroups raise theirs to 184 and the
// producer/MMA warpgroup lowers its to 128: 256 * 184 + 128 * 128 = 63,488.
constexpr int kSoftmaxRegs = 184;
constexpr int kItemRing = 4;      // items published ahead of the consumers
constexpr int kControlRegs = 128;
constexpr int kLaunchRegs = 168;

// The split above waits forever if the launch holds fewer registers than its
// sum, so a T = 2 launch first checks what the compiler gave the kernel.
template <class Kernel>
cudaError_t check_register_split(Kernel kern) {
    cudaFuncAttributes fa{};
    const cudaError_t e = cudaFuncGetAttributes(&fa, kern);
    if (e != cudaSuccess) return e;
    return fa.numRegs >= kLaunchRegs ? cudaSuccess : cudaErrorNotSupported;
}

// EXT: the instantiation for sliding windows and block-sparse masks (plain
// launches keep that arithmetic out of their registers).
template <int D, int T, bool F8, bool EXT>
__device__ __forceinline__ void prefill_body(const PrefillArgs &a, int sched_ctas = 0) {
    using S = PrefillSmem<D, T, F8>;
    // A kernel launched after this one as a programmatic dependent (decode
    // sharing the GPU) may start once every CTA of this grid is resident.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    constexpr int H = S::kHalves;
    constexpr int kProducer = 4 * T;
    constexpr int kMma = 4 * T + 1;
    constexpr int kOCols = D == 128 ? 128 : 64;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

    uint8_t *sQ = smem + S::kQ;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + S::kBars);
    constexpr int NS = S::kSlots;
    // G < NS gather warps leave the MMA a slot; with FP8 pools the two spare
    // warps widen tiles instead
    constexpr int kGatherWarps = F8 ? 1 : (NS - 1 < kGatherWarpsMax ? NS - 1 : kGatherWarpsMax);
    constexpr int NC = F8 ? S::kCSlots : NS;  // slots the MMA reads from
    constexpr int kConverters = F8 ? 2 : 0;
    constexpr bool kInPlace = S::kInPlace;
    auto land = [&](int slot) { return smem + S::kRing + slot * S::kLStride + S::kLOff; };
    uint64_t *q_full = bars;                 // 1: Q tiles of the item loaded
    uint64_t *q_empty = bars + 1;            // 1: every S MMA of the item done
    uint64_t *full = bars + 2;               // NS: slot loaded
    uint64_t *empty = full + NS;             // NS: slot consumed (by the MMAs, or widened)
    uint64_t *cfull = empty + NS;            // FP8, NC: widened slot ready
    uint64_t *cempty = cfull + (F8 ? NC : 0);  // FP8, NC: widened slot consumed by the MMAs
    uint64_t *q_conv = cempty + (F8 ? NC : 0); // FP8, 1: Q tiles widened to f16
    uint64_t *s_full = q_conv + 1;           // T
    uint64_t *p_full = s_full + T;           // T
    uint64_t *o_final = p_full + T;          // T: every MMA of O_k of an item (with keys) done
    constexpr int R = kItemRing;
    uint64_t *item_full = o_final + T;       // R: item index published
    uint64_t *item_empty = item_full + R;    // R: read by the MMA warp, every softmax warp
                                             //    and (page size 1) the other gather warps
    int *item_idx = reinterpret_cast<int *>(item_empty + R);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(item_idx + R);
    // Each role walks the same item list and keeps its own counts of items
    // (phase of q_full / q_empty), items with keys (phase of o_final), key
    // steps (phase of s_full / p_full) and K/V loads (ring slot and phase).

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const bool paged16 = (a.page_size == 16);

    if (warp == kMma) tmem_alloc(tmem_slot, 512);
    if (threadIdx.x == 0) {
        mbar_init(q_full, 1);
        mbar_init(q_empty, 1);
        for (int s = 0; s < NS; ++s) {
            mbar_init(&full[s], paged16 ? 1 : 32);
            mbar_init(&empty[s], (F8 && !kInPlace) ? kConverters : 1);
        }
        if (F8) {
            for (int s = 0; s < NC; ++s) {
                mbar_init(&cfull[s], kConverters);
                mbar_init(&cempty[s], 1);
            }
            mbar_init(q_conv, kConverters);
        }
        for (int k = 0; k < T; ++k) {
            mbar_init(&s_full[k], 1);
            mbar_init(&p_full[k], 128);
        }
        for (int k = 0; k < T; ++k) mbar_init(&o_final[k], 1);
        for (int i = 0; i < R; ++i) {
            mbar_init(&item_full[i], 1);
            mbar_init(&item_empty[i], 1 + 4 * T + (paged16 ? 0 : kGatherWarps - 1) + kConverters);
        }
        fence_mbar_init();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    // Page size 1 gathers.  gather_rows reads the page-table entries of K or
    // V tile c of item `it` (lane l holds keys l, l + 32, ...); gather_copy
    // copies those rows with cp.async into ring slot gl in the 128-byte-
    // swizzled layout TMA would produce (rows past the visible keys are
    // zero), two key rows per instruction (16 lanes x 16 bytes per 256-byte
    // row at d = 128), as one copy group.
    auto gather_rows = [&](const PrefillItem &it, int st, int (&rows)[kBN / 32]) {
        const int32_t *pt = a.page_table + (int64_t)it.b * a.pt_stride;
        const int key0 = (it.j0 + st) * kBN;
#pragma unroll
        for (int rr = 0; rr < kBN / 32; ++rr) {
            const int key = key0 + rr * 32 + lane;
            rows[rr] = key < it.kv_end ? pt[key] : -1;
        }
    };
    auto gather_copy = [&](const PrefillItem &it, int c, int st, int gl, const int (&rows)[kBN / 32]) {
        if constexpr (F8) {
            // E4M3 rows of D bytes, copied as they are (row-major, no swizzle)
            constexpr int kChunks = D / 16;
            constexpr int kRowsPerIssue = 32 / kChunks;
            uint8_t *dst = land(gl % NS);
            const uint8_t *src = (c & 1) ? a.v_cache : a.k_cache;
            const int key0 = (it.j0 + st) * kBN;
            const int q = lane % kChunks, sub = lane / kChunks;
#pragma unroll 1
            for (int rr = 0; rr < kBN / 32; ++rr) {
                int row = rr == 0 ? rows[0] : rr == 1 ? rows[1] : rr == 2 ? rows[2] : rows[3];
                if (key0 + rr * 32 + lane < it.kv_end && (row < 0 || row >= a.num_slots)) {
                    raise_error(PA_DEVERR_PAGE_RANGE);
                    row = -1;
                }
#pragma unroll 4
                for (int i = 0; i < 32 / kRowsPerIssue; ++i) {
                    const int rl = i * kRowsPerIssue + sub;
                    const int rowv = __shfl_sync(0xffffffffu, row, rl);
                    const int r = rr * 32 + rl;
                    if (rowv >= 0)
                        cp_async16(dst + r * D + q * 16, src + ((int64_t)rowv * a.num_kv_heads + it.kvh) * (int64_t)D + q * 16);
                    else
                        *reinterpret_cast<uint4 *>(dst + r * D + q * 16) = make_uint4(0, 0, 0, 0);
                }
            }
            cp_async_commit();
            return;
        }
        constexpr int kChunks = D / 8;                // 16-byte chunks per row
        constexpr int kRowsPerIssue = 32 / kChunks;   // 2 (d = 128) or 4 (d = 64)
        uint8_t *dst = smem + S::kRing + (gl % NS) * S::kTileBytes;
        const uint8_t *src = (c & 1) ? a.v_cache : a.k_cache;
        const int key0 = (it.j0 + st) * kBN;
        const int q = lane % kChunks;                 // this lane's chunk of a row
        const int hh = q / 8;
        const int sub = lane / kChunks;
        static_assert(kBN / 32 == 4, "row selection below assumes 4 blocks of 32 keys");
        // rolled loops: the kernel's code is large and instruction fetch
        // stalls were measured when this part was fully unrolled
#pragma unroll 1
        for (int rr = 0; rr < kBN / 32; ++rr) {
            int row = rr == 0 ? rows[0] : rr == 1 ? rows[1] : rr == 2 ? rows[2] : rows[3];
            if (key0 + rr * 32 + lane < it.kv_end && (row < 0 || row >= a.num_slots)) {
                raise_error(PA_DEVERR_PAGE_RANGE);
                row = -1;
            }
#pragma unroll 4
            for (int i = 0; i < 32 / kRowsPerIssue; ++i) {
                const int rl = i * kRowsPerIssue + sub;            // row within this block of 32
                const int rowv = __shfl_sync(0xffffffffu, row, rl);
                const int r = rr * 32 + rl;                        // row within the tile
                const int so = hh * 16384 + r * 128 + (((q % 8) ^ (r & 7)) * 16);
                if (rowv >= 0)
                    cp_async16(dst + so, src + ((int64_t)rowv * a.num_kv_heads + it.kvh) * (int64_t)D * 2 + q * 16);
                else
                    *reinterpret_cast<uint4 *>(dst + so) = make_uint4(0, 0, 0, 0);
            }
        }
        cp_async_commit();
    };
    // The loads of one item that gather warp g issues (page size 1): loads
    // g, g + kGatherWarps, ... of the CTA.  Each waits for its ring slot, is
    // copied and signalled (see above; the regular arrive releases the zero
    // rows written for keys past the end); the next load's page-table entries
    // are read while the copies are in flight.  False on a timeout.
    auto gather_item = [&](const PrefillItem &it, int gl0, int g) {
        const int n = 2 * it.n_kv;
        int c = ((g - gl0) % kGatherWarps + kGatherWarps) % kGatherWarps;
        if (c >= n) return true;
        StepCursor cur;
        int rows[kBN / 32];
        int st = cur.at<EXT>(a, it, c >> 1);
        gather_rows(it, st, rows);
        for (; c < n; c += kGatherWarps) {
            const int gl = gl0 + c;
            if (gl >= NS && !mbar_wait(&empty[gl % NS], ((gl / NS) - 1) & 1)) return false;
            gather_copy(it, c, st, gl, rows);
            if (c + kGatherWarps < n) {
                st = cur.at<EXT>(a, it, (c + kGatherWarps) >> 1);
                gather_rows(it, st, rows);
            }
            if constexpr (F8) {        // the widening warps read the rows with generic loads
                cp_async_mbar_arrive(&full[gl % NS]);
            } else {
                cp_async_wait_all();
                fence_proxy_async_smem();  // generic-proxy writes -> visible to the MMA
            }
            mbar_arrive(&full[gl % NS]);
        }
        return true;
    };

    if (warp >= kProducer) {
        // ------------------------------------- producer / MMA warpgroup ----
        if (T == 2) asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kControlRegs));
      if (warp == kProducer) {
        // ----------------------------------------------------- producer ----
        if (lane == 0) {
            prefetch_tmap(&a.qmap);
            if (paged16) { prefetch_tmap(&a.kmap); prefetch_tmap(&a.vmap); }
        }
        // K/V tiles are re-read by the other items of their request:
        // evict-last keeps them in L2 beside a concurrent stream (a decode
        // launch next to this one)
        const uint64_t kv_pol = l2_policy_evict_last();
        // Take item n (lane 0) and publish its index, or the end mark, to
        // the other roles.  Returns the index (all lanes), -2 on a timeout.
        auto take = [&](int n) {
            int v = 0;
            if (lane == 0) {
                v = prefill_fetch<T>(a);
                const int slot = n % R;
                if (n >= R && !mbar_wait(&item_empty[slot], ((n / R) - 1) & 1)) {
                    v = -2;
                } else {
                    item_idx[slot] = v;
                    mbar_arrive(&item_full[slot]);
                }
            }
            return __shfl_sync(0xffffffffu, v, 0);
        };
        // Page size 16: lanes 0..7 read the ids of the 8 pages of 128-key
        // step j (-1 past the visible keys); page_slot0 turns one into the
        // first slot of the page, num_slots (zero fill) when there is none or
        // the id is outside the pool.  Split so that the read is in flight
        // while the producer waits for a ring slot.
        auto page_id = [&](const PrefillItem &it, int j) {      // j: the step (relative to j0)
            const int kk = (it.j0 + j) * kBN + lane * 16;
            return (lane < kBN / 16 && kk < it.kv_end) ? a.page_table[(int64_t)it.b * a.pt_stride + kk / 16] : -1;
        };
        auto page_slot0 = [&](const PrefillItem &it, int j, int page) {
            const int kk = (it.j0 + j) * kBN + lane * 16;
            if (lane >= kBN / 16 || kk >= it.kv_end) return a.num_slots;
            if (page >= 0 && (int64_t)page * 16 < a.num_slots) return page * 16;
            raise_error(PA_DEVERR_PAGE_RANGE);
            return a.num_slots;
        };
        int local = 0, gl = 0;
        PrefillItem it;
        // An item is taken when the previous one's loads are all issued (not
        // earlier: a CTA that holds an item it has not started keeps it from
        // CTAs that are idle at the end).
        for (int v; (v = take(local)) >= 0;) {
            prefill_item<T, EXT>(a, v, it);
            // load 2j is K_j, 2j + 1 is V_j; gl counts loads over the CTA's
            // life.  The Q tiles are loaded once the previous item's last S
            // MMA is done.
            bool ok = true;
            auto load_q = [&]() {
                if (local > 0 && !mbar_wait(q_empty, (local - 1) & 1)) return false;
                if (lane == 0) {
                    mbar_arrive_expect_tx(q_full, T * S::kTileBytes);
                    for (int k = 0; k < T; ++k)
                        for (int hh = 0; hh < H; ++hh)
                            tma_load_3d(sQ + k * S::kTileBytes + hh * 16384, &a.qmap, hh * 64, it.h0 + k,
                                        it.q0 + it.tile * kBM, q_full);
                }
                return true;
            };
            if (paged16) {
                StepCursor cur;                         // load c belongs to kept step c >> 1
                int st = cur.at<EXT>(a, it, 0);
                int page = page_id(it, st);             // pages of the current step
                int slot0 = a.num_slots;
                ok = load_q();
                for (int c = 0; ok && c < 2 * it.n_kv; ++c, ++gl) {
                    if (!(c & 1)) slot0 = page_slot0(it, st, page);
                    const int slot = gl % NS, round = gl / NS;
                    if (round > 0 && !mbar_wait(&empty[slot], (round - 1) & 1)) { ok = false; break; }
                    uint8_t *dst = land(slot);
                    // lanes 0..7 each own one 16-token page of the tile
                    if (lane == 0) mbar_arrive_expect_tx(&full[slot], S::kLTile);
                    __syncwarp();
                    if (lane < kBN / 16) {
                        const CUtensorMap *map = (c & 1) ? &a.vmap : &a.kmap;
                        if constexpr (F8) {           // one (D bytes x 16 rows) box per page
                            tma_load_3d_hint(dst + lane * 16 * D, map, 0, it.kvh, slot0, &full[slot], kv_pol);
                        } else {
#pragma unroll
                            for (int hh = 0; hh < H; ++hh)
                                tma_load_3d_hint(dst + hh * 16384 + lane * 2048, map, hh * 64, it.kvh, slot0,
                                                 &full[slot], kv_pol);
                        }
                    }
                    // K_j and V_j share pages; after K_j start reading the next step's
                    if (!(c & 1) && c + 2 < 2 * it.n_kv) {
                        st = cur.at<EXT>(a, it, (c >> 1) + 1);
                        page = page_id(it, st);
                    }
                }
            } else {
                ok = load_q() && gather_item(it, gl, 0);
                gl += 2 * it.n_kv;
            }
            if (!ok) break;
            ++local;
        }
        if (lane == 0) prefill_sched_done(a, a.num_ctas > 0 ? a.num_ctas : sched_ctas);
      } else if (warp != kMma && !paged16 && warp - kMma < kGatherWarps) {
        // --------------------------------- extra gather warps (page 1) ----
        const int g = warp - kMma;                      // 1, 2
        int local = 0, gl = 0;
        PrefillItem it;
        for (;;) {
            const int slot = local % R;
            if (!__all_sync(0xffffffffu, mbar_wait(&item_full[slot], (local / R) & 1))) break;
            const int v = item_idx[slot];
            __syncwarp();
            if (lane == 0) mbar_arrive(&item_empty[slot]);
            ++local;
            if (v < 0) break;
            prefill_item<T, EXT>(a, v, it);
            if (!gather_item(it, gl, g)) break;
            gl += 2 * it.n_kv;
        }
      } else if (F8 && warp > kMma) {
        // -------------------------------------- FP8 widening (2 warps) ----
        const int cw = warp - kMma - 1;                 // 0, 1: rows [64 cw, 64 cw + 64)
        int local = 0, gl = 0;
        bool ok = true;
        PrefillItem it;
        while (ok) {
            const int slot = local % R;
            if (!__all_sync(0xffffffffu, mbar_wait(&item_full[slot], (local / R) & 1))) break;
            const int v = item_idx[slot];
            __syncwarp();
            if (lane == 0) mbar_arrive(&item_empty[slot]);
            if (v < 0) break;
            prefill_item<T, EXT>(a, v, it);
            // Q tiles: bf16 -> f16 of q * k_scale, in place
            if (!__all_sync(0xffffffffu, mbar_wait(q_full, local & 1))) break;
            ++local;
            const float ksc = __ldg(a.k_scale + it.kvh);
#pragma unroll 4
            for (int i = cw * 32 + lane; i < T * S::kTileBytes / 16; i += 64) {
                uint4 *pq = reinterpret_cast<uint4 *>(sQ + i * 16);
                *pq = bf16x8_to_f16x8_scaled(*pq, ksc);
            }
            fence_proxy_async_smem();                   // generic writes -> MMA (async proxy)
            __syncwarp();
            if (lane == 0) mbar_arrive(q_conv);
            // K/V tiles: E4M3 rows -> f16 in the swizzled K-major layout
            for (int c = 0; c < 2 * it.n_kv; ++c, ++gl) {
                const int ls = gl % NS, cs = gl % NC;
                ok = __all_sync(0xffffffffu, mbar_wait(&full[ls], (gl / NS) & 1));
                // (in place the slot was free before it was loaded)
                if (ok && !kInPlace && gl >= NC)
                    ok = __all_sync(0xffffffffu, mbar_wait(&cempty[cs], ((gl / NC) - 1) & 1));
                if (!ok) break;
                const uint8_t *src = land(ls);
                uint8_t *dst = smem + S::kConv + cs * S::kTileBytes;
                // groups of 4 x 512 bytes: all reads of a group, then (in
                // place, after the warp has read them) the writes, which
                // overwrite only rows of the same group
                constexpr int kGroup = 4;
#pragma unroll 1
                for (int i0 = 0; i0 < 64 * D / 512; i0 += kGroup) {
                    uint4 x[kGroup];
#pragma unroll
                    for (int u = 0; u < kGroup; ++u) {
                        const int byte = (i0 + u) * 512 + lane * 16;   // within this warp's 64 rows
                        x[u] = *reinterpret_cast<const uint4 *>(src + (64 * cw + byte / D) * D + (byte % D));
                    }
                    if (kInPlace) __syncwarp();
#pragma unroll
                    for (int u = 0; u < kGroup; ++u) {
                        const int byte = (i0 + u) * 512 + lane * 16;
                        const int rr = 64 * cw + byte / D;
                        const int q = (byte % D) / 16;      // 16 codes: d = 16 q .. 16 q + 15
                        uint4 lo, hi;
                        e4m3x4_to_f16x4(x[u].x, lo.x, lo.y);
                        e4m3x4_to_f16x4(x[u].y, lo.z, lo.w);
                        e4m3x4_to_f16x4(x[u].z, hi.x, hi.y);
                        e4m3x4_to_f16x4(x[u].w, hi.z, hi.w);
                        const int hh = q / 4, c0 = 2 * (q % 4);
                        uint8_t *row = dst + hh * 16384 + rr * 128;
                        *reinterpret_cast<uint4 *>(row + ((c0 ^ (rr & 7)) * 16)) = lo;
                        *reinterpret_cast<uint4 *>(row + (((c0 + 1) ^ (rr & 7)) * 16)) = hi;
                    }
                }
                // Rows of an item's last V tile at keys >= kv_end are slots
                // the store never wrote (the last page is loaded whole): P is
                // 0 there, but 0 * NaN is not, so they become zeros (this
                // warp's rows of the page that holds key kv_end - 1; later
                // pages are zero-filled by the TMA).
                if (c == 2 * it.n_kv - 1 && (it.kv_end & 15) && StepCursor().at<EXT>(a, it, it.n_kv - 1) == it.n_all - 1) {
                    __syncwarp();
                    const int kbase = (it.j0 + it.n_all - 1) * kBN;
                    const int r0 = max(it.kv_end - kbase, 64 * cw);
                    const int r1 = min(((it.kv_end + 15) & ~15) - kbase, 64 * cw + 64);
                    for (int i = lane; i < (r1 - r0) * (D / 8); i += 32) {
                        const int row = r0 + i / (D / 8), ch = i % (D / 8);
                        *reinterpret_cast<uint4 *>(dst + (ch / 8) * 16384 + row * 128 + (ch % 8) * 16) =
                            make_uint4(0u, 0u, 0u, 0u);
                    }
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(&cfull[cs]);
                    if (!kInPlace) mbar_arrive(&empty[ls]);
                }
            }
        }
      } else if (warp == kMma) {
        // ---------------------------------------------------------- MMA ----
        if (lane == 0) {
            constexpr uint32_t idesc_s = F8 ? umma_idesc_f16(kBM, kBN, false) : umma_idesc_bf16(kBM, kBN, false);
            constexpr uint32_t idesc_o = F8 ? umma_idesc_f16(kBM, D, true) : umma_idesc_bf16(kBM, D, true);
            // the slots the MMAs read (FP8: the widened ring) and their barriers
            uint8_t *mring = smem + (F8 ? S::kConv : S::kRing);
            uint64_t *mfull = F8 ? cfull : full;
            uint64_t *mempty = (F8 && !kInPlace) ? cempty : empty;   // in place: frees the loaded slot too
            // Descriptors are built once; a k-step adds its byte offset >> 4 to
            // the 14-bit start-address field (shared addresses stay < 2^18).
            const uint64_t dq0 = umma_desc_sw128(smem_u32(sQ), 16, 1024);
            const uint64_t dk0 = umma_desc_sw128(smem_u32(mring), 16, 1024);
            const uint64_t dv0 = umma_desc_sw128(smem_u32(mring), 16384, 1024);
            auto wait_full = [&](int c) { return mbar_wait(&mfull[c % NC], (c / NC) & 1); };
            auto issue_s = [&](int k, int c) {            // S_k from the K tile of load c
                const uint64_t dq = dq0 + (uint64_t)((k * S::kTileBytes) >> 4);
                const uint64_t dk = dk0 + (uint64_t)(((c % NC) * S::kTileBytes) >> 4);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint64_t o = (uint64_t)(((kk / 4) * 16384 + (kk % 4) * 32) >> 4);
                    umma_ss(tmem + 128 * k, dq + o, dk + o, idesc_s, kk > 0);
                }
                umma_commit(&s_full[k]);
            };
            int local = 0, gl = 0, gs = 0;
            bool ok = true;
            PrefillItem it;
            while (ok) {
                const int slot = local % R;
                if (!mbar_wait(&item_full[slot], (local / R) & 1)) break;
                const int v = item_idx[slot];
                mbar_arrive(&item_empty[slot]);
                if (v < 0) break;
                prefill_item<T, EXT>(a, v, it);
                const int n_kv = it.n_kv;
                if (!mbar_wait(F8 ? q_conv : q_full, local & 1)) break;
                if (n_kv > 0) {
                    if (!wait_full(gl)) break;
                    tc_fence_after();
                    for (int k = 0; k < T; ++k) issue_s(k, gl);
                    umma_commit(&mempty[gl % NC]);                       // K_0 consumed
                }
                if (n_kv <= 1) umma_commit(q_empty);                     // every S of the item issued
                for (int j = 0; ok && j < n_kv; ++j) {
                    const int cv = gl + 2 * j + 1;
                    const uint64_t dv = dv0 + (uint64_t)(((cv % NC) * S::kTileBytes) >> 4);
                    if (!F8 && paged16 && (it.kv_end & 15) && j + 1 == n_kv &&
                        StepCursor().at<EXT>(a, it, j) == it.n_all - 1) {
                        // The last page of a request is loaded whole (one
                        // 16-token TMA box), so rows of the item's last V tile
                        // at keys >= kv_end hold slots the store never wrote.
                        // P is 0 there, but 0 * NaN is not: clear those rows
                        // (at most 15, up to the end of the page; later pages
                        // are zero-filled by the TMA) once the tile has landed,
                        // while the softmax of this step still runs.  (FP8
                        // tiles are cleared by the widening warps.)
                        if (!wait_full(cv)) { ok = false; break; }
                        const int kbase = (it.j0 + it.n_all - 1) * kBN;      // the item's last step
                        const int r0 = it.kv_end - kbase;                  // first row past the keys
                        const int r1 = ((it.kv_end + 15) & ~15) - kbase;   // end of its page
                        uint8_t *vt = land(cv % NS);
                        for (int row = r0; row < r1; ++row)
#pragma unroll
                            for (int ch = 0; ch < D / 8; ++ch)
                                *reinterpret_cast<uint4 *>(vt + (ch / 8) * 16384 + row * 128 + (ch % 8) * 16) =
                                    make_uint4(0u, 0u, 0u, 0u);
                        fence_proxy_async_smem();                          // generic writes -> the MMA's reads
                    }
                    for (int k = 0; k < T; ++k) {
                        if (!mbar_wait(&p_full[k], (gs + j) & 1)) { ok = false; break; }
                        if (k == 0 && !wait_full(cv)) { ok = false; break; }
                        tc_fence_after();
                        const uint32_t o_tm = tmem + 256 + kOCols * k;
#pragma unroll
                        for (int kk = 0; kk < kBN / 16; ++kk)
                            umma_ts(o_tm, tmem + 128 * k + kk * 8, dv + (uint64_t)((kk * 16 * 128) >> 4), idesc_o,
                                    (j > 0 || kk > 0) ? 1u : 0u);
                        if (k == T - 1) umma_commit(&mempty[cv % NC]);   // V_j consumed
                        if (j + 1 == n_kv) umma_commit(&o_final[k]);     // O_k of the item complete
                        if (j + 1 < n_kv) {
                            if (k == 0) {
                                if (!wait_full(cv + 1)) { ok = false; break; }
                                tc_fence_after();
                            }
                            issue_s(k, cv + 1);
                            if (k == T - 1) {
                                umma_commit(&mempty[(cv + 1) % NC]);     // K_{j+1} consumed
                                if (j + 2 == n_kv) umma_commit(q_empty);  // last S of the item
                            }
                        }
                    }
                }
                // (items without keys write zeros and use no MMA)
                gl += 2 * n_kv;
                gs += n_kv;
                ++local;
            }
        }
      }
    } else {
        // ------------------------------------------------------ softmax ----
        if (T == 2) asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kSoftmaxRegs));
        const int k = warp >> 2;                      // query tile (head h0 + k)
        const int r = threadIdx.x & 127;              // row within the tile = TMEM lane
        const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
        const uint32_t s_tm = tmem + lane_base + 128 * k;
        const uint32_t o_tm = tmem + lane_base + 256 + kOCols * k;
        const float2 c2 = make_float2(a.scale_log2, a.scale_log2);
        int fin = 0, gs = 0, local = 0;
        bool ok = true;
        PrefillItem it;
        while (ok) {
        const int slot = local % R;
        ok = __all_sync(0xffffffffu, mbar_wait(&item_full[slot], (local / R) & 1));
        if (!ok) break;
        const int v = item_idx[slot];
        __syncwarp();
        if (lane == 0) mbar_arrive(&item_empty[slot]);
        ++local;
        if (v < 0) break;
        prefill_item<T, EXT>(a, v, it);
        const int n_kv = it.n_kv, Lk = it.Lk, off = it.off, min_vis = it.min_vis;
        const int qi = it.tile * kBM + r;             // query index within the request
        const bool row_valid = r < it.rows_here;
        const int vis_end = a.causal ? min(Lk, off + qi + 1) : Lk;   // keys [0, vis_end)
        float m_run = -INFINITY;
        float l_run = 0.f;
        StepCursor cur;                               // ordinal j -> kept step
        // tcgen05.ld / st are warp-collective (.sync.aligned): every branch
        // that encloses one is warp-uniform, and the warp reconverges after
        // each (per-lane) barrier wait.
        for (int j = 0; j < n_kv; ++j) {
            ok = __all_sync(0xffffffffu, mbar_wait(&s_full[k], (gs + j) & 1));
            if (!ok) break;
            tc_fence_after();
            uint32_t sr[kBN];
#pragma unroll
            for (int c = 0; c < kBN / 32; ++c) tmem_ld32(s_tm + c * 32, *reinterpret_cast<uint32_t(*)[32]>(&sr[c * 32]));
            tmem_wait_ld();
            const int kbase = (it.j0 + cur.at<EXT>(a, it, j)) * kBN;
            if (kbase + kBN > min_vis || (EXT && kbase < it.lo_max)) {   // diagonal / end / window edge: mask
                const int lim = row_valid ? vis_end - kbase : kBN;
                const int lo = (EXT && row_valid && a.window > 0) ? off + qi - (a.window - 1) - kbase : 0;
#pragma unroll
                for (int c = 0; c < kBN; ++c)
                    if (c >= lim || c < lo) sr[c] = __float_as_uint(-INFINITY);
            }
            // row maximum of the raw scores (scale > 0 commutes with max)
            float mx[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) mx[i] = __uint_as_float(sr[i]);
            // elements 0-7 above, then pairs of 8-element blocks, then the
            // last block on its own (kBN - 8 is not a multiple of 16)
            constexpr int kPairEnd = 8 + 16 * ((kBN - 8) / 16);
#pragma unroll
            for (int c = 8; c < kPairEnd; c += 16)
#pragma unroll
                for (int i = 0; i < 8; ++i) mx[i] = max3(mx[i], __uint_as_float(sr[c + i]), __uint_as_float(sr[c + 8 + i]));
#pragma unroll
            for (int c = kPairEnd; c < kBN; c += 8)
#pragma unroll
                for (int i = 0; i < 8; ++i) mx[i] = fmaxf(mx[i], __uint_as_float(sr[c + i]));
            const float mt = max3(max3(mx[0], mx[1], mx[2]), max3(mx[3], mx[4], mx[5]), fmaxf(mx[6], mx[7]));
            const float m_cand = mt * a.scale_log2;
            // lazy maximum: move it only when the tile maximum exceeds it by
            // more than kLazy; then O_k (PV_k(j-1) is complete: the commit of
            // S_k(j) tracks it) and l are rescaled
            const bool need = m_cand > m_run + kLazy;
            const float alpha = need ? fast_exp2(m_run - m_cand) : 1.f;
            if (j > 0 && __any_sync(0xffffffffu, need)) {
#pragma unroll
                for (int c = 0; c < D / 32; ++c) {
                    uint32_t orr[32];
                    tmem_ld32(o_tm + c * 32, orr);
                    tmem_wait_ld();
#pragma unroll
                    for (int e = 0; e < 32; ++e) orr[e] = __float_as_uint(__uint_as_float(orr[e]) * alpha);
                    tmem_st16(o_tm + c * 32, *reinterpret_cast<const uint32_t(*)[16]>(&orr[0]));
                    tmem_st16(o_tm + c * 32 + 16, *reinterpret_cast<const uint32_t(*)[16]>(&orr[16]));
                }
            }
            if (need) {
                l_run *= alpha;
                m_run = m_cand;
            }
            const float m_use = (m_run == -INFINITY) ? 0.f : m_run;
            const float2 nm2 = make_float2(-m_use, -m_use);
            float2 acc[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                             make_float2(0.f, 0.f)};
            uint32_t pk[kBN / 2];
#pragma unroll
            for (int c = 0; c < kBN / 2; ++c) {
                const float2 x = ffma2(make_float2(__uint_as_float(sr[2 * c]), __uint_as_float(sr[2 * c + 1])), c2, nm2);
                const float2 p = make_float2(fast_exp2(x.x), fast_exp2(x.y));
                acc[c & 3] = add2(acc[c & 3], p);
                pk[c] = F8 ? pack_f16x2(p.x, p.y) : pack_bf16x2(p.x, p.y);
            }
            const float2 s01 = add2(add2(acc[0], acc[1]), add2(acc[2], acc[3]));
            l_run += s01.x + s01.y;
#pragma unroll
            for (int c = 0; c < kBN / 32; ++c)
                tmem_st16(s_tm + c * 16, *reinterpret_cast<const uint32_t(*)[16]>(&pk[c * 16]));
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(&p_full[k]);
        }
        // ---- epilogue: O / l -> bf16, lse
        if (ok && n_kv > 0) ok = __all_sync(0xffffffffu, mbar_wait(&o_final[k], fin & 1));
        tc_fence_after();
        if (ok) {
            const int64_t tok = (int64_t)it.q0 + qi;
            const int h = it.h0 + k;
            const float inv = (l_run > 0.f ? 1.f / l_run : 0.f) * (F8 ? __ldg(a.v_scale + it.kvh) : 1.f);
            // Through the warp's staging buffer, 64 columns at a time: each
            // thread writes its row (16-byte pieces, XOR-swizzled by row so
            // the writes and reads below are free of bank conflicts), then the
            // warp stores 4 rows x 128 contiguous bytes per instruction.
            uint8_t *stage = smem + S::kStage + warp * 4096;
            const int rw = lane;                                   // row within the warp's 32
#pragma unroll 1
            for (int half = 0; half < D / 64; ++half) {
                // both 32-column loads in flight before one wait
                uint32_t orr[64];
                if (n_kv > 0) {                       // CTA-uniform
                    tmem_ld32(o_tm + half * 64, *reinterpret_cast<uint32_t(*)[32]>(&orr[0]));
                    tmem_ld32(o_tm + half * 64 + 32, *reinterpret_cast<uint32_t(*)[32]>(&orr[32]));
                    tmem_wait_ld();
                } else {
#pragma unroll
                    for (int e = 0; e < 64; ++e) orr[e] = 0u;
                }
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    uint4 w;
                    w.x = pack_bf16x2(__uint_as_float(orr[8 * u + 0]) * inv, __uint_as_float(orr[8 * u + 1]) * inv);
                    w.y = pack_bf16x2(__uint_as_float(orr[8 * u + 2]) * inv, __uint_as_float(orr[8 * u + 3]) * inv);
                    w.z = pack_bf16x2(__uint_as_float(orr[8 * u + 4]) * inv, __uint_as_float(orr[8 * u + 5]) * inv);
                    w.w = pack_bf16x2(__uint_as_float(orr[8 * u + 6]) * inv, __uint_as_float(orr[8 * u + 7]) * inv);
                    *reinterpret_cast<uint4 *>(stage + rw * 128 + ((u ^ (rw & 7)) * 16)) = w;
                }
                __syncwarp();
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int rr = i * 4 + (lane >> 3);
                    const int q = lane & 7;
                    const uint4 val = *reinterpret_cast<const uint4 *>(stage + rr * 128 + ((q ^ (rr & 7)) * 16));
                    const int rt = (warp & 3) * 32 + rr;                // row within the tile
                    if (rt < it.rows_here) {
                        const int64_t t = (int64_t)it.q0 + it.tile * kBM + rt;
                        *reinterpret_cast<uint4 *>(a.out + (t * a.num_q_heads + h) * D + half * 64 + q * 8) = val;
                    }
                }
                __syncwarp();
            }
            if (row_valid && a.lse != nullptr)
                a.lse[(int64_t)h * a.lse_stride + tok] =
                    l_run > 0.f ? (m_run + __log2f(l_run)) * 0.69314718055994531f : -INFINITY;
        }
        gs += n_kv;
        fin += n_kv > 0;
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == kMma) {
        __syncwarp();
        tmem_dealloc(tmem, 512);
    }
}

PFN_cuTensorMapEncodeTiled_v12000 encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess && q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// 3-D bf16 map (d, heads, rows) with a (64, 1, box_rows) box, 128-byte swizzle.
bool make_map(CUtensorMap *m, const void *base, int d, int heads, int64_t rows, int box_rows) {
    auto enc = encoder();
    if (!enc) return false;
    cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)heads, (cuuint64_t)rows};
    cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)heads * d * 2};
    cuuint32_t box[3] = {64, 1, (cuuint32_t)box_rows};
    cuuint32_t es[3] = {1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 3-D E4M3 map (d, heads, rows) with a (d, 1, box_rows) box, no swizzle.
bool make_map_fp8(CUtensorMap *m, const void *base, int d, int heads, int64_t rows, int box_rows) {
    auto enc = encoder();
    if (!enc) return false;
    cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)heads, (cuuint64_t)rows};
    cuuint64_t strides[2] = {(cuuint64_t)d, (cuuint64_t)heads * d};
    cuuint32_t box[3] = {(cuuint32_t)d, 1, (cuuint32_t)box_rows};
    cuuint32_t es[3] = {1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void *>(base), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Fill the kernel arguments of a validated pa_prefill call (tensor maps,
// metadata pointers, the work-item count; T = query heads per item).
cudaError_t prefill_setup(const pa_prefill_params &p, PrefillArgs &a, int &T) {
    a = PrefillArgs{};
    const int64_t num_slots = p.num_pages * p.page_size;
    if (!make_map(&a.qmap, p.q, p.head_dim, p.num_q_heads, p.total_q, kBM)) return cudaErrorNotSupported;
    const bool f8 = p.kv_dtype == PA_KV_FP8_E4M3;
    if (p.page_size == 16) {
        auto mk = f8 ? make_map_fp8 : make_map;
        if (!mk(&a.kmap, p.k_cache, p.head_dim, p.num_kv_heads, num_slots, 16)) return cudaErrorNotSupported;
        if (!mk(&a.vmap, p.v_cache, p.head_dim, p.num_kv_heads, num_slots, 16)) return cudaErrorNotSupported;
    }
    a.k_scale = p.k_scale;
    a.v_scale = p.v_scale;
    a.window = p.sliding_window;
    a.bmask = p.block_mask;
    a.bm_q = p.block_mask_q_blocks;
    a.bm_k = p.block_mask_k_blocks;
    a.k_cache = static_cast<const uint8_t *>(p.k_cache);
    a.v_cache = static_cast<const uint8_t *>(p.v_cache);
    a.page_table = p.page_table;
    a.pt_stride = p.page_table_stride;
    a.cu_q = p.cu_seqlens_q;
    a.cu_k = p.cu_seqlens_k;
    a.out = static_cast<__nv_bfloat16 *>(p.out);
    a.lse = p.lse;
    a.lse_stride = p.lse_stride;
    a.num_seqs = p.num_seqs;
    a.total_q = p.total_q;
    a.max_q = p.max_seqlen_q;
    a.max_k = p.max_seqlen_k;
    a.num_q_heads = p.num_q_heads;
    a.num_kv_heads = p.num_kv_heads;
    a.page_size = p.page_size;
    a.num_slots = (int32_t)num_slots;
    a.causal = p.causal;
    a.scale_log2 = p.scale * 1.4426950408889634f;
    // two query heads per CTA whenever they share a KV head
    const int group = p.num_q_heads / p.num_kv_heads;
    T = (group % 2 == 0) ? 2 : 1;
    const int64_t max_tiles = (p.max_seqlen_q + kBM - 1) / kBM;
    const int64_t virt = max_tiles * p.num_seqs * (p.num_q_heads / T);
    if (virt > INT32_MAX) return cudaErrorNotSupported;
    a.num_virtual = (int32_t)virt;
    return cudaSuccess;
}

}  // namespace
}  // namespace pa
