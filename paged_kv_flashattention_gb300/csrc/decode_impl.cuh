// Split-KV decode attention: the device code shared by the decode kernel
// and the mixed-batch kernel (prefill work items followed by decode key
// ranges in one persistent launch).  See decode.cu for the method and the
// work decomposition.
//
// "Transformer inference kernels: GEMM·Attention·FlashAttention·Fusion
// (3/10)": decode has one query token per sequence and a long cached context
// read through the page table (sections 13-14); several query heads share one
// KV head (section 15); a long key range is cut into splits whose partial
// (m, l, O) are merged by a numerically stable combine (sections 12, 16).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {
namespace {

constexpr int kStageTok = 16;     // tokens per pipeline stage
// Ring depth.  FP8 keeps 3 stages of half-length rows: the smaller ring lets
// 4 CTAs share an SM instead of 2, which measured faster than 6 stages at 2
// CTAs (each CTA's consumers work through one stage at a time).
// Three stages at every row length: at d = 64 (bf16 rows half as long), six
// stages halve the CTAs per SM and measured 1.5x slower on a Llama-3.2-1B
// shaped decode, and 1 KiB rows (8 KV heads per CTA) measured the same as 4.
// (FP8 with 8 KV heads per CTA: 2 or 4 stages measured slower than 3 too.)
template <int D, int EB, int HPC>
constexpr int stages_for() { return 3; }
// FP8 KV heads per CTA at most: 512-byte token rows at either head size (8
// heads at d = 64: Llama-3.2-1B shaped decode 45 us against 51 us with 4;
// 4 heads at d = 128: 8 measured 201 us against 194 us on a log-uniform mix).
template <int D>
constexpr int fp8_max_heads_per_cta() { return D == 64 ? 8 : 4; }
constexpr float kLazyRescale = 8.0f;  // log2 units

struct DecodeArgs {
    const __nv_bfloat16 *q;
    const uint8_t *k_cache;
    const uint8_t *v_cache;
    const int32_t *page_table;
    int64_t pt_stride;
    const int32_t *cache_seqlens;
    int32_t num_seqs;
    int32_t num_q_heads;
    int32_t num_kv_heads;
    int32_t page_size;
    int64_t num_pages;
    float scale_log2;
    int32_t min_split;            // smallest T (tokens per CTA range)
    int32_t max_seqlen_k;
    int32_t max_splits;
    int32_t head_groups;
    __nv_bfloat16 *out;
    float *lse;
    float *o_part;
    float *lse_part;
    const float *k_scale;         // FP8 pools: per-KV-head scales
    const float *v_scale;
    int32_t window;               // sliding window W (0 = none): the last W keys
    int32_t max_ctas;             // host only: cap on the persistent grid (0 = every SM)
    int32_t overlap_previous;     // host only: launch as a programmatic dependent
    int32_t *ws_header;           // [0] = T
    int32_t *ws_prefix;           // [B+1] exclusive prefix of the sequence lengths
    int32_t evict_first;          // K/V row copies with an L2 evict-first policy (beside a prefill)
};

template <int D, int HPC, int EB, int STAGES = stages_for<D, EB, HPC>()>
struct DecodeSmem {
    static constexpr int kRowBytes = HPC * D * EB;           // one token, CTA's KV heads (EB bytes each)
    static constexpr int kRowStride = kRowBytes + 16;        // +16 B: ldmatrix rows hit distinct banks
    static constexpr int kStageBytes = 2 * kStageTok * kRowStride;
    static constexpr int kStages = STAGES;
    static constexpr int kRingBytes = kStages * kStageBytes;
};

// Warp-level bf16 MMA, D(16x8, fp32) += A(16x16, row) * B(16x8, col).
__device__ __forceinline__ void mma_bf16_16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Four 8x8 b16 matrices from shared memory (each lane gives one row address).
__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(addr) : "memory");
}
__device__ __forceinline__ void ldsm_x4_trans(uint32_t (&r)[4], uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(addr) : "memory");
}

// Warp-level f16 MMA, D(16x8, fp32) += A(16x16, row) * B(16x8, col).
__device__ __forceinline__ void mma_f16_16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t f16x2_bits(float lo, float hi) {
    return (uint32_t)__half_as_ushort(__float2half_rn(lo)) | ((uint32_t)__half_as_ushort(__float2half_rn(hi)) << 16);
}

__device__ __forceinline__ uint16_t bf16_bits(float x) {
    return __bfloat16_as_ushort(__float2bfloat16_rn(x));
}

// Walks the segments of a range [g, g1) of the sequence-major row list; pb
// is the exclusive prefix of the sequence lengths, so sequence b's rows start
// at HG * pb[b] and row (b, hg) at HG * pb[b] + hg * L_b.  The split layout
// cuts the list every T rows: a row's split s is its part in the s-th T-range
// it overlaps.  A segment's partial belongs to the split of its first row;
// span > 1 when the segment runs on through further T-ranges (a walk over
// several consecutive ranges), whose split slots of this row stay empty.
struct SegmentWalk {
    const int32_t *pb;
    int B, HG;
    int64_t T, g, g1;
    __device__ bool next(int &b, int &hg, int &t0, int &t1, int &split, int &span) {
        if (g >= g1) return false;
        int lo = 0, hi = B;           // HG * pb[lo] <= g < HG * pb[hi]
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if ((int64_t)HG * pb[mid] <= g) lo = mid; else hi = mid;
        }
        b = lo;
        const int L = pb[b + 1] - pb[b];                  // > 0 by the invariant
        const int64_t local = g - (int64_t)HG * pb[b];
        hg = (int)(local / L);
        t0 = (int)(local % L);
        const int64_t want = (int64_t)t0 + (g1 - g);
        t1 = want < L ? (int)want : L;
        const int64_t row_start = (int64_t)HG * pb[b] + (int64_t)hg * L;
        split = (int)(g / T - row_start / T);
        span = (int)((g + (t1 - t0) - 1) / T - g / T) + 1;
        g += t1 - t0;
        return true;
    }
};

// Exclusive prefix of the sequence lengths, clamped to max_seqlen_k and (with
// a sliding window) to the last W keys, into prefix[0 .. B].  Called by every
// thread of the CTA (it synchronises the CTA twice).
__device__ __forceinline__ void decode_prefix(const DecodeArgs &a, int32_t *prefix) {
    const int B = a.num_seqs;
    // Exclusive prefix of the sequence lengths (clamped to max_seqlen_k):
    // loaded by all threads, scanned by warp 0.
    for (int b = threadIdx.x; b < B; b += blockDim.x) {
        int L = a.cache_seqlens[b];
        if (L < 0 || L > a.max_seqlen_k) {
            raise_error(PA_DEVERR_SEQLENS);
            L = L < 0 ? 0 : a.max_seqlen_k;
        }
        if (a.window > 0 && L > a.window) L = a.window;     // only the last W keys are read
        prefix[b + 1] = L;
    }
    if (threadIdx.x == 0) prefix[0] = 0;
    __syncthreads();
    if ((threadIdx.x >> 5) == 0) {
        const int lane = threadIdx.x & 31;
        // each lane scans a contiguous run, then the run totals are scanned
        const int per = (B + 31) / 32;
        const int lo = 1 + lane * per, hi = min(B, lane * per + per);
        int run = 0;
        for (int i = lo; i <= hi; ++i) run += prefix[i];
        int incl = run;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += v;
        }
        int acc = incl - run;
        for (int i = lo; i <= hi; ++i) {
            acc += prefix[i];
            prefix[i] = acc;
        }
    }
    __syncthreads();
}

// Rows [g0, g1) of the sequence-major (sequence, head group, key) list form
// key range `chunk` (ranges of T rows).  The producer warp streams its
// 16-token stages into the ring (per token one bulk copy of the K row and
// one of the V row), continuing the stage count of earlier ranges.  False
// on a timeout.
// part 0: this warp issues the K and the V rows of every stage (lanes 0-15
// K, 16-31 V); part 1: only the K rows; part 2: only the V rows (a second
// producer warp on the same ranges and stages: twice the copy-issue rate).
// Each producer warp arrives on a stage's full barrier once, expecting the
// bytes it copies itself (the barrier counts one arrival per producer warp).
template <int D, int HPC, int EB, int STAGES = stages_for<D, EB, HPC>()>
__device__ bool decode_produce(const DecodeArgs &a, const int32_t *prefix, int64_t T, int64_t g0,
                               int64_t g1, uint8_t *ring, uint64_t *full, uint64_t *empty, int &stage_ctr,
                               int lane, int part = 0) {
    using S = DecodeSmem<D, HPC, EB, STAGES>;
    constexpr int kStages = S::kStages;
    const int B = a.num_seqs, HG = a.head_groups;
    // every K/V row is read once: beside a prefill, evict-first keeps the
    // stream from pushing out of L2 the tiles the prefill re-reads (alone,
    // the plain copies measured faster)
    const uint64_t policy = l2_policy_evict_first();
    SegmentWalk walk{prefix, B, HG, T, g0, g1};
    int b, hg, k0, k1, split, span;
    while (walk.next(b, hg, k0, k1, split, span)) {
        const int32_t *pt = a.page_table + (int64_t)b * a.pt_stride;
        // with a sliding window the row's tokens start s0 keys in
        int Lb = a.cache_seqlens[b];
        Lb = Lb < 0 ? 0 : (Lb > a.max_seqlen_k ? a.max_seqlen_k : Lb);
        const int s0 = Lb - (prefix[b + 1] - prefix[b]);
        for (int t0 = k0; t0 < k1; t0 += kStageTok, ++stage_ctr) {
            const int slot = stage_ctr % kStages;
            const int round = stage_ctr / kStages;
            if (round > 0 && !mbar_wait(&empty[slot], (round - 1) & 1)) return false;
            const int n = min(kStageTok, k1 - t0);
            if (lane == 0) mbar_arrive_expect_tx(&full[slot], (part == 0 ? 2u : 1u) * n * S::kRowBytes);
            __syncwarp();
            const int tok = lane & 15;
            if (tok < n && (part == 0 || (part == 1) == (lane < 16))) {
                const int j = s0 + t0 + tok;
                int64_t page = pt[j / a.page_size];
                if (page < 0 || page >= a.num_pages) {   // never read outside the pool
                    raise_error(PA_DEVERR_PAGE_RANGE);
                    page = 0;
                }
                const int64_t row = page * a.page_size + (j % a.page_size);
                const int64_t off = (row * a.num_kv_heads + (int64_t)hg * HPC) * D * EB;
                uint8_t *dst = ring + slot * S::kStageBytes + (lane >> 4) * (kStageTok * S::kRowStride) +
                               tok * S::kRowStride;
                const uint8_t *src = (lane < 16 ? a.k_cache : a.v_cache) + off;
                if (a.evict_first)
                    bulk_g2s_hint(dst, src, S::kRowBytes, &full[slot], policy);
                else
                    bulk_g2s(dst, src, S::kRowBytes, &full[slot]);
            }
        }
    }
    return true;
}

// Consumer warp cw (KV head hg * HPC + cw of each segment) of the same range.
// False on a timeout.
template <int D, int G, int HPC, bool F8, int STAGES = stages_for<D, F8 ? 1 : 2, HPC>()>
__device__ bool decode_consume(const DecodeArgs &a, const int32_t *prefix, int64_t T, int64_t g0,
                               int64_t g1, uint8_t *ring, uint64_t *full, uint64_t *empty, uint16_t *pbuf,
                               int &stage_ctr, int cw, int lane) {
    constexpr int EB = F8 ? 1 : 2;
    using S = DecodeSmem<D, HPC, EB, STAGES>;
    constexpr int kStages = S::kStages;
    const int B = a.num_seqs, HG = a.head_groups;
    // ---------------------------------------------------- consumer warps ----
    // The two contractions of a 16-token stage run on the warp-level tensor
    // path (mma.sync m16n8k16, bf16 inputs, fp32 accumulate), one KV head per
    // warp, its G query heads padded to the 8 columns of the MMA:
    //   S   (16 tokens x 8 heads) = K (16 x d) . Q^T (d x 8)
    //   O^T (d x 8 heads)        += V^T (d x 16 tokens) . P^T (16 x 8)
    // The kernel stays bound by HBM; the tensor path only takes the dot
    // products off the FMA and shuffle pipes.  Fragment coordinates: r8 =
    // lane / 4, q4 = lane % 4; an S fragment holds tokens r8 and r8 + 8 of
    // heads 2*q4 and 2*q4 + 1, an O^T fragment of d-tile mt holds dims
    // 16*mt + r8 (+8) of the same two heads.
    constexpr int KS = D / 16;                       // k-steps of S = d-tiles of O
    const int r8 = lane >> 2, q4 = lane & 3;
    uint16_t *pw = pbuf + cw * 8 * kStageTok;      // P^T as [8 heads][16 tokens] bf16
    // ldmatrix: lane -> one row of one of the four 8x8 matrices
    const int a_tok = (lane & 7) + 8 * ((lane >> 3) & 1), a_dim = 8 * (lane >> 4);   // K (row-major A)
    const int v_tok = (lane & 7) + 8 * (lane >> 4), v_dim = 8 * ((lane >> 3) & 1);   // V (A = V^T)

    SegmentWalk walk{prefix, B, HG, T, g0, g1};
    int b, hg, k0, k1, split, span;
    while (walk.next(b, hg, k0, k1, split, span)) {
        const int kvh = hg * HPC + cw;
        const int h0 = kvh * G;          // first query head of this KV head

        // Q^T fragments of query head h0 + r8 (zero for the padding heads)
        uint32_t qb[KS][2];
        if (F8 && r8 < G) {
            // q * k_scale as f16, k index order 4c, 4c+1 | 4c+2, 4c+3 per 16
            const float ksc = __ldg(a.k_scale + kvh);
            const uint2 *qrow = reinterpret_cast<const uint2 *>(a.q + ((int64_t)b * a.num_q_heads + h0 + r8) * D);
#pragma unroll
            for (int kk = 0; kk < KS; ++kk) {
                const uint2 w = __ldg(qrow + kk * 4 + q4);           // d = 16 kk + 4 q4 .. + 3
                qb[kk][0] = f16x2_bits(__uint_as_float(w.x << 16) * ksc, __uint_as_float(w.x & 0xffff0000u) * ksc);
                qb[kk][1] = f16x2_bits(__uint_as_float(w.y << 16) * ksc, __uint_as_float(w.y & 0xffff0000u) * ksc);
            }
        } else if (r8 < G) {
            const uint32_t *qrow = reinterpret_cast<const uint32_t *>(a.q + ((int64_t)b * a.num_q_heads + h0 + r8) * D);
#pragma unroll
            for (int kk = 0; kk < KS; ++kk) {
                qb[kk][0] = __ldg(qrow + kk * 8 + q4);
                qb[kk][1] = __ldg(qrow + kk * 8 + q4 + 4);
            }
        } else {
#pragma unroll
            for (int kk = 0; kk < KS; ++kk) qb[kk][0] = qb[kk][1] = 0u;
        }
        float oacc[KS][4];
#pragma unroll
        for (int mt = 0; mt < KS; ++mt) oacc[mt][0] = oacc[mt][1] = oacc[mt][2] = oacc[mt][3] = 0.f;
        float m_run[2] = {-INFINITY, -INFINITY};
        float l_run[2] = {0.f, 0.f};

        bool ok = true;
        for (int t0 = k0; t0 < k1; t0 += kStageTok, ++stage_ctr) {
            const int slot = stage_ctr % kStages;
            const int round = stage_ctr / kStages;
            if (!mbar_wait(&full[slot], round & 1)) { ok = false; break; }
            __syncwarp();
            const int n = min(kStageTok, k1 - t0);
            uint8_t *kst = ring + slot * S::kStageBytes + cw * D * EB;
            uint8_t *vst = kst + kStageTok * S::kRowStride;
            if (n < kStageTok) {
                // rows past the last token hold stale shared memory: P is 0
                // there, but 0 * NaN is not, so the V rows are zeroed
                constexpr int kChunks = D * EB / 16;
                for (int i = lane; i < (kStageTok - n) * kChunks; i += 32)
                    *reinterpret_cast<uint4 *>(vst + (n + i / kChunks) * S::kRowStride + (i % kChunks) * 16) =
                        make_uint4(0u, 0u, 0u, 0u);
                __syncwarp();
            }
            const uint32_t ks = smem_u32(kst), vs = smem_u32(vst);

            // ---- S = K Q^T
            float sc[4] = {0.f, 0.f, 0.f, 0.f};
            if constexpr (F8) {
                // one ldmatrix.x4 = two k-steps: matrices (tokens 0-7 | 8-15) x
                // (codes 32 kp .. +15 | 32 kp + 16 .. +31) as b16 pairs.  One
                // chain of MMAs (two chains measured slower here)
#pragma unroll
                for (int kp = 0; kp < KS / 2; ++kp) {
                    uint32_t r[4];
                    ldsm_x4(r, ks + a_tok * S::kRowStride + kp * 32 + a_dim * 2);
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        uint32_t af[4];
                        e4m3x4_to_f16x4(r[2 * h], af[0], af[2]);
                        e4m3x4_to_f16x4(r[2 * h + 1], af[1], af[3]);
                        mma_f16_16816(sc, af, qb[2 * kp + h][0], qb[2 * kp + h][1]);
                    }
                }
            } else {
                // even and odd k-steps in two accumulators: two chains of
                // dependent MMAs half as long, added at the end
                float sc1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int kk = 0; kk < KS; kk += 2) {
                    uint32_t af[4], ag[4];
                    ldsm_x4(af, ks + a_tok * S::kRowStride + (kk * 16 + a_dim) * 2);
                    ldsm_x4(ag, ks + a_tok * S::kRowStride + (kk * 16 + 16 + a_dim) * 2);
                    mma_bf16_16816(sc, af, qb[kk][0], qb[kk][1]);
                    mma_bf16_16816(sc1, ag, qb[kk + 1][0], qb[kk + 1][1]);
                }
#pragma unroll
                for (int i = 0; i < 4; ++i) sc[i] += sc1[i];
            }
            // log2 domain; tokens past n masked
            float x[4];
            x[0] = r8 < n ? sc[0] * a.scale_log2 : -INFINITY;
            x[1] = r8 < n ? sc[1] * a.scale_log2 : -INFINITY;
            x[2] = r8 + 8 < n ? sc[2] * a.scale_log2 : -INFINITY;
            x[3] = r8 + 8 < n ? sc[3] * a.scale_log2 : -INFINITY;

            // ---- online softmax per head over the stage's 16 tokens (lazy
            // rescale: the running maximum moves only by more than 2^8)
            float p[4];
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                float mx = fmaxf(x[j], x[2 + j]);
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
                if (mx > m_run[j] + kLazyRescale) {
                    const float alpha = fast_exp2(m_run[j] - mx);   // 0 when m_run = -inf
                    l_run[j] *= alpha;
#pragma unroll
                    for (int mt = 0; mt < KS; ++mt) {
                        oacc[mt][j] *= alpha;
                        oacc[mt][2 + j] *= alpha;
                    }
                    m_run[j] = mx;
                }
                p[j] = fast_exp2(x[j] - m_run[j]);
                p[2 + j] = fast_exp2(x[2 + j] - m_run[j]);
                l_run[j] += p[j] + p[2 + j];
            }
            // ---- P^T through shared memory into the B-fragment layout
            auto pbits = [](float x) -> uint16_t {
                if constexpr (F8) return __half_as_ushort(__float2half_rn(x));
                else return bf16_bits(x);
            };
            pw[(2 * q4) * kStageTok + r8] = pbits(p[0]);
            pw[(2 * q4 + 1) * kStageTok + r8] = pbits(p[1]);
            pw[(2 * q4) * kStageTok + r8 + 8] = pbits(p[2]);
            pw[(2 * q4 + 1) * kStageTok + r8 + 8] = pbits(p[3]);
            __syncwarp();
            const uint32_t pb0 = *reinterpret_cast<const uint32_t *>(pw + r8 * kStageTok + 2 * q4);
            const uint32_t pb1 = *reinterpret_cast<const uint32_t *>(pw + r8 * kStageTok + 2 * q4 + 8);

            // ---- O^T += V^T P^T
            if constexpr (F8) {
                // transposed b16 pairs: lane (g, c) gets tokens 2c, 2c+1 of
                // codes d = 2g, 2g+1 (bytes t2c.d0 t2c.d1 t2c1.d0 t2c1.d1);
                // a byte permute groups them by d, so one register widens to
                // O^T row 2g (tokens 2c, 2c+1) and the other to row 2g + 1
#pragma unroll
                for (int mp = 0; mp < KS / 2; ++mp) {
                    uint32_t r[4];
                    ldsm_x4_trans(r, vs + a_tok * S::kRowStride + mp * 32 + a_dim * 2);
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const uint32_t p0 = __byte_perm(r[2 * h], 0u, 0x3120);
                        const uint32_t p1 = __byte_perm(r[2 * h + 1], 0u, 0x3120);
                        uint32_t vf[4];
                        e4m3x4_to_f16x4(p0, vf[0], vf[1]);
                        e4m3x4_to_f16x4(p1, vf[2], vf[3]);
                        mma_f16_16816(oacc[2 * mp + h], vf, pb0, pb1);
                    }
                }
            } else {
#pragma unroll
                for (int mt = 0; mt < KS; ++mt) {
                    uint32_t vf[4];
                    ldsm_x4_trans(vf, vs + v_tok * S::kRowStride + (mt * 16 + v_dim) * 2);
                    mma_bf16_16816(oacc[mt], vf, pb0, pb1);
                }
            }
            // the zeroed rows were generic-proxy writes; the next bulk copy
            // into this slot is an async-proxy write
            if (n < kStageTok) fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[slot]);
        }
        if (!ok) return false;

        // ---- finish: l over the stage rows (lanes with equal q4), write
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            float l = l_run[j];
            l += __shfl_xor_sync(0xffffffffu, l, 4);
            l += __shfl_xor_sync(0xffffffffu, l, 8);
            l += __shfl_xor_sync(0xffffffffu, l, 16);
            const int hh = 2 * q4 + j;                   // head within the group
            if (hh >= G) continue;
            const float inv = (l > 0.f ? 1.f / l : 0.f) * (F8 ? __ldg(a.v_scale + kvh) : 1.f);
            const float lse_v = l > 0.f ? (m_run[j] + __log2f(l)) * 0.69314718055994531f : -INFINITY;
            const int h = h0 + hh;
            if (split < 0 || split + span > a.max_splits) {   // cannot happen for valid lengths
                raise_error(PA_DEVERR_SEQLENS);
                continue;
            }
            const int64_t r = ((int64_t)b * a.num_q_heads + h) * a.max_splits + split;
            float *orow = a.o_part + r * D;
#pragma unroll
            for (int mt = 0; mt < KS; ++mt) {
                if constexpr (F8) {          // rows g, g + 8 of the tile are d = 2g, 2g + 1
                    *reinterpret_cast<float2 *>(orow + mt * 16 + 2 * r8) =
                        make_float2(oacc[mt][j] * inv, oacc[mt][2 + j] * inv);
                } else {
                    orow[mt * 16 + r8] = oacc[mt][j] * inv;
                    orow[mt * 16 + r8 + 8] = oacc[mt][2 + j] * inv;
                }
            }
            if (r8 == 0) {
                a.lse_part[r] = lse_v;
                for (int e = 1; e < span; ++e) a.lse_part[r + e] = -INFINITY;   // empty: skipped by the combine
            }
        }
    }
    return true;
}

// Kernel arguments of a validated pa_decode call and its plan (the workspace
// is laid out as [T | pad to 256][length prefix B+1 | pad][O partials][lse
// partials]).
inline DecodeArgs decode_setup(const pa_decode_params &p, const DecodePlan &plan) {
    DecodeArgs a{};
    a.q = static_cast<const __nv_bfloat16 *>(p.q);
    a.k_cache = static_cast<const uint8_t *>(p.k_cache);
    a.v_cache = static_cast<const uint8_t *>(p.v_cache);
    a.page_table = p.page_table;
    a.pt_stride = p.page_table_stride;
    a.cache_seqlens = p.cache_seqlens;
    a.num_seqs = p.num_seqs;
    a.num_q_heads = p.num_q_heads;
    a.num_kv_heads = p.num_kv_heads;
    a.page_size = p.page_size;
    a.num_pages = p.num_pages;
    a.scale_log2 = p.scale * 1.4426950408889634f;
    a.min_split = plan.kv_chunk;
    a.max_seqlen_k = p.max_seqlen_k;
    a.max_splits = plan.max_splits;
    a.head_groups = p.num_kv_heads / plan.heads_per_cta;
    a.out = static_cast<__nv_bfloat16 *>(p.out);
    a.lse = p.lse;
    a.k_scale = p.k_scale;
    a.v_scale = p.v_scale;
    a.window = p.sliding_window;
    a.max_ctas = p.max_ctas;
    a.overlap_previous = p.overlap_previous;
    {
        uint8_t *ws = static_cast<uint8_t *>(p.workspace);
        const size_t rows = (size_t)p.num_seqs * p.num_q_heads * plan.max_splits;
        const size_t pre = (((size_t)p.num_seqs + 1) * sizeof(int32_t) + 255) / 256 * 256;
        const size_t obytes = (rows * p.head_dim * sizeof(float) + 255) / 256 * 256;
        a.ws_header = reinterpret_cast<int32_t *>(ws);
        a.ws_prefix = reinterpret_cast<int32_t *>(ws + 256);
        a.o_part = reinterpret_cast<float *>(ws + 256 + pre);
        a.lse_part = reinterpret_cast<float *>(ws + 256 + pre + obytes);
    }
    return a;
}

}  // namespace
}  // namespace pa
