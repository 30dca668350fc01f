// Split-KV decode attention and the log-sum-exp combine pass.
//
// "Transformer inference kernels: GEMM·Attention·FlashAttention·Fusion
// (3/10)": decode has one query token per sequence and a long cached context
// read through the page table (sections 13-14); several query heads share one
// KV head (section 15); a long key range is cut into splits whose partial
// (m, l, O) are merged by a numerically stable combine (sections 12, 16).
//
// Work decomposition (GB300 design, not the pages'): the work is the list of
// (sequence b, KV-head group hg, token t) rows laid out sequence-major, a
// group being HPC consecutive KV heads (HPC*G query heads).  CTAs are
// persistent and each takes one contiguous, equal-sized range of that list
// (T rows, T a multiple of 16 chosen on the device from the actual lengths,
// never below the host's minimum split), so every CTA streams the same number
// of K/V bytes whatever the length mix.  A range covers one or more row
// segments; each segment yields a partial (O_s, lse_s) for split s = (CTA
// index) - (index of the CTA where its row starts), and a combine pass merges
// them.  CTA 0 publishes T and the length prefix in the workspace header for
// the combine.  Within a CTA:
//   - one producer warp streams 16-token stages into a ring of NST stages:
//     per token one cp.async.bulk of the K row and one of the V row (HPC*d
//     contiguous bf16 each, >= 512 bytes), completion counted on the stage's
//     mbarrier (transaction bytes);
//   - HPC consumer warps, one per KV head.  Per stage a warp computes the
//     16 x G scores and the P.V update with warp-level tensor-core MMAs
//     (mma.sync m16n8k16; the GQA heads fill the MMA's 8 columns), reading K
//     and V with ldmatrix from token rows padded by 16 bytes.  The online
//     softmax runs in the log2 domain and rescales lazily: the running maximum
//     moves only when a stage maximum exceeds it by more than 2^8, which keeps
//     every exponent <= 8 and skips most O rescales exactly.
// The whole kernel is bound by HBM: every K/V byte is read once.
//
// FP8 pools (E4M3 codes with a scale per KV head; the first page lists FP8 /
// quantized KV as a dispatch axis in section 19): the same kernel streams
// rows of one byte per element, half the bytes.  The contractions run in f16
// on the same MMA shape: K and V codes are read with the same ldmatrix
// patterns (pairs of codes as b16), widened exactly to f16 with the
// hardware's E4M3 conversion, and the K scale is folded into the query (q *
// k_scale as f16), the V scale into the final O.  Because an ldmatrix
// register then holds 4 consecutive codes of a row, the k index of the score
// MMA runs over d in the order 4c, 4c+1 | 4c+2, 4c+3 (the query fragment is
// loaded in the same order), and the transposed V fragment holds two
// adjacent d rows, so O^T row g of a d-tile is d = 2g and row g + 8 is
// d = 2g + 1.
#include <cuda_bf16.h>

#include <mutex>

#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {

PA_ERROR_WORD_ACCESSOR(error_word_decode)

namespace {

constexpr int kStageTok = 16;     // tokens per pipeline stage
// Ring depth.  FP8 keeps 3 stages of half-length rows: the smaller ring lets
// 4 CTAs share an SM instead of 2, which measured faster than 6 stages at 2
// CTAs (each CTA's consumers work through one stage at a time).
template <int EB>
constexpr int stages_for() { return EB == 1 ? 3 : 3; }
constexpr int kFp8MaxHeadsPerCta = 4;
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
};

template <int D, int HPC, int EB>
struct DecodeSmem {
    static constexpr int kRowBytes = HPC * D * EB;           // one token, CTA's KV heads (EB bytes each)
    static constexpr int kRowStride = kRowBytes + 16;        // +16 B: ldmatrix rows hit distinct banks
    static constexpr int kStageBytes = 2 * kStageTok * kRowStride;
    static constexpr int kStages = stages_for<EB>();
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

// Two E4M3 codes (low byte first) to two f16 (exact: every E4M3 value is an
// f16 value).
// All four codes of a register (bytes 0-1 and 2-3) to two f16x2 registers,
// the 32-bit register split into its 16-bit halves inside the asm.
__device__ __forceinline__ void e4m3x4_to_f16x4(uint32_t four_codes, uint32_t &lo, uint32_t &hi) {
    asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\t"
        "cvt.rn.f16x2.e4m3x2 %0, l;\n\tcvt.rn.f16x2.e4m3x2 %1, h;\n\t}"
        : "=r"(lo), "=r"(hi) : "r"(four_codes));
}


__device__ __forceinline__ uint32_t f16x2_bits(float lo, float hi) {
    return (uint32_t)__half_as_ushort(__float2half_rn(lo)) | ((uint32_t)__half_as_ushort(__float2half_rn(hi)) << 16);
}

__device__ __forceinline__ uint16_t bf16_bits(float x) {
    return __bfloat16_as_ushort(__float2bfloat16_rn(x));
}

// Walks the segments of one CTA's range [g, g1) of the sequence-major row
// list; pb is the exclusive prefix of the sequence lengths, so sequence b's
// rows start at HG * pb[b] and row (b, hg) at HG * pb[b] + hg * L_b.
struct SegmentWalk {
    const int32_t *pb;
    int B, HG, cta;
    int64_t T, g, g1;
    __device__ bool next(int &b, int &hg, int &t0, int &t1, int &split) {
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
        split = cta - (int)(row_start / T);
        g += t1 - t0;
        return true;
    }
};

template <int D, int G, int HPC, bool F8>
__global__ void __launch_bounds__((HPC + 1) * 32) decode_kernel(const DecodeArgs a) {
    constexpr int EB = F8 ? 1 : 2;                   // bytes per K/V element
    using S = DecodeSmem<D, HPC, EB>;
    extern __shared__ __align__(128) uint8_t smem[];
    uint8_t *ring = smem;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + S::kRingBytes);
    constexpr int kStages = S::kStages;
    uint64_t *empty = full + kStages;
    uint16_t *pbuf = reinterpret_cast<uint16_t *>(empty + kStages);   // [HPC][8 heads][16 tokens] bf16 / f16
    int32_t *prefix = reinterpret_cast<int32_t *>(pbuf + HPC * 8 * kStageTok);  // [B+1]

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int B = a.num_seqs;
    const int HG = a.head_groups;

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
    if (threadIdx.x == 0) {
        prefix[0] = 0;
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], HPC);
        }
        fence_mbar_init();
    }
    __syncthreads();
    if (warp == 0) {
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
    // equal ranges of T rows (a multiple of 16, at least min_split)
    const int64_t total = (int64_t)HG * prefix[B];
    int64_t T = (total + gridDim.x - 1) / gridDim.x;
    T = (T + 15) / 16 * 16;
    if (T < a.min_split) T = a.min_split;
    if (blockIdx.x == 0) {
        for (int b = threadIdx.x; b <= B; b += blockDim.x) a.ws_prefix[b] = prefix[b];
        if (threadIdx.x == 0) a.ws_header[0] = (int32_t)T;
    }
    const int64_t g0 = (int64_t)blockIdx.x * T;
    const int64_t g1 = min(g0 + T, total);

    if (warp == HPC) {
        // ------------------------------------------------ producer warp ----
        int stage_ctr = 0;
        SegmentWalk walk{prefix, B, HG, (int)blockIdx.x, T, g0, g1};
        int b, hg, k0, k1, split;
        while (walk.next(b, hg, k0, k1, split)) {
            const int32_t *pt = a.page_table + (int64_t)b * a.pt_stride;
            // with a sliding window the row's tokens start s0 keys in
            int Lb = a.cache_seqlens[b];
            Lb = Lb < 0 ? 0 : (Lb > a.max_seqlen_k ? a.max_seqlen_k : Lb);
            const int s0 = Lb - (prefix[b + 1] - prefix[b]);
            for (int t0 = k0; t0 < k1; t0 += kStageTok, ++stage_ctr) {
                const int slot = stage_ctr % kStages;
                const int round = stage_ctr / kStages;
                if (round > 0 && !mbar_wait(&empty[slot], (round - 1) & 1)) return;
                const int n = min(kStageTok, k1 - t0);
                if (lane == 0) mbar_arrive_expect_tx(&full[slot], 2u * n * S::kRowBytes);
                __syncwarp();
                const int tok = lane & 15;
                if (tok < n) {
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
                    bulk_g2s(dst, src, S::kRowBytes, &full[slot]);
                }
            }
        }
        return;
    }

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
    uint16_t *pw = pbuf + warp * 8 * kStageTok;      // P^T as [8 heads][16 tokens] bf16
    // ldmatrix: lane -> one row of one of the four 8x8 matrices
    const int a_tok = (lane & 7) + 8 * ((lane >> 3) & 1), a_dim = 8 * (lane >> 4);   // K (row-major A)
    const int v_tok = (lane & 7) + 8 * (lane >> 4), v_dim = 8 * ((lane >> 3) & 1);   // V (A = V^T)
    int stage_ctr = 0;

    SegmentWalk walk{prefix, B, HG, (int)blockIdx.x, T, g0, g1};
    int b, hg, k0, k1, split;
    while (walk.next(b, hg, k0, k1, split)) {
        const int kvh = hg * HPC + warp;
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
            uint8_t *kst = ring + slot * S::kStageBytes + warp * D * EB;
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
        if (!ok) return;

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
            if (split < 0 || split >= a.max_splits) {       // cannot happen for valid lengths
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
            if (r8 == 0) a.lse_part[r] = lse_v;
        }
    }
}

// One warp per row (a (sequence, head) pair): merge its splits by LSE.
template <int D>
__global__ void __launch_bounds__(256) lse_combine_kernel(
    const float *__restrict__ o_part, const float *__restrict__ lse_part,
    const int32_t *__restrict__ splits_per_row, const int32_t *__restrict__ seg_header,
    const int32_t *__restrict__ seg_prefix, int32_t head_groups, int32_t heads_per_group,
    int32_t heads_per_seq, int32_t num_rows, int32_t max_splits,
    __nv_bfloat16 *__restrict__ out, float *__restrict__ lse_out) {
    constexpr int VPL = D / 32;
    const int lane = threadIdx.x & 31;
    const int row = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    // after decode this kernel runs as its programmatic dependent: wait until
    // that grid has completed and its partials are visible (a no-op when
    // launched normally)
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (row >= num_rows) return;
    int n = max_splits;
    if (splits_per_row != nullptr) {
        n = splits_per_row[row];
    } else if (seg_header != nullptr) {
        // decode: the row's splits are the CTA ranges of T rows it overlaps
        const int64_t T = seg_header[0];
        const int b = row / heads_per_seq, hg = (row % heads_per_seq) / heads_per_group;
        const int L = seg_prefix[b + 1] - seg_prefix[b];
        const int64_t rs = (int64_t)head_groups * seg_prefix[b] + (int64_t)hg * L;
        n = L > 0 ? (int)((rs + L - 1) / T - rs / T + 1) : 0;
    }
    n = max(0, min(n, max_splits));
    const float *lrow = lse_part + (int64_t)row * max_splits;
    float M = -INFINITY;
    for (int s = lane; s < n; s += 32) M = fmaxf(M, lrow[s]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    float acc[VPL];
#pragma unroll
    for (int e = 0; e < VPL; ++e) acc[e] = 0.f;
    float den = 0.f;
    if (M != -INFINITY) {
        // four splits at a time: their loads are independent and go out together
        constexpr int U = 4;
        for (int s0 = 0; s0 < n; s0 += U) {
            float ls[U], v[U][VPL];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int s = s0 + u;
                ls[u] = s < n ? lrow[s] : -INFINITY;
                const float *orow = o_part + ((int64_t)row * max_splits + (s < n ? s : 0)) * D + lane * VPL;
                if constexpr (VPL == 4) {
                    const float4 x = *reinterpret_cast<const float4 *>(orow);
                    v[u][0] = x.x; v[u][1] = x.y; v[u][2] = x.z; v[u][3] = x.w;
                } else {
                    const float2 x = *reinterpret_cast<const float2 *>(orow);
                    v[u][0] = x.x; v[u][1] = x.y;
                }
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const float w = (ls[u] == -INFINITY) ? 0.f : __expf(ls[u] - M);
                den += w;
#pragma unroll
                for (int e = 0; e < VPL; ++e) acc[e] += w * v[u][e];
            }
        }
    }
    const float inv = den > 0.f ? 1.f / den : 0.f;
    __nv_bfloat16 *orow = out + (int64_t)row * D + lane * VPL;
    if constexpr (VPL == 4) {
        uint2 w;
        w.x = pack_bf16x2(acc[0] * inv, acc[1] * inv);
        w.y = pack_bf16x2(acc[2] * inv, acc[3] * inv);
        *reinterpret_cast<uint2 *>(orow) = w;
    } else {
        *reinterpret_cast<uint32_t *>(orow) = pack_bf16x2(acc[0] * inv, acc[1] * inv);
    }
    if (lse_out != nullptr && lane == 0) lse_out[row] = den > 0.f ? M + __logf(den) : -INFINITY;
}

template <int D, int G, int HPC, bool F8>
cudaError_t launch_decode_t(const DecodeArgs &a, int64_t items_max, cudaStream_t stream) {
    using S = DecodeSmem<D, HPC, F8 ? 1 : 2>;
    const size_t smem = S::kRingBytes + 2 * S::kStages * sizeof(uint64_t) +
                        HPC * 8 * kStageTok * sizeof(uint16_t) + (a.num_seqs + 1) * sizeof(int32_t);
    auto kern = decode_kernel<D, G, HPC, F8>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, (HPC + 1) * 32, smem);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) return cudaErrorInvalidConfiguration;
    int64_t grid = (int64_t)num_sms() * per_sm;
    if (a.max_ctas > 0 && grid > a.max_ctas) grid = a.max_ctas;
    if (grid > items_max) grid = items_max;
    if (a.overlap_previous) {
        // A programmatic dependent of the previous kernel in the stream: it is
        // scheduled as soon as every CTA of that kernel has signalled (the
        // prefill kernel does so on entry) and never waits for its results.
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)grid);
        cfg.blockDim = dim3((HPC + 1) * 32);
        cfg.dynamicSmemBytes = smem;
        cfg.stream = stream;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        return cudaLaunchKernelEx(&cfg, kern, a);
    }
    kern<<<(unsigned)grid, (HPC + 1) * 32, smem, stream>>>(a);
    return cudaGetLastError();
}

template <int D, int G, bool F8>
cudaError_t dispatch_hpc(const DecodeArgs &a, int hpc, int64_t grid, cudaStream_t s) {
    switch (hpc) {
        case 1: return launch_decode_t<D, G, 1, F8>(a, grid, s);
        case 2: return launch_decode_t<D, G, 2, F8>(a, grid, s);
        case 4: return launch_decode_t<D, G, 4, F8>(a, grid, s);
        case 8:
            if constexpr (F8) return launch_decode_t<D, G, 8, F8>(a, grid, s);
            else return cudaErrorInvalidValue;
        default: return cudaErrorInvalidValue;
    }
}

template <int D, bool F8>
cudaError_t dispatch_g(const DecodeArgs &a, int g, int hpc, int64_t grid, cudaStream_t s) {
    switch (g) {
        case 1: return dispatch_hpc<D, 1, F8>(a, hpc, grid, s);
        case 2: return dispatch_hpc<D, 2, F8>(a, hpc, grid, s);
        case 4: return dispatch_hpc<D, 4, F8>(a, hpc, grid, s);
        case 8: return dispatch_hpc<D, 8, F8>(a, hpc, grid, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

DecodePlan plan_decode(const pa_decode_params &p) {
    DecodePlan plan{};
    // KV heads per CTA: the largest power of two <= 4 dividing Hkv (token
    // rows of 512 B at d = 64, 1 KiB at d = 128; a 3-stage ring of 48 or
    // 96 KiB, so two or more CTAs fit on an SM).
    // FP8 rows are half as long: up to 8 heads, so a copy still moves >= 1 KiB
    // at d = 128.
    const int max_hpc = p.kv_dtype == PA_KV_FP8_E4M3 ? kFp8MaxHeadsPerCta : 4;
    int hpc = 1;
    while (hpc * 2 <= max_hpc && p.num_kv_heads % (hpc * 2) == 0) hpc *= 2;
    plan.heads_per_cta = hpc;
    // Minimum split (the floor of T): the caller's kv_chunk, else 1/32 of the
    // longest context (>= 64 keys).  It bounds the splits of one row by
    // ceil(max_seqlen_k / min_split) + 1 and with it the workspace.
    int32_t chunk = p.kv_chunk;
    if (chunk <= 0) {
        chunk = (p.max_seqlen_k / 32 + 15) / 16 * 16;
        if (chunk < 64) chunk = 64;
    }
    plan.kv_chunk = chunk;
    plan.max_splits = (p.max_seqlen_k + chunk - 1) / chunk + 1;
    const size_t rows = (size_t)p.num_seqs * p.num_q_heads * plan.max_splits;
    const size_t header = 256 + (((size_t)p.num_seqs + 1) * sizeof(int32_t) + 255) / 256 * 256;
    const size_t obytes = (rows * p.head_dim * sizeof(float) + 255) / 256 * 256;
    plan.workspace_bytes = header + obytes + rows * sizeof(float);
    return plan;
}

cudaError_t launch_decode(const pa_decode_params &p, const DecodePlan &plan, cudaStream_t stream) {
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
        // workspace: [T | pad to 256][prefix B+1 | pad][O partials][lse partials]
        uint8_t *ws = static_cast<uint8_t *>(p.workspace);
        const size_t rows = (size_t)p.num_seqs * p.num_q_heads * plan.max_splits;
        const size_t pre = (((size_t)p.num_seqs + 1) * sizeof(int32_t) + 255) / 256 * 256;
        const size_t obytes = (rows * p.head_dim * sizeof(float) + 255) / 256 * 256;
        a.ws_header = reinterpret_cast<int32_t *>(ws);
        a.ws_prefix = reinterpret_cast<int32_t *>(ws + 256);
        a.o_part = reinterpret_cast<float *>(ws + 256 + pre);
        a.lse_part = reinterpret_cast<float *>(ws + 256 + pre + obytes);
    }
    if (p.num_seqs == 0) return cudaSuccess;
    // Upper bound of useful CTAs: every sequence at max length, minimal split.
    const int64_t items_max = ((int64_t)p.num_seqs * p.max_seqlen_k * a.head_groups + plan.kv_chunk - 1) /
                              plan.kv_chunk + 1;
    const int g = p.num_q_heads / p.num_kv_heads;
    const bool f8 = p.kv_dtype == PA_KV_FP8_E4M3;
    cudaError_t e;
    if (f8)
        e = p.head_dim == 64 ? dispatch_g<64, true>(a, g, plan.heads_per_cta, items_max, stream)
                             : dispatch_g<128, true>(a, g, plan.heads_per_cta, items_max, stream);
    else
        e = p.head_dim == 64 ? dispatch_g<64, false>(a, g, plan.heads_per_cta, items_max, stream)
                             : dispatch_g<128, false>(a, g, plan.heads_per_cta, items_max, stream);
    if (e != cudaSuccess) return e;
    return launch_lse_combine(a.o_part, a.lse_part, nullptr, a.ws_header, a.ws_prefix, a.head_groups,
                              g * plan.heads_per_cta, p.num_q_heads, p.num_seqs * p.num_q_heads,
                              plan.max_splits, p.head_dim, p.out, p.lse, stream);
}

cudaError_t launch_lse_combine(const float *o_partial, const float *lse_partial,
                               const int32_t *splits_per_row, const int32_t *seg_header,
                               const int32_t *seg_prefix, int32_t head_groups,
                               int32_t heads_per_group, int32_t heads_per_seq, int32_t num_rows,
                               int32_t max_splits, int32_t head_dim, void *out, float *lse_out,
                               cudaStream_t stream) {
    if (num_rows == 0) return cudaSuccess;
    const int rows_per_block = 8;
    const int blocks = (num_rows + rows_per_block - 1) / rows_per_block;
    auto *o = static_cast<__nv_bfloat16 *>(out);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(blocks);
    cfg.blockDim = dim3(rows_per_block * 32);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    // after the split kernel (seg_header given) the combine is its
    // programmatic dependent: its launch is prepared while the split kernel's
    // last CTAs finish, and griddepcontrol.wait holds it until they have
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = seg_header != nullptr ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (head_dim == 64)
        return cudaLaunchKernelEx(&cfg, lse_combine_kernel<64>, o_partial, lse_partial, splits_per_row,
                                  seg_header, seg_prefix, head_groups, heads_per_group, heads_per_seq,
                                  num_rows, max_splits, o, lse_out);
    return cudaLaunchKernelEx(&cfg, lse_combine_kernel<128>, o_partial, lse_partial, splits_per_row,
                              seg_header, seg_prefix, head_groups, heads_per_group, heads_per_seq,
                              num_rows, max_splits, o, lse_out);
}

// ---------------------------------------------------------------------------
// Scratch for pa_decode_noalloc: a file-scope device array, so a caller that
// cannot allocate device memory still gets split-KV decode.  Every GPU that
// loads this library holds these bytes until the process exits.  Host code
// must not pass the symbol itself to a kernel (on the host it is only a
// stand-in, not a device address): the device address is looked up once per
// device with cudaGetSymbolAddress, with that device current.
static __device__ __align__(256) unsigned char g_decode_noalloc_scratch[kDecodeNoAllocScratchBytes];

cudaError_t decode_noalloc_scratch(void **ptr) {
    static std::mutex lock;
    static void *addr[kMaxDevices] = {nullptr};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lk(lock);
    if (addr[dev] == nullptr) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_decode_noalloc_scratch);
        if (e != cudaSuccess) return e;
        addr[dev] = p;
    }
    *ptr = addr[dev];
    return cudaSuccess;
}

}  // namespace pa
