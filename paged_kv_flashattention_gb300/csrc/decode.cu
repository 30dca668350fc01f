// Split-KV decode attention and the log-sum-exp combine pass.
//
// "Transformer inference kernels: GEMM·Attention·FlashAttention·Fusion
// (3/10)": decode has one query token per sequence and a long cached context
// read through the page table (sections 13-14); several query heads share one
// KV head (section 15); a long key range is cut into splits whose partial
// (m, l, O) are merged by a numerically stable combine (sections 12, 16).
//
// Work decomposition (GB300 design, not the pages'): a work ITEM is
// (sequence b, split s, KV-head group hg): kv_chunk keys of HPC consecutive KV
// heads, i.e. HPC*G query heads.  Each CTA is persistent; it builds the
// compacted item list from cache_seqlens in shared memory (a prefix sum of
// ceil(Lk_b / kv_chunk) per sequence, so no CTA is spent on empty splits) and
// takes items round robin.  Within a CTA:
//   - one producer warp streams 16-token stages into a ring of NST stages:
//     per token one cp.async.bulk of the K row and one of the V row (HPC*d
//     contiguous bf16 each, >= 512 bytes), completion counted on the stage's
//     mbarrier (transaction bytes);
//   - HPC consumer warps, one per KV head.  A warp's lanes form 4 groups of
//     8: group j takes token 4*step + j of the stage, lane i of the group owns
//     16-byte chunks i (and i + 8 for d = 128) of the key row, so each quarter
//     warp reads one contiguous 128-byte line of shared memory.  Dot products
//     for the G query heads use packed f32x2 FMAs (one key value feeds G
//     heads); three xor-shuffles finish each sum.  The online softmax runs in
//     the log2 domain (scale * log2 e folded into q) and rescales lazily: the
//     running maximum moves only when a stage maximum exceeds it by more than
//     2^8, which keeps every exponent <= 8 and skips most O rescales exactly.
//     P.V: each lane owns d/32 consecutive output dims for all G heads; the
//     stage's probabilities are broadcast through a 16 x G float buffer.
// The whole kernel is bound by HBM: every K/V byte is read once.
#include <cuda_bf16.h>

#include <mutex>

#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {

PA_ERROR_WORD_ACCESSOR(error_word_decode)

namespace {

constexpr int kStageTok = 16;     // tokens per pipeline stage
constexpr int kStages = 3;        // ring depth
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
    int32_t kv_chunk;
    int32_t max_splits;
    int32_t head_groups;
    __nv_bfloat16 *out;
    float *lse;
    float *o_part;
    float *lse_part;
};

template <int D, int HPC>
struct DecodeSmem {
    static constexpr int kRowBytes = HPC * D * 2;            // one token, CTA's KV heads
    static constexpr int kStageBytes = 2 * kStageTok * kRowBytes;
    static constexpr int kRingBytes = kStages * kStageBytes;
};

// Locate item -> (b, split, hg) by binary search of the prefix array.
__device__ __forceinline__ void locate_item(const int32_t *prefix, int num_seqs, int item,
                                            int head_groups, int &b, int &split, int &hg) {
    int lo = 0, hi = num_seqs;  // prefix[lo] <= item < prefix[hi]
    while (hi - lo > 1) {
        int mid = (lo + hi) >> 1;
        if (prefix[mid] <= item) lo = mid; else hi = mid;
    }
    b = lo;
    int r = item - prefix[lo];
    split = r / head_groups;
    hg = r % head_groups;
}

template <int D, int G, int HPC>
__global__ void __launch_bounds__((HPC + 1) * 32) decode_kernel(const DecodeArgs a) {
    using S = DecodeSmem<D, HPC>;
    extern __shared__ __align__(128) uint8_t smem[];
    uint8_t *ring = smem;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + S::kRingBytes);
    uint64_t *empty = full + kStages;
    float *pbuf = reinterpret_cast<float *>(empty + kStages);     // [HPC][16][G]
    int32_t *prefix = reinterpret_cast<int32_t *>(pbuf + HPC * kStageTok * G);  // [B+1]

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int B = a.num_seqs;
    const int C = a.kv_chunk;

    // Compacted item list: prefix[b] = sum_{b' < b} n_b * head_groups with
    // n_b = ceil(Lk_b / C) splits (one for an empty sequence, so its output
    // row is still written).  Loaded by all threads, scanned by warp 0.
    for (int b = threadIdx.x; b < B; b += blockDim.x) {
        int L = a.cache_seqlens[b];
        if (L < 0) { raise_error(PA_DEVERR_SEQLENS); L = 0; }
        int n = L > 0 ? (L + C - 1) / C : 1;
        if (n > a.max_splits) { raise_error(PA_DEVERR_SEQLENS); n = a.max_splits; }
        prefix[b + 1] = n * a.head_groups;
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
    const int num_items = prefix[B];

    if (warp == HPC) {
        // ------------------------------------------------ producer warp ----
        int stage_ctr = 0;
        for (int item = blockIdx.x; item < num_items; item += gridDim.x) {
            int b, split, hg;
            locate_item(prefix, B, item, a.head_groups, b, split, hg);
            int Lk = min(a.cache_seqlens[b], a.max_splits * C);
            if (Lk < 0) Lk = 0;
            const int k0 = split * C;
            const int k1 = min(Lk, k0 + C);
            const int32_t *pt = a.page_table + (int64_t)b * a.pt_stride;
            for (int t0 = k0; t0 < k1; t0 += kStageTok, ++stage_ctr) {
                const int slot = stage_ctr % kStages;
                const int round = stage_ctr / kStages;
                if (round > 0 && !mbar_wait(&empty[slot], (round - 1) & 1)) return;
                const int n = min(kStageTok, k1 - t0);
                if (lane == 0) mbar_arrive_expect_tx(&full[slot], 2u * n * S::kRowBytes);
                __syncwarp();
                const int tok = lane & 15;
                if (tok < n) {
                    const int j = t0 + tok;
                    int64_t page = pt[j / a.page_size];
                    if (page < 0 || page >= a.num_pages) {   // never read outside the pool
                        raise_error(PA_DEVERR_PAGE_RANGE);
                        page = 0;
                    }
                    const int64_t row = page * a.page_size + (j % a.page_size);
                    const int64_t off = (row * a.num_kv_heads + (int64_t)hg * HPC) * D * 2;
                    uint8_t *dst = ring + slot * S::kStageBytes + (lane >> 4) * (kStageTok * S::kRowBytes) +
                                   tok * S::kRowBytes;
                    const uint8_t *src = (lane < 16 ? a.k_cache : a.v_cache) + off;
                    bulk_g2s(dst, src, S::kRowBytes, &full[slot]);
                }
            }
        }
        return;
    }

    // ---------------------------------------------------- consumer warps ----
    constexpr int NCH = D / 64;          // 16-byte key chunks per lane
    constexpr int VPL = D / 32;          // output dims per lane
    const int grp = lane >> 3;           // token within a step
    const int sub = lane & 7;            // chunk owner
    float *pw = pbuf + warp * kStageTok * G;
    int stage_ctr = 0;

    for (int item = blockIdx.x; item < num_items; item += gridDim.x) {
        int b, split, hg;
        locate_item(prefix, B, item, a.head_groups, b, split, hg);
        int Lk = min(a.cache_seqlens[b], a.max_splits * C);
        if (Lk < 0) Lk = 0;
        const int k0 = split * C;
        const int k1 = min(Lk, k0 + C);
        const int kvh = hg * HPC + warp;
        const int h0 = kvh * G;          // first query head of this KV head

        // q for the G heads, this lane's chunks, pre-scaled by scale*log2(e)
        float2 qv[G][NCH * 4];
#pragma unroll
        for (int g = 0; g < G; ++g) {
            const uint4 *qrow = reinterpret_cast<const uint4 *>(a.q + ((int64_t)b * a.num_q_heads + h0 + g) * D);
#pragma unroll
            for (int c = 0; c < NCH; ++c) {
                uint4 w = __ldg(qrow + sub + 8 * c);
                const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    qv[g][c * 4 + e] = make_float2(bf16lo(ww[e]) * a.scale_log2, bf16hi(ww[e]) * a.scale_log2);
            }
        }
        float m_run[G], l_run[G];
        float2 o[G][VPL / 2];
#pragma unroll
        for (int g = 0; g < G; ++g) {
            m_run[g] = -INFINITY;
            l_run[g] = 0.f;
#pragma unroll
            for (int e = 0; e < VPL / 2; ++e) o[g][e] = make_float2(0.f, 0.f);
        }

        bool ok = true;
        for (int t0 = k0; t0 < k1; t0 += kStageTok, ++stage_ctr) {
            const int slot = stage_ctr % kStages;
            const int round = stage_ctr / kStages;
            if (!mbar_wait(&full[slot], round & 1)) { ok = false; break; }
            const int n = min(kStageTok, k1 - t0);
            const uint8_t *Ks = ring + slot * S::kStageBytes + warp * D * 2;
            const uint8_t *Vs = Ks + kStageTok * S::kRowBytes;

            // ---- scores s[step][g] for token 4*step + grp (log2 domain)
            float s[4][G];
#pragma unroll
            for (int st = 0; st < 4; ++st) {
                const int t = st * 4 + grp;
                float2 acc[G];
#pragma unroll
                for (int g = 0; g < G; ++g) acc[g] = make_float2(0.f, 0.f);
                if (t < n) {
#pragma unroll
                    for (int c = 0; c < NCH; ++c) {
                        const uint4 w = *reinterpret_cast<const uint4 *>(Ks + t * S::kRowBytes + (sub + 8 * c) * 16);
                        const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const float2 kf = make_float2(bf16lo(ww[e]), bf16hi(ww[e]));
#pragma unroll
                            for (int g = 0; g < G; ++g) acc[g] = ffma2(qv[g][c * 4 + e], kf, acc[g]);
                        }
                    }
                }
#pragma unroll
                for (int g = 0; g < G; ++g) s[st][g] = acc[g].x + acc[g].y;
            }
#pragma unroll
            for (int st = 0; st < 4; ++st)
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    float v = s[st][g];
                    v += __shfl_xor_sync(0xffffffffu, v, 1);
                    v += __shfl_xor_sync(0xffffffffu, v, 2);
                    v += __shfl_xor_sync(0xffffffffu, v, 4);
                    s[st][g] = (st * 4 + grp < n) ? v : -INFINITY;
                }

            // ---- online softmax over the stage (lazy rescale)
#pragma unroll
            for (int g = 0; g < G; ++g) {
                float mx = fmaxf(fmaxf(s[0][g], s[1][g]), fmaxf(s[2][g], s[3][g]));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
                if (mx > m_run[g] + kLazyRescale) {      // warp-uniform decision
                    const float alpha = fast_exp2(m_run[g] - mx);   // 0 when m_run = -inf
                    l_run[g] *= alpha;
#pragma unroll
                    for (int e = 0; e < VPL / 2; ++e) {
                        o[g][e].x *= alpha;
                        o[g][e].y *= alpha;
                    }
                    m_run[g] = mx;
                }
                float psum = 0.f;
#pragma unroll
                for (int st = 0; st < 4; ++st) {
                    const float p = fast_exp2(s[st][g] - m_run[g]);
                    s[st][g] = p;
                    psum += p;
                }
                l_run[g] += psum;
            }
            if (sub == 0) {
#pragma unroll
                for (int st = 0; st < 4; ++st)
#pragma unroll
                    for (int g = 0; g < G; ++g) pw[(st * 4 + grp) * G + g] = s[st][g];
            }
            __syncwarp();

            // ---- O += P V
            for (int t = 0; t < n; ++t) {
                float2 vf[VPL / 2];
                if constexpr (VPL == 4) {
                    const uint2 w = *reinterpret_cast<const uint2 *>(Vs + t * S::kRowBytes + lane * 8);
                    vf[0] = make_float2(bf16lo(w.x), bf16hi(w.x));
                    vf[1] = make_float2(bf16lo(w.y), bf16hi(w.y));
                } else {
                    const uint32_t w = *reinterpret_cast<const uint32_t *>(Vs + t * S::kRowBytes + lane * 4);
                    vf[0] = make_float2(bf16lo(w), bf16hi(w));
                }
                float pv[G];
                if constexpr (G % 4 == 0) {
#pragma unroll
                    for (int g = 0; g < G; g += 4) {
                        const float4 p4 = *reinterpret_cast<const float4 *>(pw + t * G + g);
                        pv[g] = p4.x; pv[g + 1] = p4.y; pv[g + 2] = p4.z; pv[g + 3] = p4.w;
                    }
                } else {
#pragma unroll
                    for (int g = 0; g < G; ++g) pv[g] = pw[t * G + g];
                }
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    const float2 pp = make_float2(pv[g], pv[g]);
#pragma unroll
                    for (int e = 0; e < VPL / 2; ++e) o[g][e] = ffma2(pp, vf[e], o[g][e]);
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[slot]);
        }
        if (!ok) return;

        // ---- finish: l over the four token groups, normalise, write
#pragma unroll
        for (int g = 0; g < G; ++g) {
            float l = l_run[g];
            l += __shfl_xor_sync(0xffffffffu, l, 8);
            l += __shfl_xor_sync(0xffffffffu, l, 16);
            const float inv = l > 0.f ? 1.f / l : 0.f;
            const float lse_v = l > 0.f ? (m_run[g] + __log2f(l)) * 0.69314718055994531f : -INFINITY;
            const int h = h0 + g;
            if (a.max_splits == 1) {
                __nv_bfloat16 *orow = a.out + ((int64_t)b * a.num_q_heads + h) * D + lane * VPL;
                if constexpr (VPL == 4) {
                    uint2 w;
                    w.x = pack_bf16x2(o[g][0].x * inv, o[g][0].y * inv);
                    w.y = pack_bf16x2(o[g][1].x * inv, o[g][1].y * inv);
                    *reinterpret_cast<uint2 *>(orow) = w;
                } else {
                    *reinterpret_cast<uint32_t *>(orow) = pack_bf16x2(o[g][0].x * inv, o[g][0].y * inv);
                }
                if (a.lse != nullptr && lane == 0) a.lse[(int64_t)b * a.num_q_heads + h] = lse_v;
            } else {
                const int64_t r = ((int64_t)b * a.num_q_heads + h) * a.max_splits + split;
                float *orow = a.o_part + r * D + lane * VPL;
                if constexpr (VPL == 4) {
                    *reinterpret_cast<float4 *>(orow) =
                        make_float4(o[g][0].x * inv, o[g][0].y * inv, o[g][1].x * inv, o[g][1].y * inv);
                } else {
                    *reinterpret_cast<float2 *>(orow) = make_float2(o[g][0].x * inv, o[g][0].y * inv);
                }
                if (lane == 0) a.lse_part[r] = lse_v;
            }
        }
    }
}

// One warp per row (a (sequence, head) pair): merge its splits by LSE.
template <int D>
__global__ void __launch_bounds__(256) lse_combine_kernel(
    const float *__restrict__ o_part, const float *__restrict__ lse_part,
    const int32_t *__restrict__ splits_per_row, const int32_t *__restrict__ cache_seqlens,
    int32_t kv_chunk, int32_t heads_per_seq, int32_t num_rows, int32_t max_splits,
    __nv_bfloat16 *__restrict__ out, float *__restrict__ lse_out) {
    constexpr int VPL = D / 32;
    const int lane = threadIdx.x & 31;
    const int row = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (row >= num_rows) return;
    int n = max_splits;
    if (splits_per_row != nullptr) {
        n = splits_per_row[row];
    } else if (cache_seqlens != nullptr) {
        const int L = cache_seqlens[row / heads_per_seq];
        n = L > 0 ? (L + kv_chunk - 1) / kv_chunk : 0;
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
        for (int s = 0; s < n; ++s) {
            const float ls = lrow[s];
            const float w = (ls == -INFINITY) ? 0.f : __expf(ls - M);
            den += w;
            const float *orow = o_part + ((int64_t)row * max_splits + s) * D + lane * VPL;
            if constexpr (VPL == 4) {
                const float4 v = *reinterpret_cast<const float4 *>(orow);
                acc[0] += w * v.x; acc[1] += w * v.y; acc[2] += w * v.z; acc[3] += w * v.w;
            } else {
                const float2 v = *reinterpret_cast<const float2 *>(orow);
                acc[0] += w * v.x; acc[1] += w * v.y;
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

template <int D, int G, int HPC>
cudaError_t launch_decode_t(const DecodeArgs &a, int64_t items_max, cudaStream_t stream) {
    using S = DecodeSmem<D, HPC>;
    const size_t smem = S::kRingBytes + 2 * kStages * sizeof(uint64_t) +
                        HPC * kStageTok * G * sizeof(float) + (a.num_seqs + 1) * sizeof(int32_t);
    auto kern = decode_kernel<D, G, HPC>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, (HPC + 1) * 32, smem);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) return cudaErrorInvalidConfiguration;
    int64_t grid = (int64_t)num_sms() * per_sm;
    if (grid > items_max) grid = items_max;
    kern<<<(unsigned)grid, (HPC + 1) * 32, smem, stream>>>(a);
    return cudaGetLastError();
}

template <int D, int G>
cudaError_t dispatch_hpc(const DecodeArgs &a, int hpc, int64_t grid, cudaStream_t s) {
    switch (hpc) {
        case 1: return launch_decode_t<D, G, 1>(a, grid, s);
        case 2: return launch_decode_t<D, G, 2>(a, grid, s);
        case 4: return launch_decode_t<D, G, 4>(a, grid, s);
        default: return cudaErrorInvalidValue;
    }
}

template <int D>
cudaError_t dispatch_g(const DecodeArgs &a, int g, int hpc, int64_t grid, cudaStream_t s) {
    switch (g) {
        case 1: return dispatch_hpc<D, 1>(a, hpc, grid, s);
        case 2: return dispatch_hpc<D, 2>(a, hpc, grid, s);
        case 4: return dispatch_hpc<D, 4>(a, hpc, grid, s);
        case 8: return dispatch_hpc<D, 8>(a, hpc, grid, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

DecodePlan plan_decode(const pa_decode_params &p) {
    DecodePlan plan{};
    // KV heads per CTA: the largest power of two <= 4 dividing Hkv (token
    // rows of 512 B at d = 64, 1 KiB at d = 128; a 3-stage ring of 48 or
    // 96 KiB, so two or more CTAs fit on an SM).
    int hpc = 1;
    while (hpc * 2 <= 4 && p.num_kv_heads % (hpc * 2) == 0) hpc *= 2;
    plan.heads_per_cta = hpc;
    int32_t chunk = p.kv_chunk;
    if (chunk <= 0) {
        // about 16 splits for the longest sequence, 128..1024 keys each
        chunk = (p.max_seqlen_k / 16 + 15) / 16 * 16;
        if (chunk < 128) chunk = 128;
        if (chunk > 1024) chunk = 1024;
    }
    plan.kv_chunk = chunk;
    plan.max_splits = p.max_seqlen_k > 0 ? (p.max_seqlen_k + chunk - 1) / chunk : 1;
    if (plan.max_splits <= 1) {
        plan.max_splits = 1;
        plan.workspace_bytes = 0;
    } else {
        const size_t rows = (size_t)p.num_seqs * p.num_q_heads * plan.max_splits;
        const size_t obytes = rows * p.head_dim * sizeof(float);
        plan.workspace_bytes = ((obytes + 255) / 256) * 256 + rows * sizeof(float);
    }
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
    a.kv_chunk = plan.kv_chunk;
    a.max_splits = plan.max_splits;
    a.head_groups = p.num_kv_heads / plan.heads_per_cta;
    a.out = static_cast<__nv_bfloat16 *>(p.out);
    a.lse = p.lse;
    if (plan.max_splits > 1) {
        const size_t rows = (size_t)p.num_seqs * p.num_q_heads * plan.max_splits;
        const size_t obytes = ((rows * p.head_dim * sizeof(float) + 255) / 256) * 256;
        a.o_part = static_cast<float *>(p.workspace);
        a.lse_part = reinterpret_cast<float *>(static_cast<uint8_t *>(p.workspace) + obytes);
    }
    if (p.num_seqs == 0) return cudaSuccess;
    // Upper bound of items: every sequence at max length.
    const int64_t items_max = (int64_t)p.num_seqs * plan.max_splits * a.head_groups;
    const int g = p.num_q_heads / p.num_kv_heads;
    cudaError_t e = p.head_dim == 64 ? dispatch_g<64>(a, g, plan.heads_per_cta, items_max, stream)
                                     : dispatch_g<128>(a, g, plan.heads_per_cta, items_max, stream);
    if (e != cudaSuccess || plan.max_splits == 1) return e;
    return launch_lse_combine(a.o_part, a.lse_part, nullptr, p.cache_seqlens, plan.kv_chunk,
                              p.num_q_heads, p.num_seqs * p.num_q_heads, plan.max_splits,
                              p.head_dim, p.out, p.lse, stream);
}

cudaError_t launch_lse_combine(const float *o_partial, const float *lse_partial,
                               const int32_t *splits_per_row, const int32_t *cache_seqlens,
                               int32_t kv_chunk, int32_t heads_per_seq, int32_t num_rows,
                               int32_t max_splits, int32_t head_dim, void *out, float *lse_out,
                               cudaStream_t stream) {
    if (num_rows == 0) return cudaSuccess;
    const int rows_per_block = 8;
    const int blocks = (num_rows + rows_per_block - 1) / rows_per_block;
    auto *o = static_cast<__nv_bfloat16 *>(out);
    if (head_dim == 64)
        lse_combine_kernel<64><<<blocks, rows_per_block * 32, 0, stream>>>(
            o_partial, lse_partial, splits_per_row, cache_seqlens, kv_chunk, heads_per_seq,
            num_rows, max_splits, o, lse_out);
    else
        lse_combine_kernel<128><<<blocks, rows_per_block * 32, 0, stream>>>(
            o_partial, lse_partial, splits_per_row, cache_seqlens, kv_chunk, heads_per_seq,
            num_rows, max_splits, o, lse_out);
    return cudaGetLastError();
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
