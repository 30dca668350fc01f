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

#include "decode_impl.cuh"
#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {

PA_ERROR_WORD_ACCESSOR(error_word_decode)

namespace {

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
    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], HPC);
        }
        fence_mbar_init();
    }
    decode_prefix(a, prefix);
    // equal ranges of T rows (a multiple of 16, at least min_split), one per CTA
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
    int stage_ctr = 0;
    if (warp == HPC)
        decode_produce<D, HPC, EB>(a, prefix, T, g0, g1, ring, full, empty, stage_ctr, lane);
    else
        decode_consume<D, G, HPC, F8>(a, prefix, T, g0, g1, ring, full, empty, pbuf, stage_ctr,
                                      warp, lane);
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
    const float *obase = o_part + (int64_t)row * max_splits * D + lane * VPL;
    // The slots are read 128 at a time (four independent loads per lane):
    // first the maximum, then, per group of 128, the weights and a warp ballot
    // of the slots that carry any.  Only their partials are loaded (an empty
    // slot, lse -inf, may have no partial written), 16 independent loads at a
    // time across the group's four 32-slot blocks.
    float M = -INFINITY;
    for (int s0 = 0; s0 < n; s0 += 128) {
#pragma unroll
        for (int b = 0; b < 4; ++b) {
            const int s = s0 + 32 * b + lane;
            if (s < n) M = fmaxf(M, lrow[s]);
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    float acc[VPL];
#pragma unroll
    for (int e = 0; e < VPL; ++e) acc[e] = 0.f;
    float den = 0.f;                       // this lane's slots; summed over the warp below
    if (M != -INFINITY) {
        constexpr int U = 16;
        for (int s0 = 0; s0 < n; s0 += 128) {
            float w[4];
            uint32_t live[4];
#pragma unroll
            for (int b = 0; b < 4; ++b) {
                const int s = s0 + 32 * b + lane;
                const float l = s < n ? lrow[s] : -INFINITY;
                w[b] = l == -INFINITY ? 0.f : __expf(l - M);
                den += w[b];
                live[b] = __ballot_sync(0xffffffffu, w[b] > 0.f);
            }
            while ((live[0] | live[1] | live[2] | live[3]) != 0u) {
                int j[U];
                float wu[U];
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    // the next live slot of the group (the same on every lane)
                    const int b = live[0] ? 0 : live[1] ? 1 : live[2] ? 2 : live[3] ? 3 : -1;
                    if (b < 0) {
                        j[u] = -1;
                        wu[u] = 0.f;
                        continue;
                    }
                    const int bit = __ffs(live[b]) - 1;
                    live[b] &= live[b] - 1u;
                    j[u] = 32 * b + bit;
                    const float wb = b == 0 ? w[0] : b == 1 ? w[1] : b == 2 ? w[2] : w[3];
                    wu[u] = __shfl_sync(0xffffffffu, wb, bit);
                }
                float v[U][VPL];
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    if (j[u] < 0) {
#pragma unroll
                        for (int e = 0; e < VPL; ++e) v[u][e] = 0.f;
                        continue;
                    }
                    const float *orow = obase + (int64_t)(s0 + j[u]) * D;
                    if constexpr (VPL == 4) {
                        const float4 x = *reinterpret_cast<const float4 *>(orow);
                        v[u][0] = x.x; v[u][1] = x.y; v[u][2] = x.z; v[u][3] = x.w;
                    } else {
                        const float2 x = *reinterpret_cast<const float2 *>(orow);
                        v[u][0] = x.x; v[u][1] = x.y;
                    }
                }
#pragma unroll
                for (int u = 0; u < U; ++u)
#pragma unroll
                    for (int e = 0; e < VPL; ++e) acc[e] += wu[u] * v[u][e];
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) den += __shfl_xor_sync(0xffffffffu, den, o);
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
    // FP8 rows are half as long: 8 heads at d = 64 and 4 at d = 128, 512 B
    // either way (fp8_max_heads_per_cta).
    const int max_hpc = p.kv_dtype != PA_KV_FP8_E4M3 ? 4
                      : p.head_dim == 64               ? fp8_max_heads_per_cta<64>()
                                                       : fp8_max_heads_per_cta<128>();
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
    const DecodeArgs a = decode_setup(p, plan);
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
