// A mixed continuous batch — prefill / extend requests and decode sequences
// sharing one paged KV pool — in ONE persistent launch ([T] section 13's two
// phases of serving, run together as a serving engine's continuous batch
// does).
//
// The first prefill_ctas CTAs (one CTA per SM; the caller's count, else
// chosen in the kernel from the work of both halves) first run the prefill
// kernel's persistent work loop (prefill_impl.cuh): they take 128-row query
// tiles from the prefill work counter until none are left, drain their
// pipelines and free TMEM.  Every CTA then turns into two decode streams over
// the same shared memory, each two producer warps and four consumer warps
// running the split-KV decode of decode_impl.cuh.  The streams take key
// ranges of the decode batch (equal numbers of (sequence, head group, key)
// rows): each stream of the CTAs without prefill work first walks most of its
// own slice of the rows, and the slices' tails are handed out from a second
// device counter in runs that shrink with the work left.  The CTAs without
// prefill work start on decode at once and the prefill CTAs join as they
// finish, so the tensor-bound prefill runs under the HBM-bound decode read
// and the decode work still spreads over every SM at the end.
// The log-sum-exp combine of the decode partials follows as a second launch
// (a programmatic dependent, as after the decode kernel).
//
// Roles in the decode phase (384 threads): stream 0 = producer warps 8 (it
// takes the key ranges and copies the K rows) and 9 (the V rows), consumers
// 0-3; stream 1 = producer warps 10 and 11, consumers 4-7.  Two producer
// warps per stream: at two streams per SM one warp's copy issue caps the
// rate of 512-byte FP8 rows (about 4.7 TB/s measured with one issuing warp
// per stream).
#include "decode_impl.cuh"
#include "prefill_impl.cuh"

namespace pa {

PA_ERROR_WORD_ACCESSOR(error_word_mixed)

namespace {

constexpr int kMixedHpc = 4;          // KV heads per decode stream
// T-ranges (the split layout's unit) per SM, at most: short ranges let the
// dynamic end of the decode phase balance; T is floored at the caller's
// kv_chunk (the workspace's split bound) in any case.
constexpr int kChunksPerSm = 64;
// Sixteenths of the T-ranges walked as one static run per stream.
constexpr int kStaticSixteenths = 14;

struct MixedArgs {
    int32_t *dsched;                  // caller's [0] next key range, [1] streams finished; 0 between launches
    int32_t num_chunks;               // T = total rows / num_chunks, at least the decode's min_split
    int32_t prefill_ctas;             // CTAs 0 .. prefill_ctas - 1 take prefill items first; 0 = chosen here
};

// The automatic prefill share: the prefill's and the decode's times alone on
// the whole GPU, estimated from their work at rates measured for these
// kernels on GB300 (about 0.9 PFLOP/s for the prefill tiles, 6.9 TB/s for
// the decode rows), give the fraction r of the SMs that finishes the prefill
// when the decode does on the others; a quarter more (plus one CTA) covers
// the prefill's slowdown beside the decode stream, and prefill CTAs that
// finish early join the decode.
constexpr float kPrefillFlopPerNs = 9.0e5f;      // bf16 pools
constexpr float kDecodeBytePerNs = 6.9e3f;
constexpr float kPrefillFlopPerNsFp8 = 8.0e5f;   // FP8 (E4M3) pools
constexpr float kDecodeBytePerNsFp8 = 5.9e3f;
// The automatic count is at most half the grid: CTAs past it start on decode
// without computing it.
constexpr int kAutoPrefillShareMax = 2;

// Called by every thread of a CTA (synchronises the CTA); every CTA reaches
// the same count from the same inputs (fp32 sums in a fixed order).
template <int D, bool F8>
__device__ int auto_prefill_ctas(const PrefillArgs &a, const DecodeArgs &da, float *red) {
    float pairs = 0.f, keys = 0.f;
    for (int b = threadIdx.x; b < a.num_seqs; b += blockDim.x) {
        const float E = (float)(a.cu_q[b + 1] - a.cu_q[b]);
        const float Lk = (float)(a.cu_k[b + 1] - a.cu_k[b]);
        pairs += a.causal ? E * (Lk - E) + E * (E + 1.f) * 0.5f : E * Lk;
    }
    for (int b = threadIdx.x; b < da.num_seqs; b += blockDim.x) {
        int L = da.cache_seqlens[b];
        L = L < 0 ? 0 : (L > da.max_seqlen_k ? da.max_seqlen_k : L);
        if (da.window > 0 && L > da.window) L = da.window;
        keys += (float)L;
    }
    for (int o = 16; o > 0; o >>= 1) {
        pairs += __shfl_xor_sync(0xffffffffu, pairs, o);
        keys += __shfl_xor_sync(0xffffffffu, keys, o);
    }
    const int warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    if ((threadIdx.x & 31) == 0) {
        red[warp] = pairs;
        red[nw + warp] = keys;
    }
    __syncthreads();
    pairs = keys = 0.f;
    for (int w = 0; w < nw; ++w) {       // the same order in every thread and CTA
        pairs += red[w];
        keys += red[nw + w];
    }
    __syncthreads();                      // red is free again
    const float t_pre = pairs * (4.f * D * a.num_q_heads) / (F8 ? kPrefillFlopPerNsFp8 : kPrefillFlopPerNs);
    const float t_dec = keys * ((F8 ? 2.f : 4.f) * D * da.num_kv_heads) / (F8 ? kDecodeBytePerNsFp8 : kDecodeBytePerNs);
    if (!(t_pre > 0.f)) return 0;
    const float r = t_pre / (t_pre + t_dec);
    const int cap = (int)gridDim.x / kAutoPrefillShareMax;
    const int n = (int)ceilf((float)gridDim.x * r * 1.25f) + 1;
    return n < cap ? n : cap;
}

// Shared-memory layout of the decode phase (from offset 0 of the aligned
// dynamic shared memory, below the prefill kernel's barriers, which are not
// reused).
template <int D, bool F8>
struct MixedSmem {
    using DS = DecodeSmem<D, kMixedHpc, F8 ? 1 : 2, 3>;
    static constexpr int kStages = DS::kStages;
    static constexpr int kRing = (DS::kRingBytes + 1023) / 1024 * 1024;
    static constexpr int kBars = 2 * kRing;                           // per stream: full, empty, chunk ring
    static constexpr int kBarsPerStream = 2 * kStages + 4;
    static constexpr int kIdx = kBars + 2 * kBarsPerStream * 8;       // per stream: 2 x (first, end) range
    static constexpr int kPbuf = kIdx + 2 * 2 * 2 * 4;                // per stream: [HPC][8][16] u16
    static constexpr int kPrefix = kPbuf + 2 * kMixedHpc * 8 * kStageTok * 2;
    static int total(int num_seqs) { return kPrefix + (num_seqs + 1) * 4; }
};

template <int D, int G, bool F8>
__global__ void __launch_bounds__(384, 1)
    mixed_kernel(const __grid_constant__ PrefillArgs a, const __grid_constant__ DecodeArgs da, const MixedArgs m) {
    using M = MixedSmem<D, F8>;
    constexpr int EB = F8 ? 1 : 2;
    constexpr int HPC = kMixedHpc;
    constexpr int kStages = M::kStages;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // prefill_ctas: the caller's count, else chosen from the work of both
    // halves by the CTAs that may be among them (the scratch is overwritten
    // by the prefill phase afterwards); with static decode runs every CTA
    // needs the count
    int prefill_ctas = m.prefill_ctas;
    if (prefill_ctas <= 0) {
        const bool candidate = kStaticSixteenths > 0 || (int)blockIdx.x < (int)gridDim.x / kAutoPrefillShareMax;
        prefill_ctas = candidate ? auto_prefill_ctas<D, F8>(a, da, reinterpret_cast<float *>(smem)) : 0;
    }
    if ((int)blockIdx.x < prefill_ctas) {
        prefill_body<D, 2, F8, false>(a, prefill_ctas);   // ends with a CTA-wide barrier; TMEM freed
        // undo the prefill phase's register split: every warp back to the
        // launch's count (the host checked that the kernel was given it)
        if (warp < 8)
            asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kLaunchRegs));
        else
            asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kLaunchRegs));
    }

    // ------------------------------------------------------ decode phase ----
    // the prefill phase's generic shared-memory writes come before the
    // stream producers' bulk copies into the same bytes
    fence_proxy_async_smem();
    if (threadIdx.x == 0) {
        for (int s = 0; s < 2; ++s) {
            uint64_t *bars = reinterpret_cast<uint64_t *>(smem + M::kBars) + s * M::kBarsPerStream;
            for (int i = 0; i < kStages; ++i) {
                mbar_init(&bars[i], 2);                      // stage full (each producer warp's expect-tx)
                mbar_init(&bars[kStages + i], HPC);          // stage empty (one arrive per consumer warp)
            }
            for (int i = 0; i < 2; ++i) {
                mbar_init(&bars[2 * kStages + i], 1);        // key range published
                mbar_init(&bars[2 * kStages + 2 + i], HPC + 1);  // key range read by the consumers and the V producer
            }
        }
        fence_mbar_init();
    }
    int32_t *prefix = reinterpret_cast<int32_t *>(smem + M::kPrefix);
    decode_prefix(da, prefix);                               // synchronises the CTA
    const int B = da.num_seqs;
    const int64_t total = (int64_t)da.head_groups * prefix[B];
    int64_t T = (total + m.num_chunks - 1) / m.num_chunks;   // rows per T-range
    T = (T + 15) / 16 * 16;
    if (T < da.min_split) T = da.min_split;
    const int stream = warp < 8 ? warp >> 2 : (warp - 8) >> 1;   // warps 0-3, 8, 9: 0; 4-7, 10, 11: 1
    // T-ranges [0, N) of the decode rows, cut into one slice of Q ranges per
    // stream of the CTAs without prefill items (of all CTAs when all have
    // some).  Each such stream first walks the first K = 7/8 of its slice:
    // together 7/8 of the work, split equally as the decode kernel splits it.
    // The slices' last R ranges (and the ranges past the last slice) are the
    // pool, taken slice by slice from a counter by whichever stream is free
    // (the prefill CTAs' streams included once their items are done) in runs
    // that shrink with the work left, down to single ranges at the end.  A
    // run that crosses into the next slice's tail is walked as two ranges.  A
    // row thus gets partials only where it crosses a slice's tail.
    const int N = (int)((total + T - 1) / T);
    const int first_static = prefill_ctas < (int)gridDim.x ? prefill_ctas : 0;
    const int n_static = 2 * ((int)gridDim.x - first_static);
    const int Q = N / n_static;
    const int K = Q * kStaticSixteenths / 16;
    const int R = Q - K;
    const int pool = n_static * R + (N - n_static * Q);
    const int my_run = (int)blockIdx.x >= first_static ? 2 * ((int)blockIdx.x - first_static) + stream : -1;

    uint8_t *ring = smem + stream * M::kRing;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + M::kBars) + stream * M::kBarsPerStream;
    uint64_t *full = bars, *empty = bars + kStages, *cfull = bars + 2 * kStages, *cempty = cfull + 2;
    int32_t *cidx = reinterpret_cast<int32_t *>(smem + M::kIdx) + 4 * stream;
    uint16_t *pbuf = reinterpret_cast<uint16_t *>(smem + M::kPbuf) + stream * HPC * 8 * kStageTok;

    if (warp == 8 || warp == 10) {
        // -------------------------------------------- stream producer ----
        if (blockIdx.x == 0 && warp == 8) {   // the combine reads the range layout from the workspace
            for (int b = lane; b <= B; b += 32) da.ws_prefix[b] = prefix[b];
            if (lane == 0) da.ws_header[0] = (int32_t)T;
        }
        // pool index d -> T-range: the tails slice by slice, then the rest
        auto pool_range = [&](int d) { return d < n_static * R ? (d / R) * Q + K + d % R : n_static * Q + (d - n_static * R); };
        int stage_ctr = 0;
        int seen = 0;                                             // the counter as of the last grab
        int rest0 = -1, rest1 = -1;                               // the second part of a run
        for (int n = 0;; ++n) {
            int c0 = -1, c1 = -1;                                 // T-ranges [c0, c1)
            if (n == 0 && my_run >= 0 && K > 0) {
                c0 = my_run * Q;
                c1 = c0 + K;
            } else if (rest0 >= 0) {
                c0 = rest0;
                c1 = rest1;
                rest0 = -1;
            } else {
                const int k = max(1, min(R > 0 ? R : 1, (pool - seen) / (4 * (int)gridDim.x)));
                int d = 0;
                if (lane == 0) d = atomicAdd(&m.dsched[0], k);
                d = __shfl_sync(0xffffffffu, d, 0);
                seen = d + k;
                if (d < pool) {
                    const int e = min(d + k, pool);               // pool indices [d, e)
                    c0 = pool_range(d);
                    // contiguous up to the end of d's tail (or of the pool)
                    int split = e;
                    if (d < n_static * R) split = min(e, (d / R + 1) * R);
                    c1 = pool_range(split - 1) + 1;
                    if (split < e) {
                        rest0 = pool_range(split);
                        rest1 = pool_range(e - 1) + 1;
                    }
                }
            }
            const int slot = n & 1;
            if (n >= 2 && !__all_sync(0xffffffffu, mbar_wait(&cempty[slot], ((n >> 1) - 1) & 1))) break;
            if (lane == 0) {
                cidx[2 * slot] = c0;
                cidx[2 * slot + 1] = c1;
                mbar_arrive(&cfull[slot]);
            }
            if (c0 < 0) break;
            const int64_t g0 = (int64_t)c0 * T, g1 = min((int64_t)c1 * T, total);
            if (!decode_produce<D, HPC, EB, kStages>(da, prefix, T, g0, g1, ring, full, empty, stage_ctr, lane, 1))
                break;
        }
        // the last stream to finish resets the counters for the next launch
        if (lane == 0) {
            __threadfence();
            if (atomicAdd(&m.dsched[1], 1) == 2 * (int)gridDim.x - 1) {
                atomicExch(&m.dsched[0], 0);
                atomicExch(&m.dsched[1], 0);
            }
        }
    } else if (warp == 9 || warp == 11) {
        // ------------------------------ stream V producer (same ranges) ----
        int stage_ctr = 0;
        for (int n = 0;; ++n) {
            const int slot = n & 1;
            if (!__all_sync(0xffffffffu, mbar_wait(&cfull[slot], (n >> 1) & 1))) break;
            const int c0 = cidx[2 * slot], c1 = cidx[2 * slot + 1];
            __syncwarp();
            if (lane == 0) mbar_arrive(&cempty[slot]);
            if (c0 < 0) break;
            const int64_t g0 = (int64_t)c0 * T, g1 = min((int64_t)c1 * T, total);
            if (!decode_produce<D, HPC, EB, kStages>(da, prefix, T, g0, g1, ring, full, empty, stage_ctr, lane, 2))
                break;
        }
    } else if (warp < 8) {
        // -------------------------------------------- stream consumers ----
        const int cw = warp & 3;
        int stage_ctr = 0;
        for (int n = 0;; ++n) {
            const int slot = n & 1;
            if (!__all_sync(0xffffffffu, mbar_wait(&cfull[slot], (n >> 1) & 1))) break;
            const int c0 = cidx[2 * slot], c1 = cidx[2 * slot + 1];
            __syncwarp();
            if (lane == 0) mbar_arrive(&cempty[slot]);
            if (c0 < 0) break;
            const int64_t g0 = (int64_t)c0 * T, g1 = min((int64_t)c1 * T, total);
            if (!decode_consume<D, G, HPC, F8, kStages>(da, prefix, T, g0, g1, ring, full, empty, pbuf, stage_ctr, cw,
                                                 lane))
                break;
        }
    }
    __syncthreads();
}

template <int D, int G, bool F8>
cudaError_t launch_mixed_t(const PrefillArgs &a, const DecodeArgs &da, const MixedArgs &m, int grid,
                           cudaStream_t stream) {
    using PS = PrefillSmem<D, 2, F8>;
    // the decode phase's layout must end below the prefill barriers
    if (MixedSmem<D, F8>::total(da.num_seqs) > PS::kBars) return cudaErrorNotSupported;
    const int smem = PS::kTotal + 1024;
    auto kern = mixed_kernel<D, G, F8>;
    static const cudaError_t regs = check_register_split(kern);
    if (regs != cudaSuccess) return regs;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    kern<<<grid, 384, smem, stream>>>(a, da, m);
    return cudaGetLastError();
}

template <bool F8>
cudaError_t dispatch_mixed(const PrefillArgs &a, const DecodeArgs &da, const MixedArgs &m, int grid, int d, int g,
                           cudaStream_t stream) {
    if (d == 128)
        return g == 2 ? launch_mixed_t<128, 2, F8>(a, da, m, grid, stream)
             : g == 4 ? launch_mixed_t<128, 4, F8>(a, da, m, grid, stream)
                      : launch_mixed_t<128, 8, F8>(a, da, m, grid, stream);
    return g == 2 ? launch_mixed_t<64, 2, F8>(a, da, m, grid, stream)
         : g == 4 ? launch_mixed_t<64, 4, F8>(a, da, m, grid, stream)
                  : launch_mixed_t<64, 8, F8>(a, da, m, grid, stream);
}

}  // namespace

cudaError_t launch_mixed(const pa_prefill_params &pp, const pa_decode_params &dp, cudaStream_t stream) {
    PrefillArgs a;
    int T = 1;
    cudaError_t e = prefill_setup(pp, a, T);
    if (e != cudaSuccess) return e;
    if (T != 2) return cudaErrorNotSupported;
    a.sched = pp.scheduler;
    DecodePlan plan = plan_decode(dp);
    if (dp.num_kv_heads % kMixedHpc != 0) return cudaErrorNotSupported;
    plan.heads_per_cta = kMixedHpc;       // the split layout's head groups of this launch
    DecodeArgs da = decode_setup(dp, plan);
    da.evict_first = 1;
    const int sms = num_sms();
    // Only some CTAs take prefill items first (prefill is tensor-bound,
    // decode HBM-bound: a few SMs of prefill hide under the decode read);
    // the others start on decode key ranges at once.  pre.max_ctas > 0 gives
    // their number; 0 lets every CTA choose the same number from the work of
    // both halves (the prefill scheduler's reset then counts the CTAs the
    // kernel passes to prefill_body: num_ctas = 0).
    const int pre_ctas = pp.max_ctas > 0 ? (pp.max_ctas < sms ? pp.max_ctas : sms) : 0;
    a.num_ctas = 0;
    MixedArgs m{pp.scheduler + 2, kChunksPerSm * sms, pre_ctas};
    const int g = dp.num_q_heads / dp.num_kv_heads;
    e = dp.kv_dtype == PA_KV_FP8_E4M3 ? dispatch_mixed<true>(a, da, m, sms, dp.head_dim, g, stream)
                                      : dispatch_mixed<false>(a, da, m, sms, dp.head_dim, g, stream);
    if (e != cudaSuccess) return e;
    return launch_lse_combine(da.o_part, da.lse_part, nullptr, da.ws_header, da.ws_prefix, da.head_groups,
                              g * plan.heads_per_cta, dp.num_q_heads, dp.num_seqs * dp.num_q_heads,
                              plan.max_splits, dp.head_dim, dp.out, dp.lse, stream);
}

}  // namespace pa
