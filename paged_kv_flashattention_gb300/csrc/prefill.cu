// Varlen causal prefill / extend attention: the kernel and its launch (the
// design is described in prefill_impl.cuh).
#include "prefill_impl.cuh"

namespace pa {

PA_ERROR_WORD_ACCESSOR(error_word_prefill)

namespace {

template <int D, int T, bool F8, bool EXT>
__global__ void __launch_bounds__(128 * (T + 1), 1) prefill_kernel(const __grid_constant__ PrefillArgs a) {
    prefill_body<D, T, F8, EXT>(a);
}

template <int D, int T, bool F8, bool EXT>
cudaError_t launch_t(const PrefillArgs &a, dim3 grid, cudaStream_t stream) {
    using S = PrefillSmem<D, T, F8>;
    static_assert(S::kSlots >= 2 && (!F8 || S::kCSlots >= 2), "ring too small");
    // One CTA per SM (it allocates all 512 TMEM columns).
    const int smem = (S::kTotal + 1024) > 120 * 1024 ? (S::kTotal + 1024) : 120 * 1024;
    auto kern = prefill_kernel<D, T, F8, EXT>;
    if (T == 2) {
        static const cudaError_t regs = check_register_split(kern);
        if (regs != cudaSuccess) return regs;
    }
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    kern<<<grid, 128 * (T + 1), smem, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace

template <bool EXT>
cudaError_t dispatch_f8(const PrefillArgs &a, bool f8, int d, int T, dim3 grid, cudaStream_t stream) {
    if (f8) {
        if (d == 128)
            return T == 2 ? launch_t<128, 2, true, EXT>(a, grid, stream) : launch_t<128, 1, true, EXT>(a, grid, stream);
        return T == 2 ? launch_t<64, 2, true, EXT>(a, grid, stream) : launch_t<64, 1, true, EXT>(a, grid, stream);
    }
    if (d == 128)
        return T == 2 ? launch_t<128, 2, false, EXT>(a, grid, stream) : launch_t<128, 1, false, EXT>(a, grid, stream);
    return T == 2 ? launch_t<64, 2, false, EXT>(a, grid, stream) : launch_t<64, 1, false, EXT>(a, grid, stream);
}

cudaError_t launch_prefill(const pa_prefill_params &p, cudaStream_t stream) {
    PrefillArgs a;
    int T = 1;
    cudaError_t e = prefill_setup(p, a, T);
    if (e != cudaSuccess) return e;
    const int64_t virt = a.num_virtual;
    const bool f8 = p.kv_dtype == PA_KV_FP8_E4M3;
    if (virt == 0) return cudaSuccess;
    a.sched = p.scheduler;
    // persistent: one CTA per SM (each holds all 512 TMEM columns)
    int64_t ctas = num_sms();
    if (p.max_ctas > 0 && p.max_ctas < ctas) ctas = p.max_ctas;   // leave SMs to a concurrent launch
    dim3 grid((unsigned)(virt < ctas ? virt : ctas));
    a.num_ctas = (int32_t)grid.x;
    return (a.window > 0 || a.bmask != nullptr) ? dispatch_f8<true>(a, f8, p.head_dim, T, grid, stream)
                                                : dispatch_f8<false>(a, f8, p.head_dim, T, grid, stream);
}

}  // namespace pa
