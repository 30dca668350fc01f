// KV-cache store (slot_mapping scatter) and the page-table metadata kernel.
//
// Store: "RoPE + KV cache store" of the layer graph in "Transformer inference
// kernels: GEMM·Attention·FlashAttention·Fusion (3/10)", sections 1-2: each
// new token's K and V rows are copied bit for bit to row slot_mapping[t] of
// the pool.  One warp moves one token: K row then V row, 16 bytes per lane
// per step, so a warp's accesses are contiguous 512-byte runs.  The work is
// pure data movement, bounded by HBM (read 2 rows, write 2 rows per token).
//
// FP8 store: the pages list FP8 / quantized KV as a dispatch axis and a KV
// layout (same page, sections 19 and 24) without fixing a format; here an
// element x of KV head h is stored as the E4M3 code nearest x / scale[h]
// (the division correctly rounded in single precision, the conversion the
// hardware's round-to-nearest-even with saturation to +-448).  One warp per
// token as above; a lane converts 8 elements (16 bytes in, 8 bytes out).
//
// Page table: "code-series sgl-project mini-sglang 07", "from ledger to
// tensors": the global table is token granular; a request's row is sliced
// with step page_size up to max_seqlen_k and floor-divided by page_size.
#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {

PA_ERROR_WORD_ACCESSOR(error_word_store)

namespace {

__global__ void __launch_bounds__(256) store_kv_kernel(const uint4 *__restrict__ k,
                                                       const uint4 *__restrict__ v,
                                                       const int32_t *__restrict__ slot_mapping,
                                                       int64_t num_tokens, uint4 *k_cache,
                                                       uint4 *v_cache, int64_t num_slots,
                                                       int32_t row_vecs) {
    const int lane = threadIdx.x & 31;
    const int64_t warps_total = (int64_t)gridDim.x * (blockDim.x >> 5);
    for (int64_t t = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); t < num_tokens;
         t += warps_total) {
        const int64_t slot = slot_mapping[t];
        if (slot < 0) continue;                 // padding token
        if (slot >= num_slots) {                // never write outside the pool
            if (lane == 0) raise_error(PA_DEVERR_PAGE_RANGE);
            continue;
        }
        const uint4 *ks = k + t * row_vecs;
        const uint4 *vs = v + t * row_vecs;
        uint4 *kd = k_cache + slot * row_vecs;
        uint4 *vd = v_cache + slot * row_vecs;
        for (int i = lane; i < row_vecs; i += 32) {
            uint4 a = __ldg(ks + i);
            uint4 b = __ldg(vs + i);
            kd[i] = a;
            vd[i] = b;
        }
    }
}

// Two floats to two E4M3 codes, lo in the low byte (the first operand of the
// conversion lands in the high byte).
__device__ __forceinline__ uint32_t f32x2_to_e4m3x2(float lo, float hi) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

__device__ __forceinline__ uint2 quantize8(uint4 x, float s) {
    const uint32_t w[4] = {x.x, x.y, x.z, x.w};
    uint32_t q[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float lo = __uint_as_float(w[i] << 16), hi = __uint_as_float(w[i] & 0xffff0000u);
        q[i] = f32x2_to_e4m3x2(__fdiv_rn(lo, s), __fdiv_rn(hi, s));
    }
    return make_uint2(q[0] | (q[1] << 16), q[2] | (q[3] << 16));
}

__global__ void __launch_bounds__(256) store_kv_fp8_kernel(const uint4 *__restrict__ k,
                                                           const uint4 *__restrict__ v,
                                                           const int32_t *__restrict__ slot_mapping,
                                                           int64_t num_tokens, uint2 *k_cache,
                                                           uint2 *v_cache, int64_t num_slots,
                                                           int32_t row_groups, int32_t head_dim,
                                                           const float *__restrict__ k_scale,
                                                           const float *__restrict__ v_scale) {
    const int lane = threadIdx.x & 31;
    const int64_t warps_total = (int64_t)gridDim.x * (blockDim.x >> 5);
    for (int64_t t = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); t < num_tokens;
         t += warps_total) {
        const int64_t slot = slot_mapping[t];
        if (slot < 0) continue;                 // padding token
        if (slot >= num_slots) {                // never write outside the pool
            if (lane == 0) raise_error(PA_DEVERR_PAGE_RANGE);
            continue;
        }
        const uint4 *ks = k + t * row_groups;
        const uint4 *vs = v + t * row_groups;
        uint2 *kd = k_cache + slot * row_groups;
        uint2 *vd = v_cache + slot * row_groups;
        for (int i = lane; i < row_groups; i += 32) {
            const int h = (i * 8) / head_dim;   // 8 | head_dim: a group never straddles heads
            kd[i] = quantize8(__ldg(ks + i), __ldg(k_scale + h));
            vd[i] = quantize8(__ldg(vs + i), __ldg(v_scale + h));
        }
    }
}

__global__ void build_page_table_kernel(const int32_t *__restrict__ token_table, int64_t tt_stride,
                                        const int32_t *__restrict__ table_idx, int32_t num_seqs,
                                        int32_t ncols, int32_t page_size, int32_t *page_table,
                                        int32_t pt_stride) {
    const int64_t n = (int64_t)num_seqs * ncols;
    for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < n;
         e += (int64_t)gridDim.x * blockDim.x) {
        const int32_t b = (int32_t)(e / ncols);
        const int32_t c = (int32_t)(e % ncols);
        const int64_t row = table_idx[b];
        const int32_t slot = token_table[row * tt_stride + (int64_t)c * page_size];
        // floor division (slots of real tokens are >= 0)
        int32_t q = slot / page_size;
        if (slot < 0 && q * page_size != slot) q -= 1;
        page_table[(int64_t)b * pt_stride + c] = q;
    }
}

}  // namespace

cudaError_t launch_store_kv_fp8(const void *k, const void *v, const int32_t *slot_mapping,
                                int64_t num_tokens, void *k_cache, void *v_cache, int64_t num_slots,
                                int32_t num_kv_heads, int32_t head_dim, const float *k_scale,
                                const float *v_scale, cudaStream_t stream) {
    if (num_tokens == 0) return cudaSuccess;
    const int warps_per_block = 8;
    int64_t blocks = (num_tokens + warps_per_block - 1) / warps_per_block;
    const int64_t cap = (int64_t)num_sms() * 16;
    if (blocks > cap) blocks = cap;
    store_kv_fp8_kernel<<<(unsigned)blocks, warps_per_block * 32, 0, stream>>>(
        static_cast<const uint4 *>(k), static_cast<const uint4 *>(v), slot_mapping, num_tokens,
        static_cast<uint2 *>(k_cache), static_cast<uint2 *>(v_cache), num_slots,
        num_kv_heads * head_dim / 8, head_dim, k_scale, v_scale);
    return cudaGetLastError();
}

cudaError_t launch_store_kv(const void *k, const void *v, const int32_t *slot_mapping,
                            int64_t num_tokens, void *k_cache, void *v_cache, int64_t num_slots,
                            int32_t row_bytes, cudaStream_t stream) {
    if (num_tokens == 0) return cudaSuccess;
    const int warps_per_block = 8;
    int64_t blocks = (num_tokens + warps_per_block - 1) / warps_per_block;
    const int64_t cap = (int64_t)num_sms() * 16;
    if (blocks > cap) blocks = cap;
    store_kv_kernel<<<(unsigned)blocks, warps_per_block * 32, 0, stream>>>(
        static_cast<const uint4 *>(k), static_cast<const uint4 *>(v), slot_mapping, num_tokens,
        static_cast<uint4 *>(k_cache), static_cast<uint4 *>(v_cache), num_slots, row_bytes / 16);
    return cudaGetLastError();
}

cudaError_t launch_build_page_table(const int32_t *token_table, int64_t tt_stride,
                                    const int32_t *table_idx, int32_t num_seqs, int32_t ncols,
                                    int32_t page_size, int32_t *page_table, int32_t pt_stride,
                                    cudaStream_t stream) {
    const int64_t n = (int64_t)num_seqs * ncols;
    if (n == 0) return cudaSuccess;
    int64_t blocks = (n + 255) / 256;
    if (blocks > (int64_t)num_sms() * 8) blocks = (int64_t)num_sms() * 8;
    build_page_table_kernel<<<(unsigned)blocks, 256, 0, stream>>>(
        token_table, tt_stride, table_idx, num_seqs, ncols, page_size, page_table, pt_stride);
    return cudaGetLastError();
}

}  // namespace pa
