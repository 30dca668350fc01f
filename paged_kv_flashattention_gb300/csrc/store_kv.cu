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
// Fused RoPE + store: the layer graph's "RoPE + KV cache store" step (same
// page, section 2) in one pass, as the mini-sglang page applies the rotary to
// q and k with the batch positions right before the backend stores K/V.  The
// rotation is the standard rotary embedding driven by a cos/sin table row
// per position (so scaled variants only change the table): a pair (a, b) of
// width-r elements becomes (a cos - b sin, b cos + a sin) in fp32 with
// separately rounded products and sum, rounded to bf16; pairs are (i, i +
// r/2) or (2i, 2i + 1).  The rotated q goes to q_out, the rotated k (bf16)
// and v are stored exactly as pa_store_kv / pa_store_kv_fp8 would store
// them.  One warp per token; a lane handles 16 rotated elements (two 16-byte
// pieces) or 8 copied ones at a time.
//
// Page table: "code-series sgl-project mini-sglang 07", "from ledger to
// tensors": the global table is token granular; a request's row is sliced
// with step page_size up to max_seqlen_k and floor-divided by page_size.
#include <cuda_bf16.h>

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

struct RopeStoreArgs {
    const uint4 *q;
    uint4 *q_out;
    const uint4 *k;
    const uint4 *v;
    const int32_t *positions;
    const float *cos_sin;         // [max_pos, rot_dim]: cos of the rot_dim/2 angles, then sin
    int32_t max_pos;
    int32_t rot_dim;
    int32_t interleaved;
    const int32_t *slot_mapping;
    int64_t num_tokens;
    int32_t num_q_heads;
    int32_t num_kv_heads;
    int32_t head_dim;
    uint8_t *k_cache;
    uint8_t *v_cache;
    int64_t num_slots;
    const float *k_scale;
    const float *v_scale;
};

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }
__device__ __forceinline__ uint32_t bf16_pair(float lo, float hi) {
    return (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(lo)) |
           ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(hi)) << 16);
}

// Rotate 8 pairs held as a[8] (first elements) and b[8] (second elements).
__device__ __forceinline__ void rotate8(float (&a)[8], float (&b)[8], const float *c, const float *s) {
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const float cj = c[j], sj = s[j];
        const float na = __fsub_rn(__fmul_rn(a[j], cj), __fmul_rn(b[j], sj));
        const float nb = __fadd_rn(__fmul_rn(b[j], cj), __fmul_rn(a[j], sj));
        a[j] = na;
        b[j] = nb;
    }
}

__device__ __forceinline__ void unpack8(uint4 x, float (&f)[8]) {
    const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        f[2 * i] = bf16_lo(w[i]);
        f[2 * i + 1] = bf16_hi(w[i]);
    }
}

__device__ __forceinline__ uint4 pack8(const float (&f)[8]) {
    return make_uint4(bf16_pair(f[0], f[1]), bf16_pair(f[2], f[3]), bf16_pair(f[4], f[5]), bf16_pair(f[6], f[7]));
}

// Store 8 bf16 values (as bits) into a pool row piece: bf16 bits, or E4M3 codes.
template <bool F8>
__device__ __forceinline__ void store8(uint8_t *pool, int64_t elem, uint4 bits, float scale) {
    if constexpr (F8) *reinterpret_cast<uint2 *>(pool + elem) = quantize8(bits, scale);
    else *reinterpret_cast<uint4 *>(pool + elem * 2) = bits;
}

template <bool F8>
__global__ void __launch_bounds__(256) rope_store_kernel(const RopeStoreArgs a) {
    const int lane = threadIdx.x & 31;
    const int64_t warps_total = (int64_t)gridDim.x * (blockDim.x >> 5);
    const int D = a.head_dim, r = a.rot_dim, h = r / 2;
    const int Hq = a.num_q_heads, Hkv = a.num_kv_heads;
    const int rot_units = r / 16, copy_units = (D - r) / 8;
    const int units = rot_units + copy_units;            // per head
    for (int64_t t = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); t < a.num_tokens;
         t += warps_total) {
        const int pos = a.positions[t];
        if (pos < 0 || pos >= a.max_pos) {                 // nothing of this token is written
            if (lane == 0) raise_error(PA_DEVERR_POSITION);
            continue;
        }
        const int64_t slot = a.slot_mapping[t];
        const bool store = slot >= 0 && slot < a.num_slots;
        if (slot >= a.num_slots && lane == 0) raise_error(PA_DEVERR_PAGE_RANGE);
        const float *cs = a.cos_sin + (int64_t)pos * r;
        // q heads then k heads, `units` pieces each; (head, piece) of item f
        // advanced incrementally instead of divided out per item
        int hd = lane / units, u = lane % units;
        const int dhd = 32 / units, du = 32 % units;
        for (int f = lane; f < (Hq + Hkv) * units; f += 32) {
            const bool is_q = hd < Hq;
            const int kvh = hd - Hq;
            const uint4 *src = is_q ? a.q + ((t * Hq + hd) * D) / 8 : a.k + ((t * Hkv + kvh) * D) / 8;
            uint4 out0, out1;
            int e0, e1 = -1;                                // element offsets within the head
            if (u < rot_units) {
                float x0[8], x1[8], ra[8], rb[8];
                if (a.interleaved) {                        // elements 16u .. 16u + 15, pairs (2j, 2j+1)
                    e0 = 16 * u;
                    e1 = e0 + 8;
                    unpack8(src[e0 / 8], x0);
                    unpack8(src[e1 / 8], x1);
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        ra[j] = x0[2 * j]; rb[j] = x0[2 * j + 1];
                        ra[4 + j] = x1[2 * j]; rb[4 + j] = x1[2 * j + 1];
                    }
                } else {                                    // elements 8u .. 8u + 7 and h + 8u ..
                    e0 = 8 * u;
                    e1 = h + 8 * u;
                    unpack8(src[e0 / 8], ra);
                    unpack8(src[e1 / 8], rb);
                }
                rotate8(ra, rb, cs + 8 * u, cs + h + 8 * u);
                if (a.interleaved) {
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        x0[2 * j] = ra[j]; x0[2 * j + 1] = rb[j];
                        x1[2 * j] = ra[4 + j]; x1[2 * j + 1] = rb[4 + j];
                    }
                    out0 = pack8(x0);
                    out1 = pack8(x1);
                } else {
                    out0 = pack8(ra);
                    out1 = pack8(rb);
                }
            } else {                                        // past the rotated width: unchanged
                e0 = r + 8 * (u - rot_units);
                out0 = src[e0 / 8];
            }
            if (is_q) {
                uint4 *dst = a.q_out + ((t * Hq + hd) * D) / 8;
                dst[e0 / 8] = out0;
                if (e1 >= 0) dst[e1 / 8] = out1;
            } else if (store) {
                const int64_t row = (slot * Hkv + kvh) * (int64_t)D;
                const float sc = F8 ? __ldg(a.k_scale + kvh) : 1.f;
                store8<F8>(a.k_cache, row + e0, out0, sc);
                if (e1 >= 0) store8<F8>(a.k_cache, row + e1, out1, sc);
            }
            u += du;
            hd += dhd;
            if (u >= units) {
                u -= units;
                ++hd;
            }
        }
        if (store) {                                        // v: copied or quantised
            for (int f = lane; f < Hkv * (D / 8); f += 32) {
                const int kvh = f / (D / 8), c = f % (D / 8);
                const uint4 x = __ldg(a.v + ((t * Hkv + kvh) * D) / 8 + c);
                store8<F8>(a.v_cache, (slot * Hkv + kvh) * (int64_t)D + 8 * c, x, F8 ? __ldg(a.v_scale + kvh) : 1.f);
            }
        }
    }
}

__global__ void build_page_table_kernel(const int32_t *__restrict__ token_table, int64_t tt_stride,
                                        int64_t tt_rows, const int32_t *__restrict__ table_idx,
                                        int32_t num_seqs, int32_t ncols, int32_t page_size,
                                        int32_t *page_table, int32_t pt_stride) {
    const int64_t n = (int64_t)num_seqs * ncols;
    for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < n;
         e += (int64_t)gridDim.x * blockDim.x) {
        const int32_t b = (int32_t)(e / ncols);
        const int32_t c = (int32_t)(e % ncols);
        const int64_t row = table_idx[b];
        if (row < 0 || row >= tt_rows) {     // never read outside the token table
            if (c == 0) raise_error(PA_DEVERR_TABLE_INDEX);
            page_table[(int64_t)b * pt_stride + c] = -1;
            continue;
        }
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

cudaError_t launch_rope_store(const pa_rope_store_params &p, cudaStream_t stream) {
    if (p.num_tokens == 0) return cudaSuccess;
    RopeStoreArgs a{};
    a.q = static_cast<const uint4 *>(p.q);
    a.q_out = static_cast<uint4 *>(p.q_out);
    a.k = static_cast<const uint4 *>(p.k);
    a.v = static_cast<const uint4 *>(p.v);
    a.positions = p.positions;
    a.cos_sin = p.cos_sin;
    a.max_pos = p.max_pos;
    a.rot_dim = p.rot_dim;
    a.interleaved = p.interleaved;
    a.slot_mapping = p.slot_mapping;
    a.num_tokens = p.num_tokens;
    a.num_q_heads = p.num_q_heads;
    a.num_kv_heads = p.num_kv_heads;
    a.head_dim = p.head_dim;
    a.k_cache = static_cast<uint8_t *>(p.k_cache);
    a.v_cache = static_cast<uint8_t *>(p.v_cache);
    a.num_slots = p.num_slots;
    a.k_scale = p.k_scale;
    a.v_scale = p.v_scale;
    const int warps_per_block = 8;
    int64_t blocks = (p.num_tokens + warps_per_block - 1) / warps_per_block;
    const int64_t cap = (int64_t)num_sms() * 16;
    if (blocks > cap) blocks = cap;
    if (p.kv_dtype == PA_KV_FP8_E4M3)
        rope_store_kernel<true><<<(unsigned)blocks, warps_per_block * 32, 0, stream>>>(a);
    else
        rope_store_kernel<false><<<(unsigned)blocks, warps_per_block * 32, 0, stream>>>(a);
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

cudaError_t launch_build_page_table(const int32_t *token_table, int64_t tt_stride, int64_t tt_rows,
                                    const int32_t *table_idx, int32_t num_seqs, int32_t ncols,
                                    int32_t page_size, int32_t *page_table, int32_t pt_stride,
                                    cudaStream_t stream) {
    const int64_t n = (int64_t)num_seqs * ncols;
    if (n == 0) return cudaSuccess;
    int64_t blocks = (n + 255) / 256;
    if (blocks > (int64_t)num_sms() * 8) blocks = (int64_t)num_sms() * 8;
    build_page_table_kernel<<<(unsigned)blocks, 256, 0, stream>>>(
        token_table, tt_stride, tt_rows, table_idx, num_seqs, ncols, page_size, page_table, pt_stride);
    return cudaGetLastError();
}

}  // namespace pa
