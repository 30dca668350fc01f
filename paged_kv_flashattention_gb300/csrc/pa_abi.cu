// The C ABI of libpa (declared in include/pa.h): argument validation on the
// host, error reporting, and dispatch to the kernels.  Nothing here touches
// device memory except pa_device_error (which reads the error words) and no
// call allocates memory.
#include <cmath>
#include <cuda_runtime.h>

#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "pa.h"
#include "pa_internal.h"

namespace pa {

namespace {
thread_local char g_last_error[512] = "";

pa_status fail(pa_status st, const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_last_error, sizeof g_last_error, fmt, ap);
    va_end(ap);
    return st;
}

pa_status cuda_fail(cudaError_t e, const char *what) {
    return fail(PA_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int g_sms[64] = {0};
std::mutex g_sms_lock;

// Shared checks of the head geometry.
pa_status check_heads(int32_t hq, int32_t hkv, int32_t d, int32_t page_size) {
    if (hq <= 0 || hkv <= 0) return fail(PA_ERR_INVALID, "head counts must be positive (Hq=%d, Hkv=%d)", hq, hkv);
    if (hq % hkv != 0) return fail(PA_ERR_INVALID, "num_q_heads %% num_kv_heads != 0 (Hq=%d, Hkv=%d)", hq, hkv);
    const int g = hq / hkv;
    if (g != 1 && g != 2 && g != 4 && g != 8)
        return fail(PA_ERR_UNSUPPORTED, "GQA group size %d not in {1,2,4,8}", g);
    if (d != 64 && d != 128) return fail(PA_ERR_UNSUPPORTED, "head_dim %d not in {64,128}", d);
    if (page_size != 1 && page_size != 16)
        return fail(PA_ERR_UNSUPPORTED, "page_size %d not in {1,16}", page_size);
    if ((int64_t)hkv * d > 4096) return fail(PA_ERR_UNSUPPORTED, "num_kv_heads * head_dim > 4096");
    return PA_OK;
}
}  // namespace

int num_sms() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 132;
    std::lock_guard<std::mutex> lk(g_sms_lock);
    if (g_sms[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 132;
        g_sms[dev] = n;
    }
    return g_sms[dev];
}

}  // namespace pa

using namespace pa;

extern "C" {

int pa_abi_version(void) { return PA_ABI_VERSION; }

const char *pa_status_string(int status) {
    switch (status) {
        case PA_OK: return "ok";
        case PA_ERR_INVALID: return "invalid argument";
        case PA_ERR_UNSUPPORTED: return "unsupported configuration";
        case PA_ERR_CUDA: return "CUDA error";
        case PA_ERR_DEVICE: return "device-side metadata error";
        default: return "unknown status";
    }
}

const char *pa_last_error(void) { return pa::g_last_error; }

pa_status pa_device_error(int32_t *bits, void *stream) {
    if (bits == nullptr) return fail(PA_ERR_INVALID, "bits is NULL");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t (*getters[])(int **) = {error_word_store, error_word_decode, error_word_prefill, error_word_mixed};
    int32_t acc = 0;
    for (auto get : getters) {
        int *addr = nullptr;
        cudaError_t e = get(&addr);
        if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(error word)");
        int32_t v = 0;
        e = cudaMemcpyAsync(&v, addr, sizeof v, cudaMemcpyDeviceToHost, s);
        if (e == cudaSuccess) e = cudaMemsetAsync(addr, 0, sizeof(int), s);
        if (e == cudaSuccess) e = cudaStreamSynchronize(s);
        if (e != cudaSuccess) return cuda_fail(e, "reading the device error word");
        acc |= v;
    }
    *bits = acc;
    return PA_OK;
}

pa_status pa_store_kv(const void *k, const void *v, const int32_t *slot_mapping, int64_t num_tokens,
                      void *k_cache, void *v_cache, int64_t num_slots, int32_t num_kv_heads,
                      int32_t head_dim, void *stream) {
    g_last_error[0] = 0;
    if (num_tokens < 0 || num_slots < 0) return fail(PA_ERR_INVALID, "negative num_tokens or num_slots");
    if (num_kv_heads <= 0 || head_dim <= 0) return fail(PA_ERR_INVALID, "num_kv_heads and head_dim must be positive");
    const int64_t row_bytes = (int64_t)num_kv_heads * head_dim * 2;
    if (row_bytes % 16 != 0) return fail(PA_ERR_UNSUPPORTED, "K/V row of %lld bytes is not a multiple of 16", (long long)row_bytes);
    if (row_bytes > (1 << 20)) return fail(PA_ERR_UNSUPPORTED, "K/V row too large");
    if (num_tokens == 0) return PA_OK;
    if (!k || !v || !slot_mapping || !k_cache || !v_cache) return fail(PA_ERR_INVALID, "NULL pointer");
    if (!aligned16(k) || !aligned16(v) || !aligned16(k_cache) || !aligned16(v_cache))
        return fail(PA_ERR_INVALID, "K/V pointers must be 16-byte aligned");
    cudaError_t e = launch_store_kv(k, v, slot_mapping, num_tokens, k_cache, v_cache, num_slots,
                                    (int32_t)row_bytes, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? PA_OK : cuda_fail(e, "store_kv launch");
}

pa_status pa_store_kv_fp8(const void *k, const void *v, const int32_t *slot_mapping, int64_t num_tokens,
                          void *k_cache, void *v_cache, int64_t num_slots, int32_t num_kv_heads,
                          int32_t head_dim, const float *k_scale, const float *v_scale, void *stream) {
    g_last_error[0] = 0;
    if (num_tokens < 0 || num_slots < 0) return fail(PA_ERR_INVALID, "negative num_tokens or num_slots");
    if (num_kv_heads <= 0 || head_dim <= 0) return fail(PA_ERR_INVALID, "num_kv_heads and head_dim must be positive");
    if (head_dim % 16 != 0) return fail(PA_ERR_UNSUPPORTED, "head_dim %d is not a multiple of 16", head_dim);
    if ((int64_t)num_kv_heads * head_dim > (1 << 20)) return fail(PA_ERR_UNSUPPORTED, "K/V row too large");
    if (num_tokens == 0) return PA_OK;
    if (!k || !v || !slot_mapping || !k_cache || !v_cache || !k_scale || !v_scale)
        return fail(PA_ERR_INVALID, "NULL pointer");
    if (!aligned16(k) || !aligned16(v) || !aligned16(k_cache) || !aligned16(v_cache))
        return fail(PA_ERR_INVALID, "K/V pointers must be 16-byte aligned");
    cudaError_t e = launch_store_kv_fp8(k, v, slot_mapping, num_tokens, k_cache, v_cache, num_slots,
                                        num_kv_heads, head_dim, k_scale, v_scale,
                                        static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? PA_OK : cuda_fail(e, "store_kv_fp8 launch");
}

pa_status pa_rope_cos_sin_table(float *cos_sin, int32_t max_pos, int32_t rot_dim, double base) {
    g_last_error[0] = 0;
    if (max_pos < 0 || rot_dim <= 0 || rot_dim % 2 != 0) return fail(PA_ERR_INVALID, "max_pos >= 0 and an even rot_dim > 0 are required");
    if (!(base > 0.0) || base != base) return fail(PA_ERR_INVALID, "base must be positive");
    if (max_pos == 0) return PA_OK;
    if (!cos_sin) return fail(PA_ERR_INVALID, "NULL pointer");
    const int h = rot_dim / 2;
    for (int32_t p = 0; p < max_pos; ++p) {
        for (int i = 0; i < h; ++i) {
            const double ang = (double)p * std::pow(base, -2.0 * (double)i / (double)rot_dim);
            cos_sin[(int64_t)p * rot_dim + i] = (float)std::cos(ang);
            cos_sin[(int64_t)p * rot_dim + h + i] = (float)std::sin(ang);
        }
    }
    return PA_OK;
}

pa_status pa_rope_store_kv(const pa_rope_store_params *p, void *stream) {
    g_last_error[0] = 0;
    if (p == nullptr) return fail(PA_ERR_INVALID, "params is NULL");
    if (p->num_tokens < 0 || p->num_slots < 0 || p->max_pos < 0) return fail(PA_ERR_INVALID, "negative sizes");
    if (p->num_q_heads <= 0 || p->num_kv_heads <= 0 || p->head_dim <= 0)
        return fail(PA_ERR_INVALID, "head counts and head_dim must be positive");
    if (p->head_dim % 16 != 0) return fail(PA_ERR_UNSUPPORTED, "head_dim %d is not a multiple of 16", p->head_dim);
    if (p->rot_dim <= 0 || p->rot_dim % 16 != 0 || p->rot_dim > p->head_dim)
        return fail(PA_ERR_UNSUPPORTED, "rot_dim %d must be a positive multiple of 16 <= head_dim", p->rot_dim);
    if (p->interleaved != 0 && p->interleaved != 1) return fail(PA_ERR_INVALID, "interleaved must be 0 or 1");
    if (p->kv_dtype != PA_KV_BF16 && p->kv_dtype != PA_KV_FP8_E4M3)
        return fail(PA_ERR_INVALID, "kv_dtype %d is neither PA_KV_BF16 nor PA_KV_FP8_E4M3", p->kv_dtype);
    if (p->num_tokens == 0) return PA_OK;
    if (!p->q || !p->q_out || !p->k || !p->v || !p->positions || !p->cos_sin || !p->slot_mapping ||
        !p->k_cache || !p->v_cache)
        return fail(PA_ERR_INVALID, "NULL pointer");
    if (p->kv_dtype == PA_KV_FP8_E4M3 && (!p->k_scale || !p->v_scale))
        return fail(PA_ERR_INVALID, "FP8 pools need k_scale and v_scale");
    if (!aligned16(p->q) || !aligned16(p->q_out) || !aligned16(p->k) || !aligned16(p->v) ||
        !aligned16(p->k_cache) || !aligned16(p->v_cache) || !aligned16(p->cos_sin))
        return fail(PA_ERR_INVALID, "q, q_out, k, v, the pools and the table must be 16-byte aligned");
    cudaError_t e = launch_rope_store(*p, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? PA_OK : cuda_fail(e, "rope_store launch");
}

pa_status pa_build_seqlens(const int32_t *cached_len, const int32_t *extend_len, int32_t num_seqs,
                           int32_t *cu_seqlens_q, int32_t *cu_seqlens_k, int32_t *cache_seqlens,
                           int32_t *max_seqlen_q, int32_t *max_seqlen_k) {
    g_last_error[0] = 0;
    if (num_seqs < 0) return fail(PA_ERR_INVALID, "num_seqs < 0");
    if (!cu_seqlens_q || !cu_seqlens_k || !max_seqlen_q || !max_seqlen_k || (num_seqs > 0 && (!cached_len || !extend_len || !cache_seqlens)))
        return fail(PA_ERR_INVALID, "NULL pointer");
    int64_t sq = 0, sk = 0;
    int32_t mq = 0, mk = 0;
    for (int32_t b = 0; b < num_seqs; ++b) {
        if (cached_len[b] < 0 || extend_len[b] < 0) return fail(PA_ERR_INVALID, "negative length at request %d", b);
        const int64_t lk = (int64_t)cached_len[b] + extend_len[b];
        if (lk > INT32_MAX) return fail(PA_ERR_INVALID, "device_len overflows int32 at request %d", b);
        if (extend_len[b] > mq) mq = extend_len[b];
        if (lk > mk) mk = (int32_t)lk;
        sq += extend_len[b];
        sk += lk;
        if (sq > INT32_MAX || sk > INT32_MAX) return fail(PA_ERR_INVALID, "cumulative length overflows int32");
    }
    // write only after validation succeeded
    int64_t aq = 0, ak = 0;
    cu_seqlens_q[0] = 0;
    cu_seqlens_k[0] = 0;
    for (int32_t b = 0; b < num_seqs; ++b) {
        const int32_t lk = cached_len[b] + extend_len[b];
        aq += extend_len[b];
        ak += lk;
        cu_seqlens_q[b + 1] = (int32_t)aq;
        cu_seqlens_k[b + 1] = (int32_t)ak;
        cache_seqlens[b] = lk;
    }
    *max_seqlen_q = mq;
    *max_seqlen_k = mk;
    return PA_OK;
}

pa_status pa_build_page_table(const int32_t *token_table, int64_t token_table_stride,
                              int64_t token_table_rows, const int32_t *table_idx, int32_t num_seqs,
                              int32_t max_seqlen_k, int32_t page_size, int32_t *page_table,
                              int32_t page_table_stride, void *stream) {
    g_last_error[0] = 0;
    if (num_seqs < 0 || max_seqlen_k < 0) return fail(PA_ERR_INVALID, "negative num_seqs or max_seqlen_k");
    if (token_table_rows < 0) return fail(PA_ERR_INVALID, "token_table_rows < 0");
    if (page_size <= 0) return fail(PA_ERR_INVALID, "page_size must be positive");
    const int64_t ncols = ((int64_t)max_seqlen_k + page_size - 1) / page_size;
    if (ncols > page_table_stride) return fail(PA_ERR_INVALID, "page_table_stride %d < %lld columns", page_table_stride, (long long)ncols);
    if ((int64_t)(ncols - 1) * page_size >= token_table_stride && ncols > 0)
        return fail(PA_ERR_INVALID, "token_table_stride %lld too small for max_seqlen_k %d", (long long)token_table_stride, max_seqlen_k);
    if (num_seqs == 0 || ncols == 0) return PA_OK;
    if (!token_table || !table_idx || !page_table) return fail(PA_ERR_INVALID, "NULL pointer");
    cudaError_t e = launch_build_page_table(token_table, token_table_stride, token_table_rows, table_idx, num_seqs,
                                            (int32_t)ncols, page_size, page_table, page_table_stride,
                                            static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? PA_OK : cuda_fail(e, "build_page_table launch");
}

// Validation of a pa_prefill call; *nothing = the call has no query rows
// (then the remaining checks are skipped and nothing is launched).
static pa_status check_prefill(const pa_prefill_params *p, bool *nothing) {
    *nothing = false;
    if (p == nullptr) return fail(PA_ERR_INVALID, "params is NULL");
    pa_status st = check_heads(p->num_q_heads, p->num_kv_heads, p->head_dim, p->page_size);
    if (st != PA_OK) return st;
    if (p->head_dim != 128 && p->head_dim != 64) return fail(PA_ERR_UNSUPPORTED, "prefill head_dim");
    if (p->num_seqs < 0 || p->max_seqlen_q < 0 || p->max_seqlen_k < 0 || p->num_pages <= 0)
        return fail(PA_ERR_INVALID, "negative sizes or empty pool");
    if (p->max_seqlen_q > p->max_seqlen_k && p->max_seqlen_k > 0)
        return fail(PA_ERR_INVALID, "max_seqlen_q %d > max_seqlen_k %d", p->max_seqlen_q, p->max_seqlen_k);
    if (p->causal != 0 && p->causal != 1) return fail(PA_ERR_INVALID, "causal must be 0 or 1");
    // The prefill softmax takes its row maximum over the raw scores, which is
    // the maximum of the scaled scores only for scale > 0 (and 0 * -inf on a
    // masked key would be NaN); decode keeps the same rule.
    if (!(p->scale > 0.f) || p->scale == INFINITY) return fail(PA_ERR_INVALID, "scale must be finite and > 0");
    if (p->total_q < 0) return fail(PA_ERR_INVALID, "total_q < 0");
    if (p->num_seqs == 0 || p->max_seqlen_q == 0 || p->total_q == 0) {
        *nothing = true;
        return PA_OK;
    }
    const int64_t ncols = ((int64_t)p->max_seqlen_k + p->page_size - 1) / p->page_size;
    if (p->page_table_stride < ncols) return fail(PA_ERR_INVALID, "page_table_stride too small for max_seqlen_k");
    if (p->lse != nullptr && p->lse_stride < p->total_q) return fail(PA_ERR_INVALID, "lse_stride < total_q");
    if (!p->q || !p->k_cache || !p->v_cache || !p->page_table || !p->cu_seqlens_q || !p->cu_seqlens_k || !p->out)
        return fail(PA_ERR_INVALID, "NULL pointer");
    if (!aligned16(p->q) || !aligned16(p->k_cache) || !aligned16(p->v_cache) || !aligned16(p->out))
        return fail(PA_ERR_INVALID, "q, caches and out must be 16-byte aligned");
    if (p->lse != nullptr && p->lse_stride <= 0) return fail(PA_ERR_INVALID, "lse_stride must be positive");
    if (p->num_pages > (int64_t)INT32_MAX / p->page_size)
        return fail(PA_ERR_UNSUPPORTED, "pool larger than 2^31 slots");
    if (p->kv_dtype != PA_KV_BF16 && p->kv_dtype != PA_KV_FP8_E4M3)
        return fail(PA_ERR_INVALID, "kv_dtype %d is neither PA_KV_BF16 nor PA_KV_FP8_E4M3", p->kv_dtype);
    if (p->kv_dtype == PA_KV_FP8_E4M3 && (!p->k_scale || !p->v_scale))
        return fail(PA_ERR_INVALID, "FP8 pools need k_scale and v_scale");
    if (p->sliding_window < 0) return fail(PA_ERR_INVALID, "sliding_window must be >= 0");
    if (p->max_ctas < 0) return fail(PA_ERR_INVALID, "max_ctas must be >= 0");
    if (p->scheduler == nullptr) return fail(PA_ERR_INVALID, "scheduler (device int32[2], zero-initialised) is NULL");
    if (p->block_mask != nullptr) {
        const int64_t need_q = ((int64_t)p->max_seqlen_q + PA_MASK_BLOCK - 1) / PA_MASK_BLOCK;
        const int64_t need_k = ((int64_t)p->max_seqlen_k + PA_MASK_BLOCK - 1) / PA_MASK_BLOCK;
        if (p->block_mask_q_blocks < need_q || p->block_mask_k_blocks < need_k || p->block_mask_q_blocks <= 0 ||
            p->block_mask_k_blocks <= 0)
            return fail(PA_ERR_INVALID, "block_mask of %d x %d blocks per request; %lld x %lld needed for max_seqlen_q %d, max_seqlen_k %d",
                        p->block_mask_q_blocks, p->block_mask_k_blocks, (long long)need_q, (long long)need_k,
                        p->max_seqlen_q, p->max_seqlen_k);
    }
    if ((reinterpret_cast<uintptr_t>(p->scheduler) & 7u) != 0) return fail(PA_ERR_INVALID, "scheduler must be 8-byte aligned");
    return PA_OK;
}

pa_status pa_prefill(const pa_prefill_params *p, void *stream) {
    g_last_error[0] = 0;
    bool nothing = false;
    pa_status st = check_prefill(p, &nothing);
    if (st != PA_OK || nothing) return st;
    cudaError_t e = launch_prefill(*p, static_cast<cudaStream_t>(stream));
    if (e == cudaErrorNotSupported) return fail(PA_ERR_UNSUPPORTED, "prefill configuration not supported by this library");
    return e == cudaSuccess ? PA_OK : cuda_fail(e, "prefill launch");
}

static pa_status check_decode(const pa_decode_params *p) {
    if (p == nullptr) return fail(PA_ERR_INVALID, "params is NULL");
    pa_status st = check_heads(p->num_q_heads, p->num_kv_heads, p->head_dim, p->page_size);
    if (st != PA_OK) return st;
    if (p->num_seqs < 0 || p->max_seqlen_k < 0 || p->num_pages <= 0)
        return fail(PA_ERR_INVALID, "negative sizes or empty pool");
    if (p->num_seqs > 16384) return fail(PA_ERR_UNSUPPORTED, "more than 16384 sequences in one decode call");
    if (p->kv_chunk < 0 || p->kv_chunk % 16 != 0) return fail(PA_ERR_INVALID, "kv_chunk must be a non-negative multiple of 16");
    // The prefill softmax takes its row maximum over the raw scores, which is
    // the maximum of the scaled scores only for scale > 0 (and 0 * -inf on a
    // masked key would be NaN); decode keeps the same rule.
    if (!(p->scale > 0.f) || p->scale == INFINITY) return fail(PA_ERR_INVALID, "scale must be finite and > 0");
    if (p->num_pages > (int64_t)INT32_MAX / p->page_size)
        return fail(PA_ERR_UNSUPPORTED, "pool larger than 2^31 slots");
    if (p->kv_dtype != PA_KV_BF16 && p->kv_dtype != PA_KV_FP8_E4M3)
        return fail(PA_ERR_INVALID, "kv_dtype %d is neither PA_KV_BF16 nor PA_KV_FP8_E4M3", p->kv_dtype);
    if (p->kv_dtype == PA_KV_FP8_E4M3 && p->num_seqs > 0 && (!p->k_scale || !p->v_scale))
        return fail(PA_ERR_INVALID, "FP8 pools need k_scale and v_scale");
    if (p->sliding_window < 0) return fail(PA_ERR_INVALID, "sliding_window must be >= 0");
    if (p->max_ctas < 0) return fail(PA_ERR_INVALID, "max_ctas must be >= 0");
    if (p->overlap_previous != 0 && p->overlap_previous != 1) return fail(PA_ERR_INVALID, "overlap_previous must be 0 or 1");
    // The split layout adds up the sequences' (window-clipped) lengths over
    // the KV-head groups in 32-bit integers on the device; sequences that
    // share prefix pages can reach sums beyond that, so bound them here.
    const int64_t eff = (p->sliding_window > 0 && p->sliding_window < p->max_seqlen_k) ? p->sliding_window
                                                                                       : p->max_seqlen_k;
    const int64_t groups = p->num_kv_heads / plan_decode(*p).heads_per_cta;
    if ((int64_t)p->num_seqs * eff * groups > (int64_t)INT32_MAX)
        return fail(PA_ERR_UNSUPPORTED,
                    "num_seqs * max_seqlen_k * KV-head groups = %lld exceeds 2^31 - 1 keys in one decode call",
                    (long long)((int64_t)p->num_seqs * eff * groups));
    return PA_OK;
}

size_t pa_decode_workspace_size(const pa_decode_params *p) {
    if (check_decode(p) != PA_OK) return 0;
    return plan_decode(*p).workspace_bytes;
}

int32_t pa_decode_kv_chunk(const pa_decode_params *p) {
    if (check_decode(p) != PA_OK) return 0;
    return plan_decode(*p).kv_chunk;
}

// The checks pa_decode makes after check_decode for a non-empty batch.
static pa_status check_decode_buffers(const pa_decode_params *p) {
    const int64_t ncols = ((int64_t)p->max_seqlen_k + p->page_size - 1) / p->page_size;
    if (p->page_table_stride < ncols) return fail(PA_ERR_INVALID, "page_table_stride too small for max_seqlen_k");
    if (!p->q || !p->k_cache || !p->v_cache || !p->page_table || !p->cache_seqlens || !p->out)
        return fail(PA_ERR_INVALID, "NULL pointer");
    if (!aligned16(p->q) || !aligned16(p->k_cache) || !aligned16(p->v_cache) || !aligned16(p->out))
        return fail(PA_ERR_INVALID, "q, caches and out must be 16-byte aligned");
    const DecodePlan plan = plan_decode(*p);
    if (plan.workspace_bytes > 0) {
        if (p->workspace == nullptr || p->workspace_bytes < plan.workspace_bytes)
            return fail(PA_ERR_INVALID, "workspace of %zu bytes needed, %zu given", plan.workspace_bytes, p->workspace_bytes);
        if (!aligned16(p->workspace)) return fail(PA_ERR_INVALID, "workspace must be 16-byte aligned");
    }
    return PA_OK;
}

pa_status pa_decode(const pa_decode_params *p, void *stream) {
    g_last_error[0] = 0;
    pa_status st = check_decode(p);
    if (st != PA_OK) return st;
    if (p->num_seqs == 0) return PA_OK;
    st = check_decode_buffers(p);
    if (st != PA_OK) return st;
    const DecodePlan plan = plan_decode(*p);
    cudaError_t e = launch_decode(*p, plan, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? PA_OK : cuda_fail(e, "decode launch");
}

pa_status pa_mixed_batch(const pa_prefill_params *pre, const pa_decode_params *dec, void *stream) {
    g_last_error[0] = 0;
    bool no_prefill = false;
    pa_status st = check_prefill(pre, &no_prefill);
    if (st != PA_OK) return st;
    st = check_decode(dec);
    if (st != PA_OK) return st;
    const bool no_decode = dec->num_seqs == 0;
    // a batch of one kind only is that kind's own launch
    if (no_prefill && no_decode) return PA_OK;
    if (no_prefill) return pa_decode(dec, stream);
    if (no_decode) return pa_prefill(pre, stream);
    st = check_decode_buffers(dec);
    if (st != PA_OK) return st;
    if (pre->k_cache != dec->k_cache || pre->v_cache != dec->v_cache || pre->num_pages != dec->num_pages ||
        pre->page_size != dec->page_size || pre->num_q_heads != dec->num_q_heads ||
        pre->num_kv_heads != dec->num_kv_heads || pre->head_dim != dec->head_dim)
        return fail(PA_ERR_INVALID, "prefill and decode halves must share the pools and the head geometry");
    if (pre->kv_dtype != dec->kv_dtype || (pre->kv_dtype == PA_KV_FP8_E4M3 &&
                                           (pre->k_scale != dec->k_scale || pre->v_scale != dec->v_scale)))
        return fail(PA_ERR_INVALID, "prefill and decode halves must share the pool type and its scales");
    if (pre->sliding_window != 0 || pre->block_mask != nullptr)
        return fail(PA_ERR_UNSUPPORTED, "the mixed-batch launch's prefill half takes no window or block mask");
    if ((pre->num_q_heads / pre->num_kv_heads) % 2 != 0 || pre->num_kv_heads % 4 != 0)
        return fail(PA_ERR_UNSUPPORTED, "the mixed-batch launch needs an even GQA group and num_kv_heads %% 4 == 0");
    if (dec->overlap_previous != 0) return fail(PA_ERR_INVALID, "overlap_previous must be 0 in a mixed-batch launch");
    // the mixed launch splits the decode rows by groups of 4 KV heads, which
    // can outnumber the standalone decode's groups checked above
    if ((int64_t)dec->num_seqs * dec->max_seqlen_k * (dec->num_kv_heads / 4) > INT32_MAX)
        return fail(PA_ERR_UNSUPPORTED, "the mixed-batch decode rows (num_seqs x max_seqlen_k x KV-head groups of 4) "
                                        "exceed 32-bit arithmetic; call pa_prefill and pa_decode");
    cudaError_t e = launch_mixed(*pre, *dec, static_cast<cudaStream_t>(stream));
    if (e == cudaErrorNotSupported) return fail(PA_ERR_UNSUPPORTED, "mixed-batch configuration not supported (too many decode sequences for one CTA's shared memory?)");
    return e == cudaSuccess ? PA_OK : cuda_fail(e, "mixed-batch launch");
}

pa_status pa_decode_noalloc(const pa_decode_params *p, void *stream) {
    g_last_error[0] = 0;
    pa_status st = check_decode(p);
    if (st != PA_OK) return st;
    if (p->num_seqs == 0) return PA_OK;
    const DecodePlan plan = plan_decode(*p);
    if (plan.workspace_bytes > kDecodeNoAllocScratchBytes)
        return fail(PA_ERR_UNSUPPORTED,
                    "pa_decode_noalloc: these sizes need %zu bytes of split scratch, more than its fixed "
                    "%zu bytes; use pa_decode with a caller-allocated workspace, or a larger kv_chunk",
                    plan.workspace_bytes, (size_t)kDecodeNoAllocScratchBytes);
    void *scratch = nullptr;
    if (plan.workspace_bytes > 0) {
        cudaError_t e = decode_noalloc_scratch(&scratch);
        if (e != cudaSuccess) return cuda_fail(e, "pa_decode_noalloc: cudaGetSymbolAddress(scratch)");
    }
    // The existing decode path, with the fixed scratch as its workspace.
    pa_decode_params q = *p;
    q.workspace = scratch;
    q.workspace_bytes = scratch ? kDecodeNoAllocScratchBytes : 0;
    return pa_decode(&q, stream);
}

pa_status pa_lse_combine(const float *o_partial, const float *lse_partial, const int32_t *splits_per_row,
                         int32_t num_rows, int32_t max_splits, int32_t head_dim, void *out, float *lse_out,
                         void *stream) {
    g_last_error[0] = 0;
    if (num_rows < 0 || max_splits < 0) return fail(PA_ERR_INVALID, "negative num_rows or max_splits");
    if (head_dim != 64 && head_dim != 128) return fail(PA_ERR_UNSUPPORTED, "head_dim %d not in {64,128}", head_dim);
    if (num_rows == 0) return PA_OK;
    if (!out || (max_splits > 0 && (!o_partial || !lse_partial))) return fail(PA_ERR_INVALID, "NULL pointer");
    if (!aligned16(o_partial) || !aligned16(out)) return fail(PA_ERR_INVALID, "o_partial and out must be 16-byte aligned");
    cudaError_t e = launch_lse_combine(o_partial, lse_partial, splits_per_row, nullptr, nullptr, 1, 1, 1,
                                       num_rows, max_splits, head_dim, out, lse_out,
                                       static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? PA_OK : cuda_fail(e, "lse_combine launch");
}

}  // extern "C"
