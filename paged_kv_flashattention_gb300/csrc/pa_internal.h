// Host-side launch functions behind the C ABI (validated arguments only).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "pa.h"

namespace pa {

cudaError_t launch_store_kv(const void *k, const void *v, const int32_t *slot_mapping,
                            int64_t num_tokens, void *k_cache, void *v_cache, int64_t num_slots,
                            int32_t row_bytes, cudaStream_t stream);

cudaError_t launch_store_kv_fp8(const void *k, const void *v, const int32_t *slot_mapping,
                                int64_t num_tokens, void *k_cache, void *v_cache, int64_t num_slots,
                                int32_t num_kv_heads, int32_t head_dim, const float *k_scale,
                                const float *v_scale, cudaStream_t stream);

cudaError_t launch_rope_store(const pa_rope_store_params &p, cudaStream_t stream);

cudaError_t launch_build_page_table(const int32_t *token_table, int64_t tt_stride, int64_t tt_rows,
                                    const int32_t *table_idx, int32_t num_seqs, int32_t ncols,
                                    int32_t page_size, int32_t *page_table, int32_t pt_stride,
                                    cudaStream_t stream);

// Decode plan: keys per split, splits of the longest sequence, KV heads per CTA.
struct DecodePlan {
    int32_t kv_chunk;
    int32_t max_splits;
    int32_t heads_per_cta;
    size_t workspace_bytes;
};
DecodePlan plan_decode(const pa_decode_params &p);
cudaError_t launch_decode(const pa_decode_params &p, const DecodePlan &plan, cudaStream_t stream);

// Merge split partials.  Row r's split count is splits_per_row[r] if given;
// else, with seg_header / seg_prefix (decode), the number of T-row CTA ranges
// its (sequence, head group) rows overlap; else max_splits.
cudaError_t launch_lse_combine(const float *o_partial, const float *lse_partial,
                               const int32_t *splits_per_row, const int32_t *seg_header,
                               const int32_t *seg_prefix, int32_t head_groups,
                               int32_t heads_per_group, int32_t heads_per_seq, int32_t num_rows,
                               int32_t max_splits, int32_t head_dim, void *out, float *lse_out,
                               cudaStream_t stream);

cudaError_t launch_prefill(const pa_prefill_params &p, cudaStream_t stream);
cudaError_t launch_mixed(const pa_prefill_params &pre, const pa_decode_params &dec, cudaStream_t stream);

int num_sms();

// Fixed-size scratch behind pa_decode_noalloc (a file-scope device array in
// decode.cu).  decode_noalloc_scratch returns its device address on the
// current device, looking it up on the first call per device.
constexpr size_t kDecodeNoAllocScratchBytes = size_t(32) << 20;
constexpr int kMaxDevices = 64;
cudaError_t decode_noalloc_scratch(void **ptr);

// Device addresses of each translation unit's error word.
cudaError_t error_word_store(int **addr);
cudaError_t error_word_decode(int **addr);
cudaError_t error_word_prefill(int **addr);
cudaError_t error_word_mixed(int **addr);

}  // namespace pa
