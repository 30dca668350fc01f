/*
 * pa.h - C ABI of the paged-KV attention library (libpa.so, sm_103a).
 *
 * Exact attention over a paged KV cache, as a serving engine runs it:
 *   pa_store_kv          write the new tokens' K/V rows into the paged pool
 *   pa_store_kv_fp8      the same into an FP8 (E4M3) pool with per-head scales
 *   pa_rope_store_kv     rotary embedding of q and k fused with the K/V store
 *   pa_rope_cos_sin_table  the rotary cos/sin table (host)
 *   pa_build_seqlens     per-request boundaries from the three lengths (host)
 *   pa_build_page_table  per-request page table from the token-granular table
 *   pa_prefill           varlen causal prefill / extend attention
 *   pa_decode            one-query-per-sequence split-KV decode attention
 *   pa_decode_noalloc    the same, with fixed library-owned split scratch
 *   pa_mixed_batch       a continuous batch (prefill + decode) in one launch
 *   pa_lse_combine       merge of split partial results by log-sum-exp
 *
 * Sources (web pages; section names as printed on them):
 *  [T] "Transformer inference kernels: GEMM·Attention·FlashAttention·Fusion
 *      (3/10)": s.1-2 layer graph (RoPE + KV cache store, then attention),
 *      s.10 scaled dot-product attention, s.11 tiled exact attention, s.12
 *      online softmax, s.13 prefill vs decode, s.14 paged-KV address
 *      translation, s.15 GQA head mapping, s.16 split-KV with stable merge,
 *      s.19 dispatch axes (FP8 / quantized KV), s.24 edge-case matrix.
 *  [M] "code-series sgl-project mini-sglang 07": "from ledger to tensors"
 *      (extend_len / device_len / cached_len, cu_seqlens_q, cu_seqlens_k,
 *      cache_seqlens, the page-size-1 global table sliced with step P and
 *      floor-divided by P), "the layer does not know the backend" (q viewed
 *      as [-1, Hq, d]).
 *
 * Conventions shared by every call
 *  - bf16 tensors are IEEE bfloat16; all metadata is int32; device offsets
 *    are computed in 64 bits (pools larger than 2^31 bytes are fine).
 *  - KV pool layout (K and V alike): [num_pages, page_size, Hkv, d], row
 *    major.  The physical row of logical key j of request b is
 *    page_table[b * page_table_stride + j / page_size] * page_size
 *    + j % page_size  ([T] s.14).  With page_size 1 the table holds slots.
 *  - GQA: query head h reads KV head h / (Hq / Hkv)  ([T] s.15).
 *  - Causal masks are aligned to the END of each request's keys: query i of
 *    a request with Lq queries and Lk keys sees keys 0 .. Lk - Lq + i
 *    (cached prefix, then the extend tokens; [M]).
 *  - A query row that sees no key yields O = 0 and lse = -inf.
 *  - Masks: causal (end-aligned), sliding window, and for pa_prefill a
 *    block-sparse mask over 128 x 128 blocks (pa_prefill_params.block_mask).
 *  - Supported: head_dim 64 or 128; page_size 1 or 16; Hq % Hkv == 0 with
 *    group size Hq / Hkv in {1, 2, 4, 8}; Hkv * head_dim <= 4096.
 *  - Every device pointer must be 16-byte aligned.  The library allocates
 *    no memory: the caller owns every buffer, including the decode workspace.
 *  - Calls are asynchronous on the given CUDA stream (a cudaStream_t passed
 *    as void*; NULL = legacy default stream) and never synchronise it.
 *  - Errors: arguments are validated on the host before any launch; a
 *    rejected call launches nothing and returns PA_ERR_INVALID or
 *    PA_ERR_UNSUPPORTED.  A failed launch returns PA_ERR_CUDA.  The text of
 *    the last failure on the calling thread is pa_last_error().  Values that
 *    live on the device (page ids, slots, cu_seqlens) cannot be checked
 *    before launch; kernels skip any access outside the pool and raise the
 *    device error word instead, which pa_device_error() reads.  There is no
 *    fallback path of any kind.
 */
#ifndef PA_H
#define PA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define PA_ABI_VERSION 3

typedef enum {
    PA_OK = 0,
    PA_ERR_INVALID = 1,      /* malformed arguments */
    PA_ERR_UNSUPPORTED = 2,  /* well-formed but outside the supported set */
    PA_ERR_CUDA = 3,         /* a CUDA runtime/driver call failed */
    PA_ERR_DEVICE = 4        /* a kernel flagged bad device-side metadata */
} pa_status;

/* Device error bits (pa_device_error). */
#define PA_DEVERR_PAGE_RANGE 1   /* a page id / slot outside the pool was skipped */
#define PA_DEVERR_SEQLENS 2      /* cu_seqlens / cache_seqlens inconsistent */
#define PA_DEVERR_TIMEOUT 4      /* a bounded wait in a kernel gave up */
#define PA_DEVERR_POSITION 8     /* a RoPE position outside the cos/sin table */
#define PA_DEVERR_TABLE_INDEX 16 /* a table_idx entry outside the token table's rows */

int pa_abi_version(void);
const char *pa_status_string(int status);
/* Message of the last failed call on this thread ("" if none). */
const char *pa_last_error(void);

/* Read and clear the device error word of the current device.  Synchronises
 * `stream` first.  *bits receives an OR of PA_DEVERR_* (0 = clean). */
pa_status pa_device_error(int32_t *bits, void *stream);

/* Element type of the K/V pools read by pa_prefill and pa_decode.  FP8 pools hold E4M3
 * codes written by pa_store_kv_fp8 with per-KV-head scales.  On FP8 pools the
 * contractions run in f16 with fp32 accumulation: q * k_scale is rounded to
 * f16 (|q * k_scale| must stay below 65504), P is rounded to f16. */
typedef enum { PA_KV_BF16 = 0, PA_KV_FP8_E4M3 = 1 } pa_kv_dtype;

/*
 * pa_store_kv - KV-cache store ([T] s.1-2, "RoPE + KV cache store"):
 *   for t in [0, num_tokens): s = slot_mapping[t];
 *     if s >= 0: k_cache_row[s] = k[t]; v_cache_row[s] = v[t]   (bit copy)
 * k, v:          device bf16 [num_tokens, Hkv, head_dim]
 * slot_mapping:  device int32 [num_tokens]; slot = page * page_size + offset;
 *                a negative slot marks a padding token and is skipped;
 *                a slot >= num_slots is skipped and raises PA_DEVERR_PAGE_RANGE.
 *                Two tokens with the same slot are a caller error.
 * k_cache, v_cache: device bf16 [num_slots, Hkv, head_dim] (a pool
 *                [num_pages, page_size, Hkv, d] has num_slots = pages * size).
 */
pa_status pa_store_kv(const void *k, const void *v, const int32_t *slot_mapping,
                      int64_t num_tokens, void *k_cache, void *v_cache, int64_t num_slots,
                      int32_t num_kv_heads, int32_t head_dim, void *stream);

/*
 * pa_store_kv_fp8 - KV-cache store into an FP8 pool ([T] s.19 and s.24 name
 * FP8 / quantized KV without fixing a format; this library's reading):
 *   for t with s = slot_mapping[t] >= 0, head h, element c:
 *     k_cache[s, h, c] = E4M3(k[t, h, c] / k_scale[h])   (same for v)
 * E4M3: 1 sign, 4 exponent (bias 7) and 3 mantissa bits, no infinities,
 * largest finite value 448; the quotient is an IEEE single division, rounded
 * to the nearest E4M3 value (ties to even), magnitudes >= 448 saturate to
 * +-448.  Attention reads the element back as value(code) * scale[h].
 * k, v:             device bf16 [num_tokens, Hkv, head_dim]
 * k_cache, v_cache: device uint8 codes [num_slots, Hkv, head_dim]
 * k_scale, v_scale: device fp32 [Hkv], positive and finite
 * slot_mapping: as for pa_store_kv.  head_dim must be a multiple of 16.
 */
pa_status pa_store_kv_fp8(const void *k, const void *v, const int32_t *slot_mapping,
                          int64_t num_tokens, void *k_cache, void *v_cache, int64_t num_slots,
                          int32_t num_kv_heads, int32_t head_dim, const float *k_scale,
                          const float *v_scale, void *stream);

/*
 * pa_rope_cos_sin_table - rotary table on the HOST ([T] s.2 "RoPE + KV cache
 * store"; the pages do not define the rotation, this library's reading is
 * the standard rotary embedding): for p < max_pos and i < rot_dim / 2,
 *   cos_sin[p * rot_dim + i]               = cos(p * base^(-2i / rot_dim))
 *   cos_sin[p * rot_dim + rot_dim / 2 + i] = sin(p * base^(-2i / rot_dim))
 * computed in double and rounded to float.  cos_sin: host fp32
 * [max_pos, rot_dim], owned by the caller (copy it to the device once).
 * Scaled variants are other tables of the same shape.
 */
pa_status pa_rope_cos_sin_table(float *cos_sin, int32_t max_pos, int32_t rot_dim, double base);

/*
 * pa_rope_store_kv - rotary embedding of q and k fused with the K/V store
 * ([T] s.2: "RoPE + KV cache store" as one step after the QKV projection;
 * [M]: the rotary is applied with the batch positions just before the
 * attention backend stores K/V).  For token t at position pos = positions[t]
 * and every pair (i, i + rot_dim/2) (or (2i, 2i+1) when interleaved) of the
 * first rot_dim elements of each q and k head, with c, s the table's entries
 * for pair i:  (a, b) -> (a*c - b*s, b*c + a*s), each product and the sum
 * rounded in fp32, the result rounded to bf16; elements past rot_dim are
 * copied.  Rotated q goes to q_out (which may be q itself); rotated k and v
 * are stored to row slot_mapping[t] exactly as pa_store_kv (bf16 pools) or
 * pa_store_kv_fp8 (FP8 pools, from the bf16 rotated k) store them; a
 * negative slot stores nothing (q is still rotated).  A position outside
 * [0, max_pos) writes nothing for that token and raises PA_DEVERR_POSITION.
 */
typedef struct {
    const void *q;               /* bf16 [num_tokens, Hq, head_dim] */
    void *q_out;                 /* bf16 [num_tokens, Hq, head_dim]; may equal q */
    const void *k;               /* bf16 [num_tokens, Hkv, head_dim] (not modified) */
    const void *v;               /* bf16 [num_tokens, Hkv, head_dim] */
    const int32_t *positions;    /* device int32 [num_tokens] */
    const float *cos_sin;        /* device fp32 [max_pos, rot_dim] (pa_rope_cos_sin_table layout) */
    int32_t max_pos;
    int32_t rot_dim;             /* multiple of 16, <= head_dim */
    int32_t interleaved;         /* 0: pairs (i, i + rot_dim/2); 1: pairs (2i, 2i+1) */
    const int32_t *slot_mapping; /* device int32 [num_tokens], as for pa_store_kv */
    int64_t num_tokens;
    int32_t num_q_heads;
    int32_t num_kv_heads;
    int32_t head_dim;            /* multiple of 16 */
    void *k_cache;               /* [num_slots, Hkv, head_dim] bf16, or E4M3 codes */
    void *v_cache;
    int64_t num_slots;
    int32_t kv_dtype;            /* pa_kv_dtype of the pools */
    const float *k_scale;        /* FP8 pools: device fp32 [Hkv] */
    const float *v_scale;
} pa_rope_store_params;

pa_status pa_rope_store_kv(const pa_rope_store_params *p, void *stream);

/*
 * pa_build_seqlens - host-side metadata ([M], "from ledger to tensors").
 * All pointers are HOST memory.  From cached_len[b] and extend_len[b]:
 *   cu_seqlens_q  [num_seqs+1] = exclusive prefix sum of extend_len
 *   cu_seqlens_k  [num_seqs+1] = exclusive prefix sum of device_len
 *   cache_seqlens [num_seqs]   = device_len = cached_len + extend_len
 *   *max_seqlen_q, *max_seqlen_k = the maxima.
 * Negative lengths or sums beyond INT32_MAX are PA_ERR_INVALID.
 */
pa_status pa_build_seqlens(const int32_t *cached_len, const int32_t *extend_len,
                           int32_t num_seqs, int32_t *cu_seqlens_q, int32_t *cu_seqlens_k,
                           int32_t *cache_seqlens, int32_t *max_seqlen_q,
                           int32_t *max_seqlen_k);

/*
 * pa_build_page_table - device-side metadata ([M]): the global table is token
 * granular (page size 1, one slot per position); request b's row
 * token_table[table_idx[b], :] is sliced with step page_size up to
 * max_seqlen_k and floor-divided by page_size:
 *   page_table[b * page_table_stride + c] =
 *       floor(token_table[table_idx[b] * token_table_stride + c * page_size] / page_size)
 *   for c < ceil(max_seqlen_k / page_size).
 * token_table, table_idx, page_table: device int32; token_table holds
 * token_table_rows rows.  Columns at and beyond ceil(max_seqlen_k /
 * page_size) are not written.  A table_idx entry outside [0,
 * token_table_rows) (device data: checked in the kernel) writes -1 across its
 * row, which the attention kernels skip as a page outside the pool, and
 * raises PA_DEVERR_TABLE_INDEX.
 */
pa_status pa_build_page_table(const int32_t *token_table, int64_t token_table_stride,
                              int64_t token_table_rows, const int32_t *table_idx, int32_t num_seqs,
                              int32_t max_seqlen_k, int32_t page_size, int32_t *page_table,
                              int32_t page_table_stride, void *stream);


/*
 * pa_prefill - varlen prefill / extend attention ([T] s.10-15, [M]).
 * For request b: Lq = cu_seqlens_q[b+1] - cu_seqlens_q[b] queries (the extend
 * tokens, rows cu_seqlens_q[b].. of q and out), Lk = cu_seqlens_k[b+1] -
 * cu_seqlens_k[b] keys read through page_table row b (Lk >= Lq unless Lk = 0).
 *   out[t, h, :] = softmax_j(scale * q[t,h,:] . K_j) V_j over the visible keys,
 *   lse[h * lse_stride + t] = ln sum_j exp(scale * q . K_j)   (optional)
 * The score matrix never leaves the chip (tiled, online softmax; [T] s.11-12).
 * max_seqlen_q / max_seqlen_k must bound every request's Lq / Lk.
 * Work is handed to persistent CTAs by two device counters in the caller's
 * `scheduler` array (PA_PREFILL_SCHEDULER_INTS int32, zero before its first
 * use; every launch that completes leaves them at zero again, so one array
 * serves any number of calls that run one after the other, e.g. on one
 * stream or in one captured graph).  Launches that may run at the same time
 * (calls on different streams, graph replays beside other prefill work) each
 * need their own array: two launches sharing one would skip or repeat work
 * items.  After a launch that raised PA_DEVERR_TIMEOUT the counters may be
 * left non-zero: clear the array before using it again.
 */
#define PA_PREFILL_SCHEDULER_INTS 2
typedef struct {
    const void *q;               /* bf16 [total_q, Hq, d] */
    const void *k_cache;         /* bf16 [num_pages, page_size, Hkv, d] */
    const void *v_cache;
    const int32_t *page_table;   /* int32 [num_seqs, page_table_stride] */
    int32_t page_table_stride;
    int32_t total_q;             /* rows of q and out (>= cu_seqlens_q[num_seqs]) */
    const int32_t *cu_seqlens_q; /* int32 [num_seqs + 1] */
    const int32_t *cu_seqlens_k; /* int32 [num_seqs + 1] */
    int32_t num_seqs;
    int32_t max_seqlen_q;
    int32_t max_seqlen_k;
    int32_t num_q_heads;
    int32_t num_kv_heads;
    int32_t head_dim;
    int32_t page_size;
    int64_t num_pages;
    int32_t causal;              /* 0 or 1 */
    float scale;                 /* finite and > 0, usually 1/sqrt(head_dim) */
    void *out;                   /* bf16 [total_q, Hq, d] */
    float *lse;                  /* optional fp32 [Hq, lse_stride]; NULL = not written */
    int64_t lse_stride;          /* >= total_q when lse != NULL */
    int32_t kv_dtype;            /* pa_kv_dtype of k_cache / v_cache (0 = bf16) */
    const float *k_scale;        /* PA_KV_FP8_E4M3: device fp32 [Hkv]; else unused */
    const float *v_scale;
    int32_t sliding_window;      /* 0 = none; W > 0: a query at position p sees only keys
                                    j >= p - (W - 1) ([T] s.19 "sliding window" mask) */
    int32_t max_ctas;            /* 0 = one persistent CTA per SM; n > 0: at most n CTAs
                                    (each holds a whole SM), leaving the other SMs to a
                                    concurrent launch, e.g. pa_decode on another stream */
    int32_t *scheduler;          /* device int32 [PA_PREFILL_SCHEDULER_INTS], owned by the
                                    caller: zero before its first use, left zero by every
                                    completed launch; required (NULL = PA_ERR_INVALID) */
    const uint8_t *block_mask;   /* optional block-sparse mask ([T] s.19 "custom sparse";
                                    the pages give no format, this library's reading):
                                    device bytes [num_seqs, block_mask_q_blocks,
                                    block_mask_k_blocks] over blocks of
                                    PA_MASK_BLOCK = 128 query rows x 128 keys; query row i
                                    of request b (i counted from the request's first row,
                                    0 .. Lq - 1) sees key j only if
                                    block_mask[b][i / 128][j / 128] != 0, on top of the
                                    causal and window limits.  Blocks that are zero are
                                    skipped (no load, no MMA).  NULL = no mask. */
    int32_t block_mask_q_blocks; /* >= ceil(max_seqlen_q / 128) when block_mask is set */
    int32_t block_mask_k_blocks; /* >= ceil(max_seqlen_k / 128) when block_mask is set */
} pa_prefill_params;
#define PA_MASK_BLOCK 128

pa_status pa_prefill(const pa_prefill_params *p, void *stream);

/*
 * pa_decode - decode attention ([T] s.13 and s.16): one query token per
 * sequence (q row b) attends to all cache_seqlens[b] keys of its page-table
 * row (the new token already stored).  Work is balanced by keys, not by
 * sequences: the batch's (sequence, head group, key) list is cut into equal
 * ranges, one per resident CTA, and each range is never shorter than
 * kv_chunk keys.  A sequence that spans several ranges gets one partial
 * (O_s, lse_s) per range in the workspace; a second, log-sum-exp combine
 * launch merges them into `out` (it always runs; a row with one partial is
 * copied).  The combine is launched as a programmatic dependent of the split
 * kernel: its launch is prepared while the split kernel finishes, and it
 * waits for that grid's completion before it reads a partial.  The split layout depends only on the device-side cache_seqlens,
 * so it is the same on every call with the same lengths (run-to-run
 * deterministic).
 */
typedef struct {
    const void *q;               /* bf16 [num_seqs, Hq, d] */
    const void *k_cache;         /* bf16 [num_pages, page_size, Hkv, d] */
    const void *v_cache;
    const int32_t *page_table;   /* int32 [num_seqs, page_table_stride] */
    int32_t page_table_stride;
    const int32_t *cache_seqlens;/* int32 [num_seqs] */
    int32_t num_seqs;
    int32_t max_seqlen_k;        /* >= every cache_seqlens[b] */
    int32_t num_q_heads;
    int32_t num_kv_heads;
    int32_t head_dim;
    int32_t page_size;
    int64_t num_pages;
    float scale;                 /* finite and > 0 */
    void *out;                   /* bf16 [num_seqs, Hq, d] */
    float *lse;                  /* optional fp32 [num_seqs, Hq]; NULL = not written */
    void *workspace;             /* device, >= pa_decode_workspace_size(p) bytes */
    size_t workspace_bytes;
    int32_t kv_chunk;            /* minimum keys per split, multiple of 16;
                                    0 = automatic (max_seqlen_k / 32, >= 64) */
    int32_t kv_dtype;            /* pa_kv_dtype of k_cache / v_cache (0 = bf16) */
    const float *k_scale;        /* PA_KV_FP8_E4M3: device fp32 [Hkv]; else unused */
    const float *v_scale;        /* (element = value(code) * scale[kv head]) */
    int32_t sliding_window;      /* 0 = none; W > 0: only the last W keys of each sequence
                                    are read and attended to */
    int32_t max_ctas;            /* 0 = every resident CTA slot; n > 0: at most n CTAs */
    int32_t overlap_previous;    /* 1: the split kernel may start while the previous kernel
                                    in the stream still runs (a programmatic dependent: it
                                    starts once every CTA of that kernel has signalled, as
                                    pa_prefill's do on entry).  Only valid when this decode
                                    reads nothing that kernel writes and that kernel does
                                    not use this workspace; with max_ctas on both
                                    calls, prefill and decode then share the SMs.  0 = no. */
} pa_decode_params;

/* Bytes of workspace pa_decode needs for these parameters (always > 0: a
 * header, a length prefix, and partials for at most
 * ceil(max_seqlen_k / kv_chunk) + 1 splits per (sequence, head)).  Reads
 * only host fields of *p. */
size_t pa_decode_workspace_size(const pa_decode_params *p);
/* The minimum split pa_decode will use for these parameters. */
int32_t pa_decode_kv_chunk(const pa_decode_params *p);

pa_status pa_decode(const pa_decode_params *p, void *stream);

/*
 * pa_mixed_batch - one continuous batch of a serving engine ([T] s.13: the
 * prefill and decode phases; [M] runs them as one batch): the prefill /
 * extend requests of `pre` and the decode sequences of `dec`, over the SAME
 * pools, in one persistent launch (plus the decode combine as a dependent
 * second launch).  The first n CTAs (one CTA per SM) take prefill work
 * items first; every CTA takes decode key ranges once it has no prefill
 * work, so CTAs without prefill work start on decode at once and the
 * tensor-bound prefill runs under the HBM-bound decode read.  n =
 * pre->max_ctas when > 0 (at most the SM count); 0 = chosen in the kernel
 * from the work of both halves (the prefill's attended (query, key) pairs
 * and the decode's K/V bytes, at rates measured for these kernels).  A
 * smaller dec->kv_chunk (the split layout's unit; the workspace grows as it
 * shrinks) balances the end of the decode more finely.  Results are those of pa_prefill(pre) and
 * pa_decode(dec) (decode may split its key ranges differently; the combine
 * is exact up to rounding).
 *  - pre->scheduler must hold PA_MIXED_SCHEDULER_INTS int32 (zero before its
 *    first use, left zero by every completed launch: [0..1] the prefill
 *    counters, [2..3] the decode ones); dec->workspace as for pa_decode.
 *  - Both halves: the same k_cache / v_cache / num_pages / page_size / head
 *    counts / head_dim and pool type (bf16, or FP8 with the same k_scale and
 *    v_scale); an even GQA group and num_kv_heads % 4 == 0; no window or
 *    block mask on the prefill half (a decode window is fine);
 *    dec->overlap_previous = 0, dec->max_ctas ignored.
 *    Otherwise PA_ERR_UNSUPPORTED / PA_ERR_INVALID, nothing launched.
 *  - A batch with no prefill rows is pa_decode(dec); one with no decode
 *    sequences pa_prefill(pre).
 */
#define PA_MIXED_SCHEDULER_INTS 4
pa_status pa_mixed_batch(const pa_prefill_params *pre, const pa_decode_params *dec, void *stream);

/*
 * pa_decode_noalloc - pa_decode for callers that cannot allocate device
 * memory.  The paper has no counterpart for this entry point; it exists for
 * deployment.  Some callers may not call cudaMalloc at all: code
 * that runs while a CUDA graph is being captured, plug-ins whose host
 * application owns every byte of device memory through its own arena,
 * latency-critical loops where an allocation could synchronise the device,
 * or runtimes with a hard memory budget.  This call takes the same
 * parameters as pa_decode except that p->workspace and p->workspace_bytes
 * are ignored: the split partials go to a fixed scratch array that is part
 * of the library image (a file-scope __device__ array of
 * PA_DECODE_NOALLOC_SCRATCH_BYTES = 32 MiB, held on every GPU that loads the
 * library until the process exits).  The caller still passes q, the pools,
 * the metadata and out/lse.
 *  - Sizes whose split scratch (pa_decode_workspace_size) exceeds 32 MiB are
 *    rejected with PA_ERR_UNSUPPORTED and a message; nothing is launched.
 *  - The first call on a device (with that device current) looks up the
 *    scratch address with cudaGetSymbolAddress; make that first call before
 *    any stream capture.  No call allocates or frees memory.
 *  - All calls on a device share the one scratch array, which keeps the last
 *    call's partials (nothing in it needs to start at zero).  Calls whose
 *    kernels overlap on the GPU (other streams, other threads) race on it:
 *    serialise them.
 */
#define PA_DECODE_NOALLOC_SCRATCH_BYTES ((size_t)32 << 20)
pa_status pa_decode_noalloc(const pa_decode_params *p, void *stream);

/*
 * pa_lse_combine - stable merge of split partials ([T] s.12 and s.16):
 * for each row r (a (sequence, head) pair) and its n_r = num_splits_of_row
 * splits: M = max_s lse_s, w_s = exp(lse_s - M),
 *   out[r, :] = sum_s w_s O_s[r, :] / sum_s w_s,  lse[r] = M + ln sum_s w_s.
 * o_partial:   device fp32 [num_rows, max_splits, head_dim] (normalised O_s)
 * lse_partial: device fp32 [num_rows, max_splits] (natural log; -inf = empty)
 * splits_per_row: device int32 [num_rows] or NULL (= max_splits for all)
 * out: device bf16 [num_rows, head_dim]; lse_out: device fp32 [num_rows] or NULL.
 * A row with no split, or only empty splits, gives zeros and -inf.
 */
pa_status pa_lse_combine(const float *o_partial, const float *lse_partial,
                         const int32_t *splits_per_row, int32_t num_rows, int32_t max_splits,
                         int32_t head_dim, void *out, float *lse_out, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* PA_H */
