/*
 * Paged-KV exact attention: the plain, slow fp64 CPU oracle.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file; only the tests, the smoke check and the benchmark's CPU
 * baseline do.  It shares no code, header or constant with the CUDA library.
 *
 * What it computes, and where the pages define it:
 *
 *  - oracle_store_kv: the KV-cache store step, "RoPE + KV cache store" in the
 *    layer graph of "Transformer inference kernels: GEMM·Attention·
 *    FlashAttention·Fusion (3/10)", sections 1-2.  Token t's K and V rows are
 *    copied bit for bit into cache row slot_mapping[t]; a negative slot is a
 *    padding token and is skipped.
 *
 *  - oracle_attention: scaled dot-product attention, same page, section 10
 *    ("O = softmax(QK^T/sqrt(d) + mask) V"), computed the naive way: the score
 *    row S is materialised in full, then a two-pass softmax (max, then
 *    exponentials and their sum), then P.V.  Keys and values are read through
 *    the page table exactly as section 14 of the same page describes the
 *    address translation: logical position j -> page_table[b, j / P] ->
 *    physical page -> row page*P + j % P of the pool.  Query head h reads KV
 *    head h / (Hq/Hkv), the consecutive grouping of section 15 (32 q heads on
 *    8 KV heads, group size 4).  Request boundaries come from cu_seqlens_q and
 *    cu_seqlens_k (exclusive prefix sums of extend_len and device_len), as in
 *    "code-series sgl-project mini-sglang 07", "from ledger to tensors".  The
 *    causal mask is aligned to the END of each request's keys: query i of a
 *    request with Lq queries and Lk keys sits at absolute position
 *    Lk - Lq + i and sees keys 0 .. Lk - Lq + i (a cached prefix of Lk - Lq
 *    tokens followed by the Lq extend tokens).  A query row with no visible
 *    key returns O = 0 and lse = -inf (the "KV: empty" edge case of section
 *    24 of the first page).  A sliding window (the first page lists
 *    "causal, sliding window, custom sparse" masks as a dispatch axis,
 *    section 19) bounds the visible keys from below: with window_left >= 0
 *    a query at absolute position p sees only keys j >= p - window_left
 *    (so window_left + 1 keys at most when causal); window_left < 0 means
 *    no window.  A block-sparse mask (the "custom sparse" entry of the same
 *    list; the pages give no format, the reading here is the plainest one
 *    that a tiled kernel can honour): per request a grid of bytes over
 *    blocks of 128 queries x 128 keys, mask[b][i / 128][j / 128] for query
 *    index i within the request's rows (0 .. Lq - 1) and key j; a zero byte
 *    hides every key of that block from every query of that block.  It is
 *    additive in the sense of section 10: a hidden key's score is -inf, on
 *    top of the causal and window limits.  A row left with no visible key
 *    returns O = 0 and lse = -inf.
 *
 *  - oracle_page_table_from_token_table: the metadata step of the
 *    mini-sglang page, "from ledger to tensors": the global table is token
 *    granular (page size 1); a request's row is sliced with step P up to
 *    max_seqlen_k and, for P > 1, floor-divided by P to turn the slot of each
 *    page's first token into that page's id.
 *
 *  - FP8 KV cache (oracle_e4m3_value, oracle_e4m3_encode,
 *    oracle_store_kv_fp8, oracle_attention_fp8).  The first page lists FP8
 *    and quantized KV as a dispatch axis and a KV layout (section 19) and
 *    "quantized" KV as an edge case (section 24); the second page ("Inference
 *    systems and kernel optimisation", section 1) names FP8 quantization as
 *    part of FlashAttention-3.  Neither fixes a format, so the reading here is
 *    the plainest one: the E4M3 format with no infinities (1 sign bit, 4
 *    exponent bits with bias 7, 3 mantissa bits; exponent field 0 encodes
 *    subnormals m/8 * 2^-6; S.1111.111 is NaN, so the largest finite value is
 *    448), one fp32 scale per KV head for K and one for V, a stored element
 *    being code = E4M3(x / scale) with x / scale an IEEE single division,
 *    rounded to the nearest E4M3 value, ties to the even code, magnitudes of
 *    448 and above saturating to 448; attention then reads code * scale.
 *
 *  - Rotary position embedding before the store (oracle_rope_table,
 *    oracle_rope_rotate, oracle_round_bf16).  The first page's layer graph
 *    has "RoPE + KV cache store" as one step after the QKV projection
 *    (section 2), RoPE variants / scaling / offset as a dispatch axis
 *    (section 19) and "scaled RoPE" / "long offset" as edge cases (section
 *    24); the mini-sglang page applies the rotary to q and k with the batch's
 *    positions right before the attention backend ("the layer does not know
 *    the backend").  The pages do not define the rotation, so the reading is
 *    the standard rotary embedding: for a rotated width r (<= d) and pair
 *    index i < r/2 the angle is pos * base^(-2i/r); pairs are (i, i + r/2)
 *    ("rotate half") or (2i, 2i+1) ("interleaved"); a pair (a, b) becomes
 *    (a cos - b sin, b cos + a sin); elements r .. d-1 are unchanged.  The
 *    rotation can also be driven by a given cos/sin table (scaled variants).
 *    Outputs are exact in double; oracle_round_bf16 rounds a double to the
 *    nearest bf16 (ties to even) in one step.
 *
 * All arithmetic on floating point is IEEE double.  bf16 inputs are widened
 * exactly (a bf16 value is the top 16 bits of an IEEE single).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_OK 0
#define ORACLE_EINVAL -1
#define ORACLE_ERANGE -2
#define ORACLE_ENOMEM -3

static double widen_bf16(uint16_t bits)
{
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* ---------------------------------------------------------- E4M3 codec */

/* Value of an E4M3 code, from the format's definition. */
double oracle_e4m3_value(uint8_t code)
{
    int s = code >> 7, e = (code >> 3) & 15, m = code & 7;
    double mag;
    if (e == 15 && m == 7) return NAN;
    if (e == 0) mag = ldexp((double)m / 8.0, -6);          /* subnormal */
    else mag = ldexp(1.0 + (double)m / 8.0, e - 7);
    return s ? -mag : mag;
}

/* Nearest E4M3 code to x (ties to the even code), saturating to +-448.
 * The non-negative finite codes 0x00..0x7E have increasing values, so the
 * code just below |x| is found by bisection and compared with its upper
 * neighbour.  NaN gives 0x7F. */
uint8_t oracle_e4m3_encode(float x)
{
    if (isnan(x)) return 0x7F;
    uint8_t sign = signbit(x) ? 0x80 : 0x00;
    double a = fabs((double)x);
    if (a >= 448.0) return sign | 0x7E;
    int lo = 0, hi = 0x7E;                 /* value(lo) <= a < value(hi) */
    while (hi - lo > 1) {
        int mid = (lo + hi) / 2;
        if (oracle_e4m3_value((uint8_t)mid) <= a) lo = mid; else hi = mid;
    }
    double dlo = a - oracle_e4m3_value((uint8_t)lo);
    double dhi = oracle_e4m3_value((uint8_t)hi) - a;
    int c;
    if (dlo < dhi) c = lo;
    else if (dhi < dlo) c = hi;
    else c = (lo & 1) ? hi : lo;           /* tie: the even code */
    return sign | (uint8_t)c;
}

static float widen_bf16_f32(uint16_t bits)
{
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* FP8 KV store.  k, v: [T, Hkv, d] bf16 bits; caches: [num_slots, Hkv, d]
 * E4M3 codes; k_scale, v_scale: [Hkv].  Element c of head h of token t goes
 * to row slot_mapping[t] as E4M3(x / scale[h]), the division in IEEE single. */
int oracle_store_kv_fp8(const uint16_t *k, const uint16_t *v, const int32_t *slot_mapping,
                        int64_t num_tokens, uint8_t *k_cache, uint8_t *v_cache,
                        int64_t num_slots, int32_t Hkv, int32_t d,
                        const float *k_scale, const float *v_scale)
{
    if (num_tokens < 0 || num_slots < 0 || Hkv <= 0 || d <= 0) return ORACLE_EINVAL;
    int64_t row = (int64_t)Hkv * d;
    for (int64_t t = 0; t < num_tokens; ++t) {
        int64_t slot = slot_mapping[t];
        if (slot < 0) continue;
        if (slot >= num_slots) return ORACLE_ERANGE;
        for (int32_t h = 0; h < Hkv; ++h) {
            for (int32_t c = 0; c < d; ++c) {
                int64_t src = t * row + (int64_t)h * d + c, dst = slot * row + (int64_t)h * d + c;
                volatile float qk = widen_bf16_f32(k[src]) / k_scale[h];
                volatile float qv = widen_bf16_f32(v[src]) / v_scale[h];
                k_cache[dst] = oracle_e4m3_encode(qk);
                v_cache[dst] = oracle_e4m3_encode(qv);
            }
        }
    }
    return ORACLE_OK;
}

/* ------------------------------------------------------------- threads */

int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void oracle_set_threads(int n)
{
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

/* KV store.  k, v: [T, row_elems] bf16 bits; caches: [num_slots, row_elems]. */
int oracle_store_kv(const uint16_t *k, const uint16_t *v, const int32_t *slot_mapping,
                    int64_t num_tokens, uint16_t *k_cache, uint16_t *v_cache,
                    int64_t num_slots, int64_t row_elems)
{
    if (num_tokens < 0 || num_slots < 0 || row_elems <= 0) return ORACLE_EINVAL;
    for (int64_t t = 0; t < num_tokens; ++t) {
        int64_t slot = slot_mapping[t];
        if (slot < 0) continue;
        if (slot >= num_slots) return ORACLE_ERANGE;
        memcpy(k_cache + slot * row_elems, k + t * row_elems, (size_t)row_elems * 2);
        memcpy(v_cache + slot * row_elems, v + t * row_elems, (size_t)row_elems * 2);
    }
    return ORACLE_OK;
}

/* Metadata: page table [B, out_cols] from the token-granular global table.
 * token_table: [num_rows, tt_stride]; table_idx[b] selects request b's row.
 * Column c of the result is token_table[table_idx[b], c * P] / P (floor). */
int oracle_page_table_from_token_table(const int32_t *token_table, int64_t tt_stride,
                                       const int32_t *table_idx, int32_t num_seqs,
                                       int32_t max_seqlen_k, int32_t page_size,
                                       int32_t *out, int64_t out_cols)
{
    if (page_size <= 0 || num_seqs < 0 || max_seqlen_k < 0) return ORACLE_EINVAL;
    int64_t cols = ((int64_t)max_seqlen_k + page_size - 1) / page_size;
    if (cols > out_cols) return ORACLE_EINVAL;
    for (int32_t b = 0; b < num_seqs; ++b) {
        const int32_t *row = token_table + (int64_t)table_idx[b] * tt_stride;
        for (int64_t c = 0; c < cols; ++c) {
            int64_t slot = row[c * page_size];
            /* floor division; slots are non-negative for real tokens */
            int64_t q = slot / page_size;
            if (slot < 0 && q * page_size != slot) q -= 1;
            out[(int64_t)b * out_cols + c] = (int32_t)q;
        }
    }
    return ORACLE_OK;
}

/* Metadata: per-request boundaries from the three lengths.  extend_len is the
 * query length and device_len = cached_len + extend_len the key length of each
 * request; cu_q / cu_k are their exclusive prefix sums starting at 0 and
 * cache_seqlens is device_len itself ("from ledger to tensors"). */
int oracle_seqlens(const int32_t *cached_len, const int32_t *extend_len, int32_t num_seqs,
                   int32_t *cu_q, int32_t *cu_k, int32_t *cache_seqlens,
                   int32_t *max_seqlen_q, int32_t *max_seqlen_k)
{
    if (num_seqs < 0) return ORACLE_EINVAL;
    int64_t sq = 0, sk = 0;
    int32_t mq = 0, mk = 0;
    cu_q[0] = 0;
    cu_k[0] = 0;
    for (int32_t b = 0; b < num_seqs; ++b) {
        int64_t lq = extend_len[b];
        int64_t lk = (int64_t)cached_len[b] + extend_len[b];
        if (lq < 0 || cached_len[b] < 0) return ORACLE_EINVAL;
        sq += lq;
        sk += lk;
        if (sq > INT32_MAX || sk > INT32_MAX) return ORACLE_ERANGE;
        cu_q[b + 1] = (int32_t)sq;
        cu_k[b + 1] = (int32_t)sk;
        cache_seqlens[b] = (int32_t)lk;
        if (lq > mq) mq = (int32_t)lq;
        if (lk > mk) mk = (int32_t)lk;
    }
    *max_seqlen_q = mq;
    *max_seqlen_k = mk;
    return ORACLE_OK;
}

/* One attention row: query token t (global index into q), query head h.
 * Writes d doubles to o and one to *lse.  scratch holds >= Lk doubles. */
/* The K/V pools as attention reads them: bf16 bits, or E4M3 codes with a
 * scale per KV head (value = code value * scale). */
typedef struct {
    const void *k, *v;
    int fp8;
    const float *k_scale, *v_scale;
} kv_pools;

/* Optional block-sparse mask: bytes [num_seqs][nq][nk] over 128 x 128 blocks
 * (m == NULL: none). */
typedef struct {
    const uint8_t *m;
    int32_t nq, nk;
} block_mask;

#define ORACLE_MASK_BLOCK 128

static double kv_value(const void *cache, int fp8, const float *scale, int64_t idx, int32_t kvh)
{
    if (!fp8) return widen_bf16(((const uint16_t *)cache)[idx]);
    return oracle_e4m3_value(((const uint8_t *)cache)[idx]) * (double)scale[kvh];
}

static int attention_row(const uint16_t *q, const kv_pools *kv,
                         const int32_t *page_table, int64_t pt_stride,
                         const int32_t *cu_q, const int32_t *cu_k, int32_t num_seqs,
                         int32_t Hq, int32_t Hkv, int32_t d, int32_t P, int64_t num_pages,
                         int causal, int32_t window_left, const block_mask *bm, double scale,
                         int64_t t, int32_t h, double *o, double *lse, double *s_row)
{
    /* request b owning query token t */
    int32_t b = -1;
    for (int32_t i = 0; i < num_seqs; ++i) {
        if (cu_q[i] <= t && t < cu_q[i + 1]) { b = i; break; }
    }
    if (b < 0) return ORACLE_EINVAL;
    int64_t Lq = cu_q[b + 1] - cu_q[b];
    int64_t Lk = cu_k[b + 1] - cu_k[b];
    int64_t i = t - cu_q[b];
    int64_t off = Lk - Lq;                 /* cached prefix length */
    int64_t n_vis = Lk;
    if (causal) {
        int64_t lim = off + i + 1;         /* keys 0 .. off+i are visible */
        if (lim < n_vis) n_vis = lim;
        if (n_vis < 0) n_vis = 0;
    }
    int64_t j_lo = 0;                      /* sliding window: keys >= off + i - window_left */
    if (window_left >= 0) {
        j_lo = off + i - window_left;
        if (j_lo < 0) j_lo = 0;
    }
    int32_t g = Hq / Hkv;
    int32_t kvh = h / g;
    const uint16_t *qrow = q + (t * Hq + h) * (int64_t)d;

    for (int c = 0; c < d; ++c) o[c] = 0.0;
    if (n_vis <= j_lo) { *lse = -INFINITY; return ORACLE_OK; }
    /* the block-mask row of this query (NULL: every block visible) */
    const uint8_t *mrow = NULL;
    if (bm && bm->m) {
        if (i / ORACLE_MASK_BLOCK >= bm->nq || (n_vis - 1) / ORACLE_MASK_BLOCK >= bm->nk) return ORACLE_EINVAL;
        mrow = bm->m + ((int64_t)b * bm->nq + i / ORACLE_MASK_BLOCK) * (int64_t)bm->nk;
    }

    /* pass 0: materialise the score row S[j] = scale * q . K_j (-inf where
     * the block mask hides the key) */
    for (int64_t j = j_lo; j < n_vis; ++j) {
        if (mrow && mrow[j / ORACLE_MASK_BLOCK] == 0) { s_row[j] = -INFINITY; continue; }
        int64_t page = page_table[b * pt_stride + j / P];
        if (page < 0 || page >= num_pages) return ORACLE_ERANGE;
        int64_t row = page * P + j % P;
        int64_t kbase = (row * Hkv + kvh) * (int64_t)d;
        double acc = 0.0;
        for (int c = 0; c < d; ++c)
            acc += widen_bf16(qrow[c]) * kv_value(kv->k, kv->fp8, kv->k_scale, kbase + c, kvh);
        s_row[j] = scale * acc;
    }
    /* pass 1: row maximum */
    double m = -INFINITY;
    for (int64_t j = j_lo; j < n_vis; ++j) if (s_row[j] > m) m = s_row[j];
    if (m == -INFINITY) { *lse = -INFINITY; return ORACLE_OK; }   /* every key hidden */
    /* pass 2: exponentials, their sum, and P.V */
    double l = 0.0;
    for (int64_t j = j_lo; j < n_vis; ++j) {
        double p = exp(s_row[j] - m);
        l += p;
        int64_t page = page_table[b * pt_stride + j / P];
        int64_t row = page * P + j % P;
        int64_t vbase = (row * Hkv + kvh) * (int64_t)d;
        for (int c = 0; c < d; ++c) o[c] += p * kv_value(kv->v, kv->fp8, kv->v_scale, vbase + c, kvh);
    }
    for (int c = 0; c < d; ++c) o[c] /= l;
    *lse = m + log(l);
    return ORACLE_OK;
}

/* Attention over paged K/V.
 * q: [Tq, Hq, d] bf16 bits; k_cache, v_cache: [num_pages*P, Hkv, d] bf16 bits;
 * page_table: [num_seqs, pt_stride] int32; cu_q, cu_k: [num_seqs+1] int32.
 * rows == NULL: every (token, head) row; out [Tq, Hq, d], lse [Tq, Hq].
 * rows != NULL: nrows pairs (token, head) as int64; out [nrows, d], lse [nrows]. */
static int attention_all(const uint16_t *q, const kv_pools *kv,
                         const int32_t *page_table, int64_t pt_stride,
                         const int32_t *cu_q, const int32_t *cu_k, int32_t num_seqs,
                         int32_t Hq, int32_t Hkv, int32_t d, int32_t P, int64_t num_pages,
                         int causal, int32_t window_left, const block_mask *bm, double scale,
                         const int64_t *rows, int64_t nrows, double *out, double *lse)
{
    if (num_seqs < 0 || Hq <= 0 || Hkv <= 0 || d <= 0 || P <= 0 || Hq % Hkv) return ORACLE_EINVAL;
    int64_t Tq = num_seqs > 0 ? cu_q[num_seqs] : 0;
    int64_t max_lk = 0;
    for (int32_t b = 0; b < num_seqs; ++b) {
        int64_t Lq = cu_q[b + 1] - cu_q[b], Lk = cu_k[b + 1] - cu_k[b];
        /* more queries than keys is malformed, except over an empty KV
         * range (a padded or dummy request): then every row sees nothing */
        if (Lq < 0 || Lk < 0 || (Lq > Lk && Lk > 0)) return ORACLE_EINVAL;
        if (Lk > max_lk) max_lk = Lk;
    }
    int64_t n = rows ? nrows : Tq * Hq;
    int status = ORACLE_OK;
#pragma omp parallel
    {
        double *s_row = (double *)malloc(sizeof(double) * (size_t)(max_lk > 0 ? max_lk : 1));
        if (!s_row) {
#pragma omp atomic write
            status = ORACLE_ENOMEM;
        } else {
#pragma omp for schedule(dynamic, 4)
            for (int64_t r = 0; r < n; ++r) {
                int64_t t = rows ? rows[2 * r] : r / Hq;
                int32_t h = (int32_t)(rows ? rows[2 * r + 1] : r % Hq);
                if (t < 0 || t >= Tq || h < 0 || h >= Hq) {
#pragma omp atomic write
                    status = ORACLE_EINVAL;
                    continue;
                }
                int st = attention_row(q, kv, page_table, pt_stride, cu_q, cu_k,
                                       num_seqs, Hq, Hkv, d, P, num_pages, causal, window_left, bm, scale,
                                       t, h, out + r * (int64_t)d, lse + r, s_row);
                if (st != ORACLE_OK) {
#pragma omp atomic write
                    status = st;
                }
            }
            free(s_row);
        }
    }
    return status;
}

int oracle_attention(const uint16_t *q, const uint16_t *k_cache, const uint16_t *v_cache,
                     const int32_t *page_table, int64_t pt_stride,
                     const int32_t *cu_q, const int32_t *cu_k, int32_t num_seqs,
                     int32_t Hq, int32_t Hkv, int32_t d, int32_t P, int64_t num_pages,
                     int causal, int32_t window_left, double scale, const int64_t *rows,
                     int64_t nrows, double *out, double *lse)
{
    kv_pools kv = {k_cache, v_cache, 0, NULL, NULL};
    return attention_all(q, &kv, page_table, pt_stride, cu_q, cu_k, num_seqs, Hq, Hkv, d, P,
                         num_pages, causal, window_left, NULL, scale, rows, nrows, out, lse);
}

/* The same with a block-sparse mask bmask [num_seqs][bm_q][bm_k] (bytes;
 * zero = the 128 x 128 block is hidden). */
int oracle_attention_bm(const uint16_t *q, const uint16_t *k_cache, const uint16_t *v_cache,
                        const int32_t *page_table, int64_t pt_stride,
                        const int32_t *cu_q, const int32_t *cu_k, int32_t num_seqs,
                        int32_t Hq, int32_t Hkv, int32_t d, int32_t P, int64_t num_pages,
                        int causal, int32_t window_left, const uint8_t *bmask, int32_t bm_q,
                        int32_t bm_k, double scale, const int64_t *rows, int64_t nrows, double *out,
                        double *lse)
{
    if (bmask && (bm_q <= 0 || bm_k <= 0)) return ORACLE_EINVAL;
    kv_pools kv = {k_cache, v_cache, 0, NULL, NULL};
    block_mask bm = {bmask, bm_q, bm_k};
    return attention_all(q, &kv, page_table, pt_stride, cu_q, cu_k, num_seqs, Hq, Hkv, d, P,
                         num_pages, causal, window_left, &bm, scale, rows, nrows, out, lse);
}

/* The same over E4M3 pools (codes [num_pages*P, Hkv, d]) with per-KV-head
 * scales k_scale[Hkv], v_scale[Hkv]. */
int oracle_attention_fp8(const uint16_t *q, const uint8_t *k_cache, const uint8_t *v_cache,
                         const float *k_scale, const float *v_scale,
                         const int32_t *page_table, int64_t pt_stride,
                         const int32_t *cu_q, const int32_t *cu_k, int32_t num_seqs,
                         int32_t Hq, int32_t Hkv, int32_t d, int32_t P, int64_t num_pages,
                         int causal, int32_t window_left, double scale, const int64_t *rows,
                         int64_t nrows, double *out, double *lse)
{
    kv_pools kv = {k_cache, v_cache, 1, k_scale, v_scale};
    return attention_all(q, &kv, page_table, pt_stride, cu_q, cu_k, num_seqs, Hq, Hkv, d, P,
                         num_pages, causal, window_left, NULL, scale, rows, nrows, out, lse);
}

int oracle_attention_fp8_bm(const uint16_t *q, const uint8_t *k_cache, const uint8_t *v_cache,
                            const float *k_scale, const float *v_scale,
                            const int32_t *page_table, int64_t pt_stride,
                            const int32_t *cu_q, const int32_t *cu_k, int32_t num_seqs,
                            int32_t Hq, int32_t Hkv, int32_t d, int32_t P, int64_t num_pages,
                            int causal, int32_t window_left, const uint8_t *bmask, int32_t bm_q,
                            int32_t bm_k, double scale, const int64_t *rows, int64_t nrows,
                            double *out, double *lse)
{
    if (bmask && (bm_q <= 0 || bm_k <= 0)) return ORACLE_EINVAL;
    kv_pools kv = {k_cache, v_cache, 1, k_scale, v_scale};
    block_mask bm = {bmask, bm_q, bm_k};
    return attention_all(q, &kv, page_table, pt_stride, cu_q, cu_k, num_seqs, Hq, Hkv, d, P,
                         num_pages, causal, window_left, &bm, scale, rows, nrows, out, lse);
}

/* ---------------------------------------------------------------- RoPE */

/* cos / sin tables [max_pos, r/2]: angle(p, i) = p * base^(-2i/r). */
int oracle_rope_table(double *cos_t, double *sin_t, int32_t max_pos, int32_t r, double base)
{
    if (max_pos < 0 || r <= 0 || r % 2 || !(base > 0.0)) return ORACLE_EINVAL;
    int32_t h = r / 2;
    for (int32_t p = 0; p < max_pos; ++p) {
        for (int32_t i = 0; i < h; ++i) {
            double ang = (double)p * pow(base, -2.0 * (double)i / (double)r);
            cos_t[(int64_t)p * h + i] = cos(ang);
            sin_t[(int64_t)p * h + i] = sin(ang);
        }
    }
    return ORACLE_OK;
}

/* Rotate x: [T, H, d] bf16 bits, token t at position positions[t], with the
 * tables [max_pos, r/2]; out: [T, H, d] double (exact products and sums). */
int oracle_rope_rotate(const uint16_t *x, const int32_t *positions, int64_t T, int32_t H, int32_t d,
                       int32_t r, int interleaved, const double *cos_t, const double *sin_t,
                       int32_t max_pos, double *out)
{
    if (T < 0 || H <= 0 || d <= 0 || r <= 0 || r > d || r % 2) return ORACLE_EINVAL;
    int32_t h = r / 2;
    for (int64_t t = 0; t < T; ++t) {
        int32_t p = positions[t];
        if (p < 0 || p >= max_pos) return ORACLE_ERANGE;
        for (int32_t hd = 0; hd < H; ++hd) {
            const uint16_t *xr = x + (t * H + hd) * (int64_t)d;
            double *o = out + (t * H + hd) * (int64_t)d;
            for (int32_t c = 0; c < d; ++c) o[c] = widen_bf16(xr[c]);
            for (int32_t i = 0; i < h; ++i) {
                int32_t ia = interleaved ? 2 * i : i;
                int32_t ib = interleaved ? 2 * i + 1 : i + h;
                double a = widen_bf16(xr[ia]), b = widen_bf16(xr[ib]);
                double cs = cos_t[(int64_t)p * h + i], sn = sin_t[(int64_t)p * h + i];
                o[ia] = a * cs - b * sn;
                o[ib] = b * cs + a * sn;
            }
        }
    }
    return ORACLE_OK;
}

/* Nearest bf16 (8 significant bits, ties to even) of each double, as bits. */
int oracle_round_bf16(const double *x, int64_t n, uint16_t *out)
{
    for (int64_t k = 0; k < n; ++k) {
        double v = x[k];
        float f;
        if (isnan(v)) {
            f = NAN;
        } else if (v == 0.0 || isinf(v)) {
            f = (float)v;
        } else {
            int e;
            frexp(v, &e);                          /* |v| in [2^(e-1), 2^e) */
            int q = e - 8;                         /* quantum of 8 significant bits */
            if (q < -133) q = -133;                /* bf16 subnormal quantum */
            double scaled = ldexp(v, -q);
            double rr = nearbyint(scaled);         /* ties to even */
            double rv = ldexp(rr, q);
            f = (float)rv;                         /* exact: 8 significant bits */
            if (fabs(rv) > 3.3895313892515355e38) f = v > 0 ? INFINITY : -INFINITY;
        }
        uint32_t u;
        memcpy(&u, &f, sizeof u);
        out[k] = (uint16_t)(u >> 16);
    }
    return ORACLE_OK;
}
