/*
 * A plain C program that uses libpa.so through include/pa.h alone (no Python,
 * no C++): it stores the newest token of two sequences with pa_store_kv, then
 * runs pa_decode, pa_decode_noalloc and pa_prefill on cases whose answers have
 * a closed form.
 *
 * Every key of the used pages is the same vector, so all visible scores of a
 * query are equal and attention is the plain mean of the visible V rows.  V
 * row j of a sequence holds the value j in every element.  Decode sees all L
 * keys: the output is (L - 1) / 2 everywhere, and lse = score + ln L, where
 * score = scale * q . k.  Prefill of the last Lq keys of each sequence: the
 * query at position p sees keys 0 .. p, so its output is p / 2 and its lse
 * score + ln(p + 1).  Unused page-table entries point at a page full of NaN,
 * so any read through a wrong entry shows up in the output, and so do the
 * slots past a sequence's end inside its last page (never written: a kernel
 * that lets one of them reach an output fails).  Splits of 16 keys force
 * decode's split-and-merge path.
 *
 * Exit status 0 = every check passed.
 */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime.h>

#include "pa.h"

#define B 2
#define HQ 4
#define HKV 2
#define D 64
#define P 16
#define PAGES 8
#define POISON 7
#define STRIDE 3

static const int kLen[B] = {20, 40};
static const int kLq[B] = {5, 12};          /* prefill: the last Lq keys are the queries */
static const int kPages[B][STRIDE] = {{3, 1, POISON}, {0, 5, 2}};

static uint16_t bf16(float x) {       /* exact for the small values used here */
    uint32_t u;
    memcpy(&u, &x, 4);
    return (uint16_t)(u >> 16);
}

static float from_bf16(uint16_t h) {
    uint32_t u = (uint32_t)h << 16;
    float x;
    memcpy(&x, &u, 4);
    return x;
}

#define CK(call)                                                                  \
    do {                                                                          \
        cudaError_t e_ = (call);                                                  \
        if (e_ != cudaSuccess) {                                                  \
            fprintf(stderr, "%s:%d %s: %s\n", __FILE__, __LINE__, #call,          \
                    cudaGetErrorString(e_));                                      \
            return 1;                                                             \
        }                                                                         \
    } while (0)

#define PK(call)                                                                  \
    do {                                                                          \
        pa_status s_ = (call);                                                    \
        if (s_ != PA_OK) {                                                        \
            fprintf(stderr, "%s:%d %s: %s (%s)\n", __FILE__, __LINE__, #call,     \
                    pa_status_string(s_), pa_last_error());                       \
            return 1;                                                             \
        }                                                                         \
    } while (0)

static int check(const uint16_t *out, const float *lse, float scale, const char *what) {
    int bad = 0;
    const float score = scale * (float)D * 0.5f;           /* q = 0.5, k = 1 */
    for (int b = 0; b < B; ++b) {
        const float want = 0.5f * (float)(kLen[b] - 1);
        const float want_lse = score + logf((float)kLen[b]);
        for (int h = 0; h < HQ; ++h) {
            for (int c = 0; c < D; ++c) {
                const float got = from_bf16(out[((size_t)b * HQ + h) * D + c]);
                if (!(fabsf(got - want) <= 1e-2f)) {
                    if (bad < 5) fprintf(stderr, "%s: out[%d,%d,%d] = %g, want %g\n", what, b, h, c, got, want);
                    ++bad;
                }
            }
            const float l = lse[b * HQ + h];
            if (!(fabsf(l - want_lse) <= 2e-3f)) {
                if (bad < 5) fprintf(stderr, "%s: lse[%d,%d] = %g, want %g\n", what, b, h, l, want_lse);
                ++bad;
            }
        }
    }
    return bad;
}

int main(void) {
    if (pa_abi_version() != PA_ABI_VERSION) {
        fprintf(stderr, "ABI version %d, header %d\n", pa_abi_version(), PA_ABI_VERSION);
        return 1;
    }
    const size_t row = (size_t)HKV * D;                    /* elements per slot */
    const size_t pool_elems = (size_t)PAGES * P * row;
    uint16_t *hk = malloc(pool_elems * 2), *hv = malloc(pool_elems * 2);
    for (size_t i = 0; i < pool_elems; ++i) hk[i] = hv[i] = 0x7FC0;   /* NaN */
    /* the pages of each sequence: K = 1, V = key index, NaN past the end;
       the last key is left NaN here and written by pa_store_kv below */
    for (int b = 0; b < B; ++b)
        for (int j = 0; j + 1 < kLen[b]; ++j) {
            const size_t slot = (size_t)kPages[b][j / P] * P + j % P;
            for (size_t e = 0; e < row; ++e) {
                hk[slot * row + e] = bf16(1.0f);
                hv[slot * row + e] = bf16((float)j);
            }
        }
    uint16_t hq[B * HQ * D], hknew[B * HKV * D], hvnew[B * HKV * D];
    int32_t hslot[B], hpt[B * STRIDE], hlen[B];
    for (int i = 0; i < B * HQ * D; ++i) hq[i] = bf16(0.5f);
    for (int b = 0; b < B; ++b) {
        const int j = kLen[b] - 1;
        hslot[b] = kPages[b][j / P] * P + j % P;
        hlen[b] = kLen[b];
        for (int s = 0; s < STRIDE; ++s) hpt[b * STRIDE + s] = kPages[b][s];
        for (int e = 0; e < HKV * D; ++e) {
            hknew[b * HKV * D + e] = bf16(1.0f);
            hvnew[b * HKV * D + e] = bf16((float)j);
        }
    }

    void *k_cache, *v_cache, *q, *k_new, *v_new, *out, *ws;
    int32_t *slot, *pt, *len;
    float *lse;
    CK(cudaMalloc(&k_cache, pool_elems * 2));
    CK(cudaMalloc(&v_cache, pool_elems * 2));
    CK(cudaMalloc(&q, sizeof hq));
    CK(cudaMalloc(&k_new, sizeof hknew));
    CK(cudaMalloc(&v_new, sizeof hvnew));
    CK(cudaMalloc((void **)&slot, sizeof hslot));
    CK(cudaMalloc((void **)&pt, sizeof hpt));
    CK(cudaMalloc((void **)&len, sizeof hlen));
    CK(cudaMalloc(&out, (size_t)B * HQ * D * 2));
    CK(cudaMalloc((void **)&lse, (size_t)B * HQ * 4));
    CK(cudaMemcpy(k_cache, hk, pool_elems * 2, cudaMemcpyHostToDevice));
    CK(cudaMemcpy(v_cache, hv, pool_elems * 2, cudaMemcpyHostToDevice));
    CK(cudaMemcpy(q, hq, sizeof hq, cudaMemcpyHostToDevice));
    CK(cudaMemcpy(k_new, hknew, sizeof hknew, cudaMemcpyHostToDevice));
    CK(cudaMemcpy(v_new, hvnew, sizeof hvnew, cudaMemcpyHostToDevice));
    CK(cudaMemcpy(slot, hslot, sizeof hslot, cudaMemcpyHostToDevice));
    CK(cudaMemcpy(pt, hpt, sizeof hpt, cudaMemcpyHostToDevice));
    CK(cudaMemcpy(len, hlen, sizeof hlen, cudaMemcpyHostToDevice));

    PK(pa_store_kv(k_new, v_new, slot, B, k_cache, v_cache, (int64_t)PAGES * P, HKV, D, NULL));

    pa_decode_params p;
    memset(&p, 0, sizeof p);
    p.q = q;
    p.k_cache = k_cache;
    p.v_cache = v_cache;
    p.page_table = pt;
    p.page_table_stride = STRIDE;
    p.cache_seqlens = len;
    p.num_seqs = B;
    p.max_seqlen_k = 40;
    p.num_q_heads = HQ;
    p.num_kv_heads = HKV;
    p.head_dim = D;
    p.page_size = P;
    p.num_pages = PAGES;
    p.scale = 0.125f;
    p.out = out;
    p.lse = lse;
    p.kv_chunk = 16;
    p.kv_dtype = PA_KV_BF16;
    const size_t wsb = pa_decode_workspace_size(&p);
    if (wsb == 0) {
        fprintf(stderr, "workspace size 0: %s\n", pa_last_error());
        return 1;
    }
    CK(cudaMalloc(&ws, wsb));
    p.workspace = ws;
    p.workspace_bytes = wsb;

    uint16_t hout[B * HQ * D];
    float hlse[B * HQ];
    int bad = 0;
    for (int pass = 0; pass < 2; ++pass) {          /* pa_decode, then pa_decode_noalloc */
        CK(cudaMemset(out, 0xFF, (size_t)B * HQ * D * 2));   /* NaN until written */
        CK(cudaMemset(lse, 0xFF, (size_t)B * HQ * 4));
        if (pass == 0) PK(pa_decode(&p, NULL));
        else PK(pa_decode_noalloc(&p, NULL));
        int32_t bits = 0;
        PK(pa_device_error(&bits, NULL));
        if (bits != 0) {
            fprintf(stderr, "device error bits %d\n", bits);
            return 1;
        }
        CK(cudaMemcpy(hout, out, sizeof hout, cudaMemcpyDeviceToHost));
        CK(cudaMemcpy(hlse, lse, sizeof hlse, cudaMemcpyDeviceToHost));
        bad += check(hout, hlse, p.scale, pass == 0 ? "pa_decode" : "pa_decode_noalloc");
    }

    /* prefill / extend of the last Lq keys of each sequence */
    enum { TQ = 5 + 12 };
    int32_t hcuq[B + 1] = {0, kLq[0], kLq[0] + kLq[1]}, hcuk[B + 1] = {0, kLen[0], kLen[0] + kLen[1]};
    uint16_t hqp[TQ * HQ * D], houtp[TQ * HQ * D];
    float hlsep[HQ * TQ];
    for (int i = 0; i < TQ * HQ * D; ++i) hqp[i] = bf16(0.5f);
    void *qp, *outp;
    int32_t *cuq, *cuk, *sched;
    float *lsep;
    CK(cudaMalloc((void **)&sched, PA_PREFILL_SCHEDULER_INTS * sizeof(int32_t)));
    CK(cudaMemset(sched, 0, PA_PREFILL_SCHEDULER_INTS * sizeof(int32_t)));
    CK(cudaMalloc(&qp, sizeof hqp));
    CK(cudaMalloc(&outp, sizeof houtp));
    CK(cudaMalloc((void **)&lsep, sizeof hlsep));
    CK(cudaMalloc((void **)&cuq, sizeof hcuq));
    CK(cudaMalloc((void **)&cuk, sizeof hcuk));
    CK(cudaMemcpy(qp, hqp, sizeof hqp, cudaMemcpyHostToDevice));
    CK(cudaMemcpy(cuq, hcuq, sizeof hcuq, cudaMemcpyHostToDevice));
    CK(cudaMemcpy(cuk, hcuk, sizeof hcuk, cudaMemcpyHostToDevice));
    CK(cudaMemset(outp, 0xFF, sizeof houtp));
    CK(cudaMemset(lsep, 0xFF, sizeof hlsep));
    pa_prefill_params f;
    memset(&f, 0, sizeof f);
    f.q = qp;
    f.k_cache = k_cache;
    f.v_cache = v_cache;
    f.page_table = pt;
    f.page_table_stride = STRIDE;
    f.total_q = TQ;
    f.cu_seqlens_q = cuq;
    f.cu_seqlens_k = cuk;
    f.num_seqs = B;
    f.max_seqlen_q = 12;
    f.max_seqlen_k = 40;
    f.num_q_heads = HQ;
    f.num_kv_heads = HKV;
    f.head_dim = D;
    f.page_size = P;
    f.num_pages = PAGES;
    f.causal = 1;
    f.scale = 0.125f;
    f.out = outp;
    f.lse = lsep;
    f.lse_stride = TQ;
    f.kv_dtype = PA_KV_BF16;
    f.scheduler = sched;
    PK(pa_prefill(&f, NULL));
    int32_t bits = 0;
    PK(pa_device_error(&bits, NULL));
    if (bits != 0) {
        fprintf(stderr, "prefill: device error bits %d\n", bits);
        return 1;
    }
    CK(cudaMemcpy(houtp, outp, sizeof houtp, cudaMemcpyDeviceToHost));
    CK(cudaMemcpy(hlsep, lsep, sizeof hlsep, cudaMemcpyDeviceToHost));
    const float score = f.scale * (float)D * 0.5f;
    for (int b = 0; b < B; ++b)
        for (int i = 0; i < kLq[b]; ++i) {
            const int t = hcuq[b] + i, pos = kLen[b] - kLq[b] + i;
            for (int h = 0; h < HQ; ++h) {
                for (int c = 0; c < D; ++c) {
                    const float got = from_bf16(houtp[((size_t)t * HQ + h) * D + c]);
                    if (!(fabsf(got - 0.5f * (float)pos) <= 1e-2f)) {
                        if (bad < 5) fprintf(stderr, "prefill: out[%d,%d,%d] = %g, want %g\n", t, h, c, got, 0.5f * pos);
                        ++bad;
                    }
                }
                const float l = hlsep[h * TQ + t], want = score + logf((float)(pos + 1));
                if (!(fabsf(l - want) <= 2e-3f)) {
                    if (bad < 5) fprintf(stderr, "prefill: lse[%d,%d] = %g, want %g\n", h, t, l, want);
                    ++bad;
                }
            }
        }
    if (bad) {
        fprintf(stderr, "%d mismatches\n", bad);
        return 1;
    }
    printf("ok: store + decode (split 16) + decode_noalloc + prefill through the C ABI\n");
    free(hk);
    free(hv);
    return 0;
}
