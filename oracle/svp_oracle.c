/*
 * svp_oracle.c -- plain, slow fp64 CPU oracle for packed speculative verification.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may include, link or call
 * this file: only the tests, the smoke check and the benchmark's CPU-baseline leg use
 * it.  It shares no header, helper or constant with the CUDA library.
 *
 * Sources (page title, then section / figure):
 *   [DScale]  "DScale: Scaling Block-Diffusion Speculative Decoding with Adaptive
 *             Verification" -- SIII-B (tile routing), SIII-C (Flat-buffer packer, Fig. 6),
 *             SIII-D (graph integration: request-local causal masking over packed rows;
 *             Prefix verifier: row offset_i + a_i supplies the successor).
 *   [MiniLab] "DFlash-Mini-Lab" README -- one verifier call on [anchor + draft suffix],
 *             accept the exact prefix; top-1/top-2 draft-logit margin (DFlash7-ACT).
 *
 * Readings where the pages are silent (the mask equation is missing from the text):
 *   - row j of request i attends to all ctx_len[i] context tokens, then to its own
 *     candidates c = 0..j (diagonal inclusive); rows never see other requests;
 *   - query head h uses KV head h / (hq / hkv) (contiguous GQA grouping);
 *   - softmax scale is passed in (1/sqrt(d) in every workload);
 *   - row offset_i + j holds candidate j (j = 0 is the anchor); its logits predict
 *     candidate j + 1.
 *
 * Every stored input value (fp32 or bf16) is widened exactly to double before use.
 * Attention is computed straight from the definition: s_t = scale * <q, k_t>,
 * m = max_t s_t, p_t = exp(s_t - m), o = sum_t p_t v_t / sum_t p_t,
 * lse = m + log(sum_t p_t).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { ORC_F32 = 0, ORC_BF16 = 1 };

/* Read element idx of a stored array as double (bf16 = upper 16 bits of an fp32). */
static double orc_load(const void *base, int dtype, int64_t idx)
{
    if (dtype == ORC_F32)
        return (double)((const float *)base)[idx];
    uint32_t bits = (uint32_t)((const uint16_t *)base)[idx] << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

static float orc_load_f32(const void *base, int dtype, int64_t idx)
{
    return (float)orc_load(base, dtype, idx);
}

/* ------------------------------------------------------------------------------ */
/* Packing offsets: exclusive prefix sum of the per-request slot counts k_i
 * ([DScale] SIII-C, Flat-buffer packer; Fig. 6 gives k = [6,10,7,9] -> [0,6,16,23], 32). */
void orc_offsets(const int32_t *k, int32_t n, int32_t *cu)
{
    cu[0] = 0;
    for (int32_t i = 0; i < n; ++i)
        cu[i + 1] = cu[i] + k[i];
}

/* ------------------------------------------------------------------------------ */
/* Attention over packed candidate rows.                                          */

typedef struct {
    int dtype;
    int32_t n, hq, hkv, d;
    double scale;
    const void *q, *k_new, *v_new;   /* [m_cap, hq, d], [m_cap, hkv, d] x2        */
    int paged;
    const void *k_ctx, *v_ctx;       /* contiguous: [sum L, hkv, d]                */
    const int64_t *cu_ctx;           /* contiguous: [n + 1] token offsets          */
    const int32_t *block_table;      /* paged: [n, max_pages]                      */
    int32_t max_pages, page_size;
    int64_t s_page, s_head, s_tok;   /* paged cache strides, in elements           */
    const int32_t *ctx_len;          /* [n]                                        */
    const int32_t *cu_slots;         /* [n + 1]                                    */
    const uint8_t *want;             /* optional [n]: compute request i iff want[i] */
    double *out;                     /* [m_cap, hq, d]                              */
    double *lse;                     /* [m_cap, hq] (nullable)                      */
    /* work distribution over (request, q head) items */
    int64_t n_items;
    int64_t next_item;
    pthread_mutex_t lock;
} orc_attn_job;

/* Element e of context key (or value) token t of request i, KV head g. */
static double orc_ctx_elem(const orc_attn_job *J, const void *base, int32_t i, int32_t g,
                           int64_t t, int32_t e)
{
    if (!J->paged) {
        int64_t row = J->cu_ctx[i] + t;
        return orc_load(base, J->dtype, (row * J->hkv + g) * J->d + e);
    }
    int64_t page = J->block_table[(int64_t)i * J->max_pages + t / J->page_size];
    int64_t slot = t % J->page_size;
    return orc_load(base, J->dtype, page * J->s_page + g * J->s_head + slot * J->s_tok + e);
}

/* One (request i, query head h): every candidate row j of the request. */
static void orc_attn_item(orc_attn_job *J, int32_t i, int32_t h, double *s_buf)
{
    const int32_t G = J->hq / J->hkv;
    const int32_t g = h / G;
    const int32_t d = J->d;
    const int32_t off = J->cu_slots[i];
    const int32_t k = J->cu_slots[i + 1] - off;
    const int64_t L = J->ctx_len[i];

    for (int32_t j = 0; j < k; ++j) {
        const int64_t qrow = ((int64_t)(off + j) * J->hq + h) * d;
        const int64_t n_keys = L + j + 1;   /* context, then candidates 0..j */

        /* scores */
        double m = -INFINITY;
        for (int64_t t = 0; t < n_keys; ++t) {
            double dot = 0.0;
            for (int32_t e = 0; e < d; ++e) {
                double kv;
                if (t < L)
                    kv = orc_ctx_elem(J, J->k_ctx, i, g, t, e);
                else
                    kv = orc_load(J->k_new, J->dtype,
                                  ((int64_t)(off + (t - L)) * J->hkv + g) * d + e);
                dot += orc_load(J->q, J->dtype, qrow + e) * kv;
            }
            s_buf[t] = J->scale * dot;
            if (s_buf[t] > m)
                m = s_buf[t];
        }

        /* softmax weights and weighted sum of values */
        double denom = 0.0;
        double *o = J->out + qrow;
        for (int32_t e = 0; e < d; ++e)
            o[e] = 0.0;
        for (int64_t t = 0; t < n_keys; ++t) {
            const double p = exp(s_buf[t] - m);
            denom += p;
            for (int32_t e = 0; e < d; ++e) {
                double vv;
                if (t < L)
                    vv = orc_ctx_elem(J, J->v_ctx, i, g, t, e);
                else
                    vv = orc_load(J->v_new, J->dtype,
                                  ((int64_t)(off + (t - L)) * J->hkv + g) * d + e);
                o[e] += p * vv;
            }
        }
        for (int32_t e = 0; e < d; ++e)
            o[e] /= denom;
        if (J->lse)
            J->lse[(int64_t)(off + j) * J->hq + h] = m + log(denom);
    }
}

static void *orc_attn_worker(void *arg)
{
    orc_attn_job *J = (orc_attn_job *)arg;
    int64_t max_keys = 1;
    for (int32_t i = 0; i < J->n; ++i) {
        int64_t nk = (int64_t)J->ctx_len[i] + (J->cu_slots[i + 1] - J->cu_slots[i]);
        if (nk > max_keys)
            max_keys = nk;
    }
    double *s_buf = (double *)malloc(sizeof(double) * (size_t)max_keys);
    if (!s_buf)
        return (void *)1;
    for (;;) {
        pthread_mutex_lock(&J->lock);
        int64_t it = J->next_item++;
        pthread_mutex_unlock(&J->lock);
        if (it >= J->n_items)
            break;
        int32_t i = (int32_t)(it / J->hq);
        int32_t h = (int32_t)(it % J->hq);
        if (J->want && !J->want[i])
            continue;
        orc_attn_item(J, i, h, s_buf);
    }
    free(s_buf);
    return NULL;
}

/* Returns 0 on success, nonzero on a bad argument or allocation failure. */
int orc_attention(int dtype, int32_t n, int32_t hq, int32_t hkv, int32_t d, double scale,
                  const void *q, const void *k_new, const void *v_new,
                  int paged, const void *k_ctx, const void *v_ctx, const int64_t *cu_ctx,
                  const int32_t *block_table, int32_t max_pages, int32_t page_size,
                  int64_t s_page, int64_t s_head, int64_t s_tok,
                  const int32_t *ctx_len, const int32_t *cu_slots, const uint8_t *want,
                  int32_t threads, double *out, double *lse)
{
    if (n < 0 || hq <= 0 || hkv <= 0 || hq % hkv != 0 || d <= 0)
        return 1;
    if (dtype != ORC_F32 && dtype != ORC_BF16)
        return 1;
    if (paged && page_size <= 0)
        return 1;
    orc_attn_job J;
    memset(&J, 0, sizeof J);
    J.dtype = dtype; J.n = n; J.hq = hq; J.hkv = hkv; J.d = d; J.scale = scale;
    J.q = q; J.k_new = k_new; J.v_new = v_new;
    J.paged = paged; J.k_ctx = k_ctx; J.v_ctx = v_ctx; J.cu_ctx = cu_ctx;
    J.block_table = block_table; J.max_pages = max_pages; J.page_size = page_size;
    J.s_page = s_page; J.s_head = s_head; J.s_tok = s_tok;
    J.ctx_len = ctx_len; J.cu_slots = cu_slots; J.want = want;
    J.out = out; J.lse = lse;
    J.n_items = (int64_t)n * hq;
    J.next_item = 0;
    pthread_mutex_init(&J.lock, NULL);

    if (threads < 1)
        threads = 1;
    int rc = 0;
    pthread_t *tid = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)threads);
    if (!tid) {
        pthread_mutex_destroy(&J.lock);
        return 2;
    }
    int started = 0;
    for (int32_t t = 0; t < threads; ++t) {
        if (pthread_create(&tid[t], NULL, orc_attn_worker, &J) != 0)
            break;
        ++started;
    }
    if (started == 0)
        rc = (orc_attn_worker(&J) != NULL) ? 2 : 0;
    for (int t = 0; t < started; ++t) {
        void *ret = NULL;
        pthread_join(tid[t], &ret);
        if (ret)
            rc = 2;
    }
    free(tid);
    pthread_mutex_destroy(&J.lock);
    return rc;
}

/* ------------------------------------------------------------------------------ */
/* Row top-1 / top-2 / margin ([MiniLab] DFlash7-ACT top-1/top-2 draft-logit margin;
 * [DScale] SII-B, Top1-Top2 logit gap).  One scalar pass over the row:
 *   top1      = the largest value; top1_idx = its smallest index;
 *   top2      = the second element of the row sorted descending as a multiset
 *               (a repeated maximum gives top2 == top1);
 *   margin    = top1 - top2, evaluated in fp32 so that it is bit-comparable. */
void orc_row_top2(int dtype, const void *logits, int64_t row_stride, int32_t rows,
                  int32_t vocab, int32_t *top1_idx, float *top1, float *top2, float *margin)
{
    for (int32_t r = 0; r < rows; ++r) {
        const int64_t base = (int64_t)r * row_stride;
        float v1 = orc_load_f32(logits, dtype, base);
        int32_t i1 = 0;
        float v2 = -INFINITY;
        for (int32_t e = 1; e < vocab; ++e) {
            float x = orc_load_f32(logits, dtype, base + e);
            if (x > v1) {
                v2 = v1;
                v1 = x;
                i1 = e;
            } else if (x > v2) {
                v2 = x;
            }
        }
        volatile float a = v1, b = v2;   /* keep the subtraction in fp32 */
        if (top1_idx) top1_idx[r] = i1;
        if (top1) top1[r] = v1;
        if (top2) top2[r] = v2;
        if (margin) margin[r] = a - b;
    }
}

/* ------------------------------------------------------------------------------ */
/* Greedy prefix acceptance ([DScale] SIII-D, Prefix verifier at temperature 0;
 * [MiniLab] "accept exact prefix").  For request i with k_i = cu[i+1] - cu[i] slots:
 *   draft j (1 <= j < k_i) sits in row off_i + j and is accepted iff it equals the
 *   target argmax of row off_i + j - 1; a_i is the longest accepted prefix;
 *   accept_len = 1 + a_i (the anchor counts); next_token = argmax of row off_i + a_i.
 *   k_i = 0 (inactive request): accept_len = 0 and next_token = -1. */
void orc_greedy_accept(const int32_t *target_argmax, const int32_t *tokens,
                       const int32_t *cu_slots, int32_t n, int32_t *accept_len,
                       int32_t *next_token)
{
    for (int32_t i = 0; i < n; ++i) {
        const int32_t off = cu_slots[i];
        const int32_t k = cu_slots[i + 1] - off;
        if (k <= 0) {
            accept_len[i] = 0;
            next_token[i] = -1;
            continue;
        }
        int32_t a = 0;
        while (a + 1 < k && tokens[off + a + 1] == target_argmax[off + a])
            ++a;
        accept_len[i] = 1 + a;
        next_token[i] = target_argmax[off + a];
    }
}
