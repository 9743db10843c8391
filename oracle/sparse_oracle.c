/*
 * sparse_oracle.c -- plain fp64 CPU oracle for sparse MLA decode (attention
 * over per-query selected tokens).
 *
 * TEST INFRASTRUCTURE ONLY (as mla_oracle.c): nothing in the product path
 * links, loads or calls this file; it shares no code with the CUDA library.
 *
 * Source: "[DeepSeek-3] FlashMLA：把 MLA 的 KV Cache 优势变成 GPU 吞吐", sec. 11
 * (Sparse FlashMLA): an upper layer picks, for every query token, the top-k
 * cached tokens and passes their physical positions indices[b][s_q][topk],
 * index = page_id * page_block_size + offset, so no block table is needed;
 * the kernel only gathers those tokens and runs QK -> online softmax -> PV.
 * The row computation is the same as for dense decode (sec. 3: one 576-dim
 * cache row is K, its first dv dims are V):
 *   For request i, query token s, head h:
 *     keys   K = [ indices[i][s][k] : 0 <= k < topk, the index usable ]
 *     x_k    = scale * sum_{c<d} q[i][s][h][c] * kv[idx_k][c]
 *     lse[i][h][s] = M + ln sum_k exp(x_k - M),  M = max_k x_k
 *     out[i][s][h] = sum_k exp(x_k - lse) * kv[idx_k][0:dv]
 * Readings of what the page leaves open:
 *   - an index < 0 is padding: that slot contributes nothing;
 *   - an index >= num_pages * page points outside the cache: it contributes
 *     nothing and the call reports it (return -5);
 *   - a token listed twice counts twice (the list is attended as given);
 *   - no causal mask (the selector decides what a query may see);
 *   - an empty key list gives out = 0 and lse = -inf, as for an empty
 *     sequence in dense decode.
 *
 * Parity status: pinned by the CPU tests (equality with the
 * dense oracle when the indices list a request's tokens in order; duplicate
 * keys, padding, the empty list and out-of-range indices in closed form).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

static double sp_bf16(uint16_t bits) {
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

typedef struct {
    const uint16_t *q;       /* [b][s_q][h_q][d]          */
    const uint16_t *kv;      /* [num_pages * page][d]      */
    const int32_t *indices;  /* [b][s_q][topk]            */
    int b, s_q, h_q, topk, d, dv;
    int64_t num_tokens;      /* num_pages * page          */
    double scale;
} sparse_t;

/* One row; xbuf holds topk doubles.  Returns 0, or -5 when an index pointed
 * outside the cache (that key was left out). */
static int sparse_row(const sparse_t *P, int i, int s, int h, double *xbuf, double *o,
                      double *lse) {
    const uint16_t *qrow = P->q + (((int64_t)i * P->s_q + s) * P->h_q + h) * P->d;
    const int32_t *idx = P->indices + ((int64_t)i * P->s_q + s) * P->topk;
    int status = 0;
    double M = -INFINITY;
    for (int k = 0; k < P->topk; ++k) {
        xbuf[k] = NAN;  /* marks "not a key" */
        if (idx[k] < 0) continue;
        if ((int64_t)idx[k] >= P->num_tokens) {
            status = -5;
            continue;
        }
        const uint16_t *kvt = P->kv + (int64_t)idx[k] * P->d;
        double acc = 0.0;
        for (int c = 0; c < P->d; ++c) acc += sp_bf16(qrow[c]) * sp_bf16(kvt[c]);
        xbuf[k] = P->scale * acc;
        if (xbuf[k] > M) M = xbuf[k];
    }
    for (int c = 0; c < P->dv; ++c) o[c] = 0.0;
    if (M == -INFINITY) {
        *lse = -INFINITY;
        return status;
    }
    double sum = 0.0;
    for (int k = 0; k < P->topk; ++k)
        if (!isnan(xbuf[k])) sum += exp(xbuf[k] - M);
    double l = M + log(sum);
    for (int k = 0; k < P->topk; ++k) {
        if (isnan(xbuf[k])) continue;
        double w = exp(xbuf[k] - l);
        const uint16_t *kvt = P->kv + (int64_t)idx[k] * P->d;
        for (int c = 0; c < P->dv; ++c) o[c] += w * sp_bf16(kvt[c]);
    }
    *lse = l;
    return status;
}

typedef struct {
    const sparse_t *P;
    const int32_t *units; /* pairs (i, row = s*h_q + h) */
    int64_t u0, u1;
    double *out, *lse;
    int status;
} sp_job_t;

static void *sp_run(void *arg) {
    sp_job_t *J = (sp_job_t *)arg;
    const sparse_t *P = J->P;
    double *xbuf = (double *)malloc(sizeof(double) * (size_t)(P->topk > 0 ? P->topk : 1));
    if (!xbuf) {
        J->status = -2;
        return NULL;
    }
    for (int64_t u = J->u0; u < J->u1; ++u) {
        int i = J->units[2 * u], row = J->units[2 * u + 1];
        int st = sparse_row(P, i, row / P->h_q, row % P->h_q, xbuf, J->out + u * P->dv, J->lse + u);
        if (st && !J->status) J->status = st;
    }
    free(xbuf);
    return NULL;
}

/*
 * oracle_mla_sparse_rows: the definition above for a list of (request, row)
 * units.  Returns 0; -2 out of memory; -3 bad sizes; -5 an index outside the
 * cache (the results are still written, without that key).
 */
int oracle_mla_sparse_rows(const uint16_t *q, const uint16_t *kv, const int32_t *indices, int b,
                           int s_q, int h_q, int topk, int d, int dv, int64_t num_tokens,
                           double scale, const int32_t *units, int64_t n_units, double *out_rows,
                           double *lse_rows, int nthreads) {
    if (b < 0 || s_q <= 0 || h_q <= 0 || topk < 0 || d <= 0 || dv <= 0 || dv > d ||
        num_tokens < 0)
        return -3;
    for (int64_t u = 0; u < n_units; ++u)
        if (units[2 * u] < 0 || units[2 * u] >= b || units[2 * u + 1] < 0 ||
            units[2 * u + 1] >= s_q * h_q)
            return -3;
    sparse_t P = {q, kv, indices, b, s_q, h_q, topk, d, dv, num_tokens, scale};
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    if ((int64_t)nthreads > n_units) nthreads = n_units > 0 ? (int)n_units : 1;
    pthread_t th[256];
    sp_job_t jobs[256];
    for (int k = 0; k < nthreads; ++k) {
        jobs[k].P = &P;
        jobs[k].units = units;
        jobs[k].u0 = n_units * k / nthreads;
        jobs[k].u1 = n_units * (k + 1) / nthreads;
        jobs[k].out = out_rows;
        jobs[k].lse = lse_rows;
        jobs[k].status = 0;
    }
    if (nthreads == 1) {
        sp_run(&jobs[0]);
    } else {
        for (int k = 0; k < nthreads; ++k) pthread_create(&th[k], NULL, sp_run, &jobs[k]);
        for (int k = 0; k < nthreads; ++k) pthread_join(th[k], NULL);
    }
    int st = 0;
    for (int k = 0; k < nthreads; ++k) {
        if (jobs[k].status == -2) return -2;
        if (jobs[k].status) st = jobs[k].status;
    }
    return st;
}

/*
 * oracle_mla_sparse: every row.  out is [b][s_q][h_q][dv], lse [b][h_q][s_q]
 * (the dense decode's output shapes).
 */
int oracle_mla_sparse(const uint16_t *q, const uint16_t *kv, const int32_t *indices, int b,
                      int s_q, int h_q, int topk, int d, int dv, int64_t num_tokens, double scale,
                      double *out, double *lse, int nthreads) {
    int64_t R = (int64_t)s_q * h_q, n = (int64_t)b * R;
    int32_t *units = (int32_t *)malloc(sizeof(int32_t) * 2 * (size_t)(n > 0 ? n : 1));
    double *lrow = (double *)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
    if (!units || !lrow) {
        free(units);
        free(lrow);
        return -2;
    }
    for (int64_t u = 0; u < n; ++u) {
        units[2 * u] = (int32_t)(u / R);
        units[2 * u + 1] = (int32_t)(u % R);
    }
    int st = oracle_mla_sparse_rows(q, kv, indices, b, s_q, h_q, topk, d, dv, num_tokens, scale,
                                    units, n, out, lrow, nthreads);
    if (st == 0 || st == -5) {
        for (int64_t u = 0; u < n; ++u) {
            int i = (int)(u / R), row = (int)(u % R), s = row / h_q, h = row % h_q;
            lse[((int64_t)i * h_q + h) * s_q + s] = lrow[u];
        }
    }
    free(units);
    free(lrow);
    return st;
}
