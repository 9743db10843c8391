/*
 * mla_oracle.c -- plain fp64 CPU oracle for paged MLA decode.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path links, loads or
 * calls this file: only the tests, the smoke check and the benchmark's CPU
 * baseline leg do.  It shares no code, header, table or helper with the CUDA
 * library; it is deliberately slow and written to be checked by eye.
 *
 * Sources (web pages; cited by title and section):
 *   [Overview]  "[DeepSeek-3] FlashMLA：把 MLA 的 KV Cache 优势变成 GPU 吞吐"
 *   [DeepDive]  "FlashMLA 新内核深度解析：Seesaw 调度、细粒度 TMA 流水线与
 *                H800 上的 660 TFlops MLA 解码"
 *   [SplitKV]   "CUTLASS 从零重写 FlashAttention：Split KV 并行优化实战"
 *   [AttnBook]  "3.4 Attention kernel" (LLM learning path, part 3)
 *
 * What is computed (the plain definition, [Overview] sec. 3 "一个 576 维缓存
 * 为什么同时充当 K 和 V" and sec. 4 "Paged KV Cache"):
 *   For request i, query token s, head h (row rho = s*h_q + h):
 *     visible keys  V = { t < L_i : not causal, or t <= L_i - s_q + s }
 *     kv_t          = k_cache[block_table[i][t / page]][t % page][0][:]
 *     x_t           = scale * sum_{c<d} q[i][s][h][c] * kv_t[c]
 *     lse[i][h][s]  = M + ln sum_t exp(x_t - M),  M = max_t x_t
 *     out[i][s][h]  = sum_t exp(x_t - lse) * kv_t[0:dv]
 *   The causal rule is the bottom-right aligned lower triangle of [AttnBook]
 *   "代码" (tril with diagonal offset len(K) - N).  An empty visible set gives
 *   out = 0 ([SplitKV] sec. 3.3) and lse = -inf (the identity of the merge).
 *   lse is the natural log of the sum of exp(scaled score) ([AttnBook]
 *   "FlashAttention:分块", step 3: m + log l).
 *
 * Parity status: every function here is pinned by the CPU tests against
 * closed forms, library routines, brute force and worked numbers from the
 * pages.  No function is "parity unpinned".
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* bf16 -> double: a bf16 value is the top 16 bits of an IEEE binary32. */
static double bf16_to_double(uint16_t bits) {
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

typedef struct {
    const uint16_t *q;           /* [b][s_q][h_q][d]            */
    const uint16_t *kv;          /* [num_pages][page][d] (h_kv=1) */
    const int32_t *block_table;  /* [b][max_blocks]             */
    const int32_t *seqlens;      /* [b]                          */
    int b, s_q, h_q, d, dv, page, max_blocks, num_pages;
    double scale;
    int causal;
} problem_t;

/* Pointer to the cached row of logical token t of request i, or NULL when the
 * block table points outside the cache (the caller reports an error). */
static const uint16_t *kv_row(const problem_t *P, int i, int t) {
    int32_t phys = P->block_table[(int64_t)i * P->max_blocks + t / P->page];
    if (phys < 0 || phys >= P->num_pages) return NULL;
    return P->kv + ((int64_t)phys * P->page + (t % P->page)) * P->d;
}

/* Number of keys the row of query token s of request i may see: keys
 * t < limit are visible ([AttnBook] "代码": tril(k = len(K) - N)). */
static int visible_limit(const problem_t *P, int i, int s) {
    int L = P->seqlens[i];
    if (L < 0) L = 0;
    if (!P->causal) return L;
    int lim = L - P->s_q + s + 1;
    if (lim < 0) lim = 0;
    if (lim > L) lim = L;
    return lim;
}

/* Scaled score x_t = scale * q_row . kv_t over the full d (K uses all d
 * dims; [Overview] sec. 3). */
static double score(const problem_t *P, const uint16_t *qrow, const uint16_t *kvt) {
    double acc = 0.0;
    for (int c = 0; c < P->d; ++c) acc += bf16_to_double(qrow[c]) * bf16_to_double(kvt[c]);
    return P->scale * acc;
}

/* Attention of one row restricted to keys t in [t_begin, t_end) that are also
 * visible.  Two passes: the max, then the sums.  Writes o[dv] (normalised) and
 * *lse.  Returns 0, or -1 on a block-table entry outside the cache. */
static int attend_range(const problem_t *P, int i, int rho, int t_begin, int t_end,
                        double *xbuf, double *o, double *lse) {
    int s = rho / P->h_q;
    const uint16_t *qrow = P->q + ((int64_t)i * P->s_q * P->h_q + rho) * P->d;
    int lim = visible_limit(P, i, s);
    if (t_end > lim) t_end = lim;
    if (t_begin < 0) t_begin = 0;
    for (int c = 0; c < P->dv; ++c) o[c] = 0.0;
    if (t_end <= t_begin) {
        *lse = -INFINITY;
        return 0;
    }
    double M = -INFINITY;
    for (int t = t_begin; t < t_end; ++t) {
        const uint16_t *kvt = kv_row(P, i, t);
        if (!kvt) return -1;
        xbuf[t - t_begin] = score(P, qrow, kvt);
        if (xbuf[t - t_begin] > M) M = xbuf[t - t_begin];
    }
    double sum = 0.0;
    for (int t = t_begin; t < t_end; ++t) sum += exp(xbuf[t - t_begin] - M);
    double l = M + log(sum);
    for (int t = t_begin; t < t_end; ++t) {
        double w = exp(xbuf[t - t_begin] - l);
        const uint16_t *kvt = kv_row(P, i, t);
        for (int c = 0; c < P->dv; ++c) o[c] += w * bf16_to_double(kvt[c]);
    }
    *lse = l;
    return 0;
}

/* ---- multi-threaded driver over a list of (request, row) units ---- */

typedef struct {
    const problem_t *P;
    const int32_t *units; /* pairs (i, rho) */
    int64_t n_units, u0, u1;
    double *out; /* [n_units][dv] */
    double *lse; /* [n_units]     */
    int status;
} job_t;

static void *run_job(void *arg) {
    job_t *J = (job_t *)arg;
    const problem_t *P = J->P;
    int maxL = 0;
    for (int i = 0; i < P->b; ++i)
        if (P->seqlens[i] > maxL) maxL = P->seqlens[i];
    double *xbuf = (double *)malloc(sizeof(double) * (size_t)(maxL > 0 ? maxL : 1));
    if (!xbuf) {
        J->status = -2;
        return NULL;
    }
    for (int64_t u = J->u0; u < J->u1; ++u) {
        int i = J->units[2 * u], rho = J->units[2 * u + 1];
        if (attend_range(P, i, rho, 0, P->seqlens[i], xbuf, J->out + u * P->dv, J->lse + u) != 0)
            J->status = -1;
    }
    free(xbuf);
    return NULL;
}

static int check_problem(const problem_t *P) {
    if (P->b < 0 || P->s_q <= 0 || P->h_q <= 0 || P->d <= 0 || P->dv <= 0 || P->dv > P->d ||
        P->page <= 0 || P->max_blocks < 0 || P->num_pages < 0)
        return -3;
    for (int i = 0; i < P->b; ++i)
        if (P->seqlens[i] > (int64_t)P->max_blocks * P->page) return -4;
    return 0;
}

/*
 * oracle_mla_decode_rows: the definition above for an explicit list of units
 * (request i, row rho = s*h_q + h).  out_rows is [n_units][dv], lse_rows
 * [n_units].  nthreads >= 1 splits the list into contiguous slices; the
 * arithmetic of each unit does not depend on it.
 * Returns 0; -1 block table outside the cache; -2 out of memory; -3 bad
 * sizes; -4 a sequence longer than its block-table row.
 */
int oracle_mla_decode_rows(const uint16_t *q, const uint16_t *kv, const int32_t *block_table,
                           const int32_t *seqlens, int b, int s_q, int h_q, int d, int dv, int page,
                           int max_blocks, int num_pages, double scale, int causal,
                           const int32_t *units, int64_t n_units, double *out_rows,
                           double *lse_rows, int nthreads) {
    problem_t P = {q, kv, block_table, seqlens, b, s_q, h_q, d, dv, page, max_blocks, num_pages,
                   scale, causal};
    int st = check_problem(&P);
    if (st) return st;
    for (int64_t u = 0; u < n_units; ++u) {
        if (units[2 * u] < 0 || units[2 * u] >= b || units[2 * u + 1] < 0 ||
            units[2 * u + 1] >= s_q * h_q)
            return -3;
    }
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    if ((int64_t)nthreads > n_units) nthreads = n_units > 0 ? (int)n_units : 1;
    pthread_t th[256];
    job_t jobs[256];
    for (int k = 0; k < nthreads; ++k) {
        jobs[k].P = &P;
        jobs[k].units = units;
        jobs[k].n_units = n_units;
        jobs[k].u0 = n_units * k / nthreads;
        jobs[k].u1 = n_units * (k + 1) / nthreads;
        jobs[k].out = out_rows;
        jobs[k].lse = lse_rows;
        jobs[k].status = 0;
    }
    if (nthreads == 1) {
        run_job(&jobs[0]);
    } else {
        for (int k = 0; k < nthreads; ++k) pthread_create(&th[k], NULL, run_job, &jobs[k]);
        for (int k = 0; k < nthreads; ++k) pthread_join(th[k], NULL);
    }
    for (int k = 0; k < nthreads; ++k)
        if (jobs[k].status) return jobs[k].status;
    return 0;
}

/*
 * oracle_mla_decode: every row of every request.  out is [b][s_q][h_q][dv]
 * (row-major), lse is [b][h_q][s_q] -- note the transpose of lse relative to
 * out, as in the output shapes of [Overview] sec. 3.
 */
int oracle_mla_decode(const uint16_t *q, const uint16_t *kv, const int32_t *block_table,
                      const int32_t *seqlens, int b, int s_q, int h_q, int d, int dv, int page,
                      int max_blocks, int num_pages, double scale, int causal, double *out,
                      double *lse, int nthreads) {
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
    int st = oracle_mla_decode_rows(q, kv, block_table, seqlens, b, s_q, h_q, d, dv, page,
                                    max_blocks, num_pages, scale, causal, units, n, out, lrow,
                                    nthreads);
    if (st == 0) {
        for (int64_t u = 0; u < n; ++u) {
            int i = (int)(u / R), rho = (int)(u % R), s = rho / h_q, h = rho % h_q;
            lse[((int64_t)i * h_q + h) * s_q + s] = lrow[u];
        }
    }
    free(units);
    free(lrow);
    return st;
}

/*
 * oracle_mla_partial: Split-KV partial result of one row over the key range
 * [t_begin, t_end) ([AttnBook] "解码 attention 与 Flash-Decoding"; [Overview]
 * sec. 6): o[dv] is the partial output already divided by its own sum, lse its
 * log-sum-exp.  A range with no visible key gives o = 0, lse = -inf
 * ([SplitKV] sec. 3.2, the fully masked split).
 */
int oracle_mla_partial(const uint16_t *q, const uint16_t *kv, const int32_t *block_table,
                       const int32_t *seqlens, int b, int s_q, int h_q, int d, int dv, int page,
                       int max_blocks, int num_pages, double scale, int causal, int i, int rho,
                       int t_begin, int t_end, double *o, double *lse) {
    problem_t P = {q, kv, block_table, seqlens, b, s_q, h_q, d, dv, page, max_blocks, num_pages,
                   scale, causal};
    int st = check_problem(&P);
    if (st) return st;
    if (i < 0 || i >= b || rho < 0 || rho >= s_q * h_q) return -3;
    int n = t_end - t_begin;
    double *xbuf = (double *)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
    if (!xbuf) return -2;
    st = attend_range(&P, i, rho, t_begin, t_end, xbuf, o, lse);
    free(xbuf);
    return st;
}

/*
 * oracle_merge_pair: the two-way merge of unnormalised partial states
 * ([AttnBook] "在线 softmax", last paragraph; [Overview] sec. 7):
 *   m = max(m1, m2); l = e^{m1-m} l1 + e^{m2-m} l2; o~ = e^{m1-m} o~1 + e^{m2-m} o~2.
 * A state with l == 0 (nothing seen, m = -inf) is skipped, as [SplitKV]
 * sec. 3.2 prescribes, so that exp(-inf - (-inf)) never appears.
 * In/out: (m1, l1, o1[dv]) is updated in place with (m2, l2, o2).
 */
void oracle_merge_pair(double *m1, double *l1, double *o1, double m2, double l2, const double *o2,
                       int dv) {
    if (l2 == 0.0) return;
    if (*l1 == 0.0) {
        *m1 = m2;
        *l1 = l2;
        for (int c = 0; c < dv; ++c) o1[c] = o2[c];
        return;
    }
    double m = *m1 > m2 ? *m1 : m2;
    double a = exp(*m1 - m), bb = exp(m2 - m);
    *l1 = a * (*l1) + bb * l2;
    for (int c = 0; c < dv; ++c) o1[c] = a * o1[c] + bb * o2[c];
    *m1 = m;
}

/*
 * oracle_lse_combine: the n-way combine of normalised partials (o_k, lse_k)
 * ([DeepDive] "Programmatic Dependent Launch", the combine paragraph): take
 * the max lse, weight each partial by exp(lse_k - max), sum, normalise, and
 * the final lse is max + log(sum of weights).  All partials empty (every
 * lse_k = -inf) gives o = 0, lse = -inf ([SplitKV] sec. 3.3).
 * lse_parts[n], o_parts[n][dv] -> o[dv], *lse.
 */
void oracle_lse_combine(int n, const double *lse_parts, const double *o_parts, int dv, double *o,
                        double *lse) {
    double M = -INFINITY;
    for (int k = 0; k < n; ++k)
        if (lse_parts[k] > M) M = lse_parts[k];
    for (int c = 0; c < dv; ++c) o[c] = 0.0;
    if (M == -INFINITY) {
        *lse = -INFINITY;
        return;
    }
    double wsum = 0.0;
    for (int k = 0; k < n; ++k) {
        if (lse_parts[k] == -INFINITY) continue;
        double w = exp(lse_parts[k] - M);
        wsum += w;
        for (int c = 0; c < dv; ++c) o[c] += w * o_parts[(int64_t)k * dv + c];
    }
    for (int c = 0; c < dv; ++c) o[c] /= wsum;
    *lse = M + log(wsum);
}
