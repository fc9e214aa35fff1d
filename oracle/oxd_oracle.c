/*
 * Oracle for batched paged-KV decode attention -- TEST INFRASTRUCTURE ONLY.
 * See oxd_oracle.h for the definition it restates and where it comes from.
 *
 * Deliberately plain: one query head at a time, tokens visited in logical
 * order (page by page through the block table, then token by token inside a
 * page), every bf16 widened exactly to double, every sum in double, no
 * blocking, no online rescaling, no fusion. Threads only split the list of
 * independent query heads, so the result does not depend on the thread count.
 */
#include "oxd_oracle.h"

#include <math.h>
#include <pthread.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

/* bf16 is the upper half of an IEEE binary32; widening is exact. */
static double bf16_to_f64(uint16_t bits) {
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Element offset of (page, token t, kv head h, dim d) in a K or V pool. */
static size_t pool_offset(int layout, int64_t page, int t, int h, int d, int page_size, int Hkv,
                          int D) {
    if (layout == ORACLE_LAYOUT_NHD)
        return (((size_t)page * (size_t)page_size + (size_t)t) * (size_t)Hkv + (size_t)h) *
                   (size_t)D +
               (size_t)d;
    return (((size_t)page * (size_t)Hkv + (size_t)h) * (size_t)page_size + (size_t)t) *
               (size_t)D +
           (size_t)d;
}

int64_t oracle_kv_len(const int32_t* indptr, const int32_t* last_page_len, int page_size, int b) {
    int64_t pages = (int64_t)indptr[b + 1] - (int64_t)indptr[b];
    return (pages - 1) * (int64_t)page_size + (int64_t)last_page_len[b];
}

/* Checks the block tables the way the definition needs them. */
static int check_tables(int B, int page_size, int64_t num_pages, const int32_t* indptr,
                        const int32_t* indices, const int32_t* last_page_len) {
    for (int b = 0; b < B; ++b) {
        if (indptr[b + 1] - indptr[b] < 1) return ORACLE_EINVAL;
        if (last_page_len[b] < 1 || last_page_len[b] > page_size) return ORACLE_EINVAL;
        for (int32_t p = indptr[b]; p < indptr[b + 1]; ++p)
            if (indices[p] < 0 || (int64_t)indices[p] >= num_pages) return ORACLE_EINVAL;
    }
    return ORACLE_OK;
}

typedef struct {
    int B, Hq, Hkv, D, page_size, layout;
    const uint16_t *q, *k, *v;
    const int32_t *indptr, *indices, *last_page_len;
    double sm_scale;
} problem;

/*
 * Logits of head (b, hq) for logical tokens [t0, t1) of request b, written to
 * s[0 .. t1-t0). Logical token j lives in page indices[indptr[b] + j / ps] at
 * slot j % ps.
 */
static void logits(const problem* P, int b, int hq, int64_t t0, int64_t t1, double* s) {
    int G = P->Hq / P->Hkv;
    int h = hq / G; /* consecutive query heads share one KV head */
    const uint16_t* qrow = P->q + ((size_t)b * (size_t)P->Hq + (size_t)hq) * (size_t)P->D;
    for (int64_t j = t0; j < t1; ++j) {
        int64_t page = P->indices[P->indptr[b] + j / P->page_size];
        int t = (int)(j % P->page_size);
        double dot = 0.0;
        for (int d = 0; d < P->D; ++d)
            dot += bf16_to_f64(qrow[d]) *
                   bf16_to_f64(P->k[pool_offset(P->layout, page, t, h, d, P->page_size,
                                                P->Hkv, P->D)]);
        s[j - t0] = P->sm_scale * dot;
    }
}

/* Softmax-weighted mean of V over tokens [t0, t1) and its log-sum-exp. */
static int head_state(const problem* P, int b, int hq, int64_t t0, int64_t t1, double* o,
                      double* lse) {
    for (int d = 0; d < P->D; ++d) o[d] = 0.0;
    if (t1 <= t0) {
        *lse = -INFINITY;
        return ORACLE_OK;
    }
    int64_t n = t1 - t0;
    double* s = (double*)malloc((size_t)n * sizeof(double));
    if (!s) return ORACLE_ENOMEM;
    logits(P, b, hq, t0, t1, s);

    double M = -INFINITY;
    for (int64_t j = 0; j < n; ++j)
        if (s[j] > M) M = s[j];
    double Z = 0.0;
    for (int64_t j = 0; j < n; ++j) Z += exp(s[j] - M);

    int G = P->Hq / P->Hkv;
    int h = hq / G;
    for (int64_t j = 0; j < n; ++j) {
        double w = exp(s[j] - M) / Z;
        int64_t lj = t0 + j;
        int64_t page = P->indices[P->indptr[b] + lj / P->page_size];
        int t = (int)(lj % P->page_size);
        for (int d = 0; d < P->D; ++d)
            o[d] += w * bf16_to_f64(P->v[pool_offset(P->layout, page, t, h, d, P->page_size,
                                                     P->Hkv, P->D)]);
    }
    *lse = M + log(Z);
    free(s);
    return ORACLE_OK;
}

typedef struct {
    const problem* P;
    const int32_t* heads; /* NULL: all heads in (b, hq) order */
    int n_heads;
    int worker, nworkers;
    double *out, *lse;
    int status;
} job;

static void* run_job(void* arg) {
    job* J = (job*)arg;
    const problem* P = J->P;
    J->status = ORACLE_OK;
    for (int i = J->worker; i < J->n_heads; i += J->nworkers) {
        int b, hq;
        if (J->heads) {
            b = J->heads[2 * i];
            hq = J->heads[2 * i + 1];
        } else {
            b = i / P->Hq;
            hq = i % P->Hq;
        }
        int64_t L = oracle_kv_len(P->indptr, P->last_page_len, P->page_size, b);
        int rc = head_state(P, b, hq, 0, L, J->out + (size_t)i * (size_t)P->D, J->lse + i);
        if (rc != ORACLE_OK) {
            J->status = rc;
            return NULL;
        }
    }
    return NULL;
}

static int check_shape(int B, int Hq, int Hkv, int D, int page_size, int layout) {
    if (B < 1 || Hq < 1 || Hkv < 1 || D < 1 || page_size < 1) return ORACLE_EINVAL;
    if (Hq % Hkv != 0) return ORACLE_EINVAL;
    if (layout != ORACLE_LAYOUT_NHD && layout != ORACLE_LAYOUT_HND) return ORACLE_EINVAL;
    return ORACLE_OK;
}

int oracle_paged_decode_f64(int B, int Hq, int Hkv, int D, int page_size, int layout,
                            int64_t num_pages, const uint16_t* q, const uint16_t* k,
                            const uint16_t* v, const int32_t* indptr, const int32_t* indices,
                            const int32_t* last_page_len, double sm_scale,
                            const int32_t* heads, int n_heads, double* out, double* lse,
                            int nthreads) {
    if (check_shape(B, Hq, Hkv, D, page_size, layout) != ORACLE_OK) return ORACLE_EINVAL;
    if (check_tables(B, page_size, num_pages, indptr, indices, last_page_len) != ORACLE_OK)
        return ORACLE_EINVAL;
    if (heads) {
        for (int i = 0; i < n_heads; ++i)
            if (heads[2 * i] < 0 || heads[2 * i] >= B || heads[2 * i + 1] < 0 ||
                heads[2 * i + 1] >= Hq)
                return ORACLE_EINVAL;
    } else {
        n_heads = B * Hq;
    }
    problem P = {B, Hq, Hkv, D, page_size, layout, q, k, v, indptr, indices, last_page_len,
                 sm_scale};

    if (nthreads <= 0) nthreads = (int)sysconf(_SC_NPROCESSORS_ONLN);
    if (nthreads < 1) nthreads = 1;
    if (nthreads > n_heads) nthreads = n_heads > 0 ? n_heads : 1;

    job* jobs = (job*)calloc((size_t)nthreads, sizeof(job));
    pthread_t* tids = (pthread_t*)calloc((size_t)nthreads, sizeof(pthread_t));
    if (!jobs || !tids) {
        free(jobs);
        free(tids);
        return ORACLE_ENOMEM;
    }
    for (int w = 0; w < nthreads; ++w) {
        jobs[w] = (job){&P, heads, n_heads, w, nthreads, out, lse, ORACLE_OK};
        if (w > 0) pthread_create(&tids[w], NULL, run_job, &jobs[w]);
    }
    run_job(&jobs[0]);
    int status = jobs[0].status;
    for (int w = 1; w < nthreads; ++w) {
        pthread_join(tids[w], NULL);
        if (jobs[w].status != ORACLE_OK) status = jobs[w].status;
    }
    free(jobs);
    free(tids);
    return status;
}

int oracle_partial_state_f64(int B, int Hq, int Hkv, int D, int page_size, int layout,
                             int64_t num_pages, const uint16_t* q, const uint16_t* k,
                             const uint16_t* v, const int32_t* indptr, const int32_t* indices,
                             const int32_t* last_page_len, double sm_scale, int b, int hq,
                             int64_t tok_begin, int64_t tok_end, double* o, double* lse) {
    if (check_shape(B, Hq, Hkv, D, page_size, layout) != ORACLE_OK) return ORACLE_EINVAL;
    if (check_tables(B, page_size, num_pages, indptr, indices, last_page_len) != ORACLE_OK)
        return ORACLE_EINVAL;
    if (b < 0 || b >= B || hq < 0 || hq >= Hq) return ORACLE_EINVAL;
    int64_t L = oracle_kv_len(indptr, last_page_len, page_size, b);
    if (tok_begin < 0 || tok_end > L || tok_begin > tok_end) return ORACLE_EINVAL;
    problem P = {B, Hq, Hkv, D, page_size, layout, q, k, v, indptr, indices, last_page_len,
                 sm_scale};
    return head_state(&P, b, hq, tok_begin, tok_end, o, lse);
}

void oracle_merge_states_f64(int S, int D, const double* v, const double* s, double* out,
                             double* lse) {
    double M = -INFINITY;
    for (int i = 0; i < S; ++i)
        if (s[i] > M) M = s[i];
    for (int d = 0; d < D; ++d) out[d] = 0.0;
    if (M == -INFINITY) {
        *lse = -INFINITY;
        return;
    }
    double W = 0.0;
    for (int i = 0; i < S; ++i) W += exp(s[i] - M);
    for (int i = 0; i < S; ++i) {
        double w = exp(s[i] - M) / W;
        for (int d = 0; d < D; ++d) out[d] += w * v[(size_t)i * (size_t)D + (size_t)d];
    }
    *lse = M + log(W);
}

/* ------------------------------------------------------------------ causal prefill */

/*
 * State of one query row `qrow` (D values) against logical tokens [0, t1) of
 * request b through KV head h: the same definition as head_state, with the
 * query row given directly.
 */
static int row_state(const problem* P, const uint16_t* qrow, int b, int h, int64_t t1, double* o,
                     double* lse) {
    for (int d = 0; d < P->D; ++d) o[d] = 0.0;
    if (t1 <= 0) {
        *lse = -INFINITY;
        return ORACLE_OK;
    }
    double* s = (double*)malloc((size_t)t1 * sizeof(double));
    if (!s) return ORACLE_ENOMEM;
    for (int64_t j = 0; j < t1; ++j) {
        int64_t page = P->indices[P->indptr[b] + j / P->page_size];
        int t = (int)(j % P->page_size);
        double dot = 0.0;
        for (int d = 0; d < P->D; ++d)
            dot += bf16_to_f64(qrow[d]) *
                   bf16_to_f64(P->k[pool_offset(P->layout, page, t, h, d, P->page_size,
                                                P->Hkv, P->D)]);
        s[j] = P->sm_scale * dot;
    }
    double M = -INFINITY;
    for (int64_t j = 0; j < t1; ++j)
        if (s[j] > M) M = s[j];
    double Z = 0.0;
    for (int64_t j = 0; j < t1; ++j) Z += exp(s[j] - M);
    for (int64_t j = 0; j < t1; ++j) {
        double w = exp(s[j] - M) / Z;
        int64_t page = P->indices[P->indptr[b] + j / P->page_size];
        int t = (int)(j % P->page_size);
        for (int d = 0; d < P->D; ++d)
            o[d] += w * bf16_to_f64(P->v[pool_offset(P->layout, page, t, h, d, P->page_size,
                                                     P->Hkv, P->D)]);
    }
    *lse = M + log(Z);
    free(s);
    return ORACLE_OK;
}

typedef struct {
    const problem* P;
    const int32_t* qo_indptr;
    const int32_t* rows; /* NULL: every (t, hq) in order */
    int n_rows;
    int worker, nworkers;
    double *out, *lse;
    int status;
} prefill_job;

static void* run_prefill_job(void* arg) {
    prefill_job* J = (prefill_job*)arg;
    const problem* P = J->P;
    J->status = ORACLE_OK;
    for (int i = J->worker; i < J->n_rows; i += J->nworkers) {
        int t, hq;
        if (J->rows) {
            t = J->rows[2 * i];
            hq = J->rows[2 * i + 1];
        } else {
            t = i / P->Hq;
            hq = i % P->Hq;
        }
        /* the request that owns query token t */
        int b = 0;
        while (J->qo_indptr[b + 1] <= t) ++b;
        const int64_t L = oracle_kv_len(P->indptr, P->last_page_len, P->page_size, b);
        const int64_t q_len = (int64_t)J->qo_indptr[b + 1] - J->qo_indptr[b];
        const int64_t pos = L - q_len + (t - J->qo_indptr[b]);
        const int G = P->Hq / P->Hkv;
        const uint16_t* qrow = P->q + ((size_t)t * (size_t)P->Hq + (size_t)hq) * (size_t)P->D;
        int rc = row_state(P, qrow, b, hq / G, pos + 1, J->out + (size_t)i * (size_t)P->D,
                           J->lse + i);
        if (rc != ORACLE_OK) {
            J->status = rc;
            return NULL;
        }
    }
    return NULL;
}

int oracle_paged_prefill_f64(int B, int Hq, int Hkv, int D, int page_size, int layout,
                             int64_t num_pages, const uint16_t* q, const uint16_t* k,
                             const uint16_t* v, const int32_t* qo_indptr, const int32_t* indptr,
                             const int32_t* indices, const int32_t* last_page_len,
                             double sm_scale, const int32_t* rows, int n_rows, double* out,
                             double* lse, int nthreads) {
    if (check_shape(B, Hq, Hkv, D, page_size, layout) != ORACLE_OK) return ORACLE_EINVAL;
    if (check_tables(B, page_size, num_pages, indptr, indices, last_page_len) != ORACLE_OK)
        return ORACLE_EINVAL;
    if (qo_indptr[0] != 0) return ORACLE_EINVAL;
    for (int b = 0; b < B; ++b) {
        const int64_t q_len = (int64_t)qo_indptr[b + 1] - qo_indptr[b];
        if (q_len < 0 || q_len > oracle_kv_len(indptr, last_page_len, page_size, b))
            return ORACLE_EINVAL;
    }
    const int64_t n_tok = qo_indptr[B];
    if (rows) {
        for (int i = 0; i < n_rows; ++i)
            if (rows[2 * i] < 0 || rows[2 * i] >= n_tok || rows[2 * i + 1] < 0 ||
                rows[2 * i + 1] >= Hq)
                return ORACLE_EINVAL;
    } else {
        if (n_tok * Hq > 0x7fffffff) return ORACLE_EINVAL;
        n_rows = (int)(n_tok * Hq);
    }
    problem P = {B, Hq, Hkv, D, page_size, layout, q, k, v, indptr, indices, last_page_len,
                 sm_scale};
    if (nthreads <= 0) nthreads = (int)sysconf(_SC_NPROCESSORS_ONLN);
    if (nthreads < 1) nthreads = 1;
    if (nthreads > n_rows) nthreads = n_rows > 0 ? n_rows : 1;
    prefill_job* jobs = (prefill_job*)calloc((size_t)nthreads, sizeof(prefill_job));
    pthread_t* tids = (pthread_t*)calloc((size_t)nthreads, sizeof(pthread_t));
    if (!jobs || !tids) {
        free(jobs);
        free(tids);
        return ORACLE_ENOMEM;
    }
    for (int w = 0; w < nthreads; ++w) {
        jobs[w] = (prefill_job){&P, qo_indptr, rows, n_rows, w, nthreads, out, lse, ORACLE_OK};
        if (w > 0) pthread_create(&tids[w], NULL, run_prefill_job, &jobs[w]);
    }
    run_prefill_job(&jobs[0]);
    int status = jobs[0].status;
    for (int w = 1; w < nthreads; ++w) {
        pthread_join(tids[w], NULL);
        if (jobs[w].status != ORACLE_OK) status = jobs[w].status;
    }
    free(jobs);
    free(tids);
    return status;
}

/* ------------------------------------------------------------------ RoPE and append */

void oracle_rope_f64(int n, int D, const double* x, const int32_t* pos, double theta, double* y) {
    const int h = D / 2;
    for (int r = 0; r < n; ++r) {
        const double* xr = x + (size_t)r * (size_t)D;
        double* yr = y + (size_t)r * (size_t)D;
        for (int i = 0; i < h; ++i) {
            const double f = pow(theta, -2.0 * (double)i / (double)D);
            const double a = (double)pos[r] * f;
            const double c = cos(a), s = sin(a);
            yr[i] = xr[i] * c - xr[i + h] * s;
            yr[i + h] = xr[i + h] * c + xr[i] * s;
        }
    }
}

uint16_t oracle_f64_to_bf16(double x) {
    /* bfloat16: a sign bit, 8 exponent bits (bias 127) and 7 fraction bits,
     * so normal values carry 8 significant bits down to 2^-126 and below that
     * the numbers are multiples of 2^-133 (the subnormal step). The f64 value
     * is rounded once, to nearest with ties to even (nearbyint in the default
     * rounding mode): to 8 significant bits at or above 2^-126, to a multiple
     * of 2^-133 below it. The rounded value is exact in f32, whose upper 16
     * bits are then the bf16 pattern; a value that rounds to 2^128 or beyond
     * is an infinity. */
    double r;
    if (x == 0.0 || isnan(x) || isinf(x)) {
        r = x;
    } else if (fabs(x) < ldexp(1.0, -126)) {
        r = ldexp(nearbyint(ldexp(x, 133)), -133);
    } else {
        int e;
        const double m = frexp(x, &e);           /* x = m * 2^e, 0.5 <= |m| < 1 */
        r = ldexp(nearbyint(ldexp(m, 8)), e - 8);
    }
    if (fabs(r) >= ldexp(1.0, 128)) return (uint16_t)(signbit(r) ? 0xFF80u : 0x7F80u);
    const float f = (float)r;
    uint32_t u;
    memcpy(&u, &f, 4);
    return (uint16_t)(u >> 16);
}

int oracle_rope_append(int T, int B, int Hq, int Hkv, int D, int page_size, int layout,
                       int64_t num_pages, const uint16_t* q, const uint16_t* k,
                       const uint16_t* v, const int32_t* token_request, const int32_t* positions,
                       const int32_t* indptr, const int32_t* indices, const int32_t* refcount,
                       double theta, uint16_t* q_out, uint16_t* k_pages, uint16_t* v_pages,
                       int32_t* status) {
    if (T < 0 || B < 1 || Hq < 1 || Hkv < 1 || D < 2 || (D & 1) || page_size < 1 ||
        (layout != ORACLE_LAYOUT_NHD && layout != ORACLE_LAYOUT_HND) || num_pages < 1)
        return ORACLE_EINVAL;
    double* xr = (double*)malloc(sizeof(double) * (size_t)D);
    double* yr = (double*)malloc(sizeof(double) * (size_t)D);
    if (xr == NULL || yr == NULL) {
        free(xr);
        free(yr);
        return ORACLE_ENOMEM;
    }
    int not_written = 0;
    for (int t = 0; t < T; ++t) {
        const int32_t p = positions[t];
        /* q_out: every query head of the token, whatever happens to its KV */
        for (int hq = 0; hq < Hq; ++hq) {
            const size_t off = ((size_t)t * (size_t)Hq + (size_t)hq) * (size_t)D;
            for (int d = 0; d < D; ++d) xr[d] = bf16_to_f64(q[off + (size_t)d]);
            oracle_rope_f64(1, D, xr, &p, theta, yr);
            for (int d = 0; d < D; ++d) q_out[off + (size_t)d] = oracle_f64_to_bf16(yr[d]);
        }
        const int b = token_request[t];
        int st = ORACLE_APPEND_WRITTEN;
        int64_t page = -1;
        if (b < 0 || b >= B || p < 0 ||
            (int64_t)p >= ((int64_t)indptr[b + 1] - indptr[b]) * (int64_t)page_size) {
            st = ORACLE_APPEND_BAD_POSITION;
        } else {
            page = indices[indptr[b] + p / page_size];
            if (page < 0 || page >= num_pages)
                st = ORACLE_APPEND_BAD_PAGE;
            else if (refcount[page] != 1)
                st = ORACLE_APPEND_SHARED_PAGE;
        }
        status[t] = st;
        if (st != ORACLE_APPEND_WRITTEN) {
            ++not_written;
            continue;
        }
        const int slot = p % page_size;
        for (int h = 0; h < Hkv; ++h) {
            const size_t src = ((size_t)t * (size_t)Hkv + (size_t)h) * (size_t)D;
            const size_t dst = pool_offset(layout, page, slot, h, 0, page_size, Hkv, D);
            for (int d = 0; d < D; ++d) xr[d] = bf16_to_f64(k[src + (size_t)d]);
            oracle_rope_f64(1, D, xr, &p, theta, yr);
            for (int d = 0; d < D; ++d) {
                k_pages[dst + (size_t)d] = oracle_f64_to_bf16(yr[d]);
                v_pages[dst + (size_t)d] = v[src + (size_t)d];
            }
        }
    }
    free(xr);
    free(yr);
    return not_written;
}
