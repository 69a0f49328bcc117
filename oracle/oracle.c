/*
 * oracle.c -- fp64 CPU oracle for exact attention (forward and backward).
 *
 * TEST INFRASTRUCTURE ONLY: loaded by the test suite, the smoke check and the
 * benchmark's CPU-baseline leg; never by the product path.  Plain C11 + pthreads,
 * deliberately slow and obvious: one query row at a time, the full score row and
 * probability row materialised, every sum a plain loop.  See oracle.h for the
 * definition and the sources it follows.
 */
#include "oracle.h"

#include <math.h>
#include <pthread.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

/* ------------------------------------------------------------------------- */
/* input access                                                              */
/* ------------------------------------------------------------------------- */

/* bfloat16 is the upper half of an IEEE binary32; widening is exact. */
static double bf16_bits_to_double(uint16_t b) {
    uint32_t u = ((uint32_t)b) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Copy `n` consecutive elements starting at element `off` into fp64. */
static void load_elems(const void* base, int dtype, long off, long n, double* out) {
    if (dtype == ORACLE_F64) {
        const double* p = (const double*)base + off;
        for (long c = 0; c < n; ++c) out[c] = p[c];
    } else {
        const uint16_t* p = (const uint16_t*)base + off;
        for (long c = 0; c < n; ++c) out[c] = bf16_bits_to_double(p[c]);
    }
}

/* One head's Q, K, V (and dO) widened to fp64, [N][d] each. */
typedef struct {
    double* q;
    double* k;
    double* v;
    double* dout;
} head_t;

static void free_head(head_t* h) {
    free(h->q); free(h->k); free(h->v); free(h->dout);
    memset(h, 0, sizeof *h);
}

static int load_head(head_t* h, const void* q, const void* k, const void* v, const void* dout,
                     int dtype, long bh, long N, long d) {
    size_t n = (size_t)N * (size_t)d;
    memset(h, 0, sizeof *h);
    h->q = (double*)malloc(n * sizeof(double));
    h->k = (double*)malloc(n * sizeof(double));
    h->v = (double*)malloc(n * sizeof(double));
    if (dout) h->dout = (double*)malloc(n * sizeof(double));
    if (!h->q || !h->k || !h->v || (dout && !h->dout)) { free_head(h); return -2; }
    long off = bh * N * d;
    load_elems(q, dtype, off, (long)n, h->q);
    load_elems(k, dtype, off, (long)n, h->k);
    load_elems(v, dtype, off, (long)n, h->v);
    if (dout) load_elems(dout, dtype, off, (long)n, h->dout);
    return 0;
}

/* ------------------------------------------------------------------------- */
/* a minimal parallel-for: workers pull item indices from a shared counter   */
/* ------------------------------------------------------------------------- */

typedef void (*item_fn)(void* ctx, long item, double* scratch);

typedef struct {
    item_fn fn;
    void* ctx;
    long n_items;
    long next;          /* shared counter, advanced atomically */
    size_t scratch_len; /* doubles of private scratch per worker */
    int failed;
} pool_t;

static void* pool_worker(void* arg) {
    pool_t* p = (pool_t*)arg;
    double* scratch = (double*)malloc((p->scratch_len ? p->scratch_len : 1) * sizeof(double));
    if (!scratch) { __atomic_store_n(&p->failed, 1, __ATOMIC_SEQ_CST); return NULL; }
    for (;;) {
        long it = __atomic_fetch_add(&p->next, 1, __ATOMIC_SEQ_CST);
        if (it >= p->n_items) break;
        p->fn(p->ctx, it, scratch);
    }
    free(scratch);
    return NULL;
}

int oracle_default_threads(void) {
    long n = sysconf(_SC_NPROCESSORS_ONLN);
    return n > 0 ? (int)n : 1;
}

static int parallel_for(item_fn fn, void* ctx, long n_items, size_t scratch_len, int nthreads) {
    pool_t p = { fn, ctx, n_items, 0, scratch_len, 0 };
    if (nthreads <= 0) nthreads = oracle_default_threads();
    if (nthreads > n_items) nthreads = (int)(n_items > 0 ? n_items : 1);
    pthread_t* th = (pthread_t*)calloc((size_t)nthreads, sizeof(pthread_t));
    if (!th) return -2;
    int started = 0;
    for (int t = 0; t < nthreads; ++t) {
        if (pthread_create(&th[t], NULL, pool_worker, &p) != 0) break;
        ++started;
    }
    if (started == 0) pool_worker(&p);
    for (int t = 0; t < started; ++t) pthread_join(th[t], NULL);
    free(th);
    return p.failed ? -2 : 0;
}

/* ------------------------------------------------------------------------- */
/* the definition, one query row                                             */
/* ------------------------------------------------------------------------- */

static double dot(const double* a, const double* b, long d) {
    double acc = 0.0;
    for (long c = 0; c < d; ++c) acc += a[c] * b[c];
    return acc;
}

/* Number of keys query row i may attend to. */
static long n_keys(long i, long N, int causal) { return causal ? i + 1 : N; }

/* Scores, safe softmax and output of query row i of one head.
 * s, p: scratch rows of length >= N.  Writes o_row[d] and returns lse; also
 * returns the row max and the row sum through m_out / l_out. */
static double attend_row(const head_t* h, long i, long N, long d, double scale, int causal,
                         double* s, double* p, double* o_row, double* m_out, double* l_out) {
    long nk = n_keys(i, N, causal);
    const double* qi = h->q + i * d;
    /* step 1: the score row */
    for (long j = 0; j < nk; ++j) s[j] = scale * dot(qi, h->k + j * d, d);
    /* step 2: safe softmax (subtract the row max) */
    double m = -INFINITY;
    for (long j = 0; j < nk; ++j) if (s[j] > m) m = s[j];
    double l = 0.0;
    for (long j = 0; j < nk; ++j) { p[j] = exp(s[j] - m); l += p[j]; }
    for (long j = 0; j < nk; ++j) p[j] /= l;
    /* step 3: O = P V */
    for (long c = 0; c < d; ++c) o_row[c] = 0.0;
    for (long j = 0; j < nk; ++j) {
        const double* vj = h->v + j * d;
        for (long c = 0; c < d; ++c) o_row[c] += p[j] * vj[c];
    }
    if (m_out) *m_out = m;
    if (l_out) *l_out = l;
    return m + log(l);
}

/* ------------------------------------------------------------------------- */
/* online softmax on one row of given scores                                 */
/* ------------------------------------------------------------------------- */

int oracle_online_row(const double* s, const double* v, long n, long dv, long block,
                      double* m_out, double* l_out, double* u_out) {
    if (!s || n < 0 || dv < 0 || block < 1 || !m_out || !l_out) return -1;
    if (dv > 0 && (!v || !u_out)) return -1;
    double m = -INFINITY, l = 0.0;
    for (long c = 0; c < dv; ++c) u_out[c] = 0.0;
    for (long b0 = 0; b0 < n; b0 += block) {
        long b1 = b0 + block < n ? b0 + block : n;
        /* max of the new block, then the new running max */
        double mb = -INFINITY;
        for (long j = b0; j < b1; ++j) if (s[j] > mb) mb = s[j];
        double m_new = m > mb ? m : mb;
        /* re-base the old sum and weighted sum onto m_new.  With nothing seen
         * yet (m = -inf) there is nothing to re-base; this also avoids forming
         * (-inf) - (-inf) on a block whose scores are all -inf. */
        double alpha = (m == -INFINITY) ? 0.0 : exp(m - m_new);
        double ref = (m_new == -INFINITY) ? 0.0 : m_new;
        l *= alpha;
        for (long c = 0; c < dv; ++c) u_out[c] *= alpha;
        for (long j = b0; j < b1; ++j) {
            double e = exp(s[j] - ref);
            l += e;
            for (long c = 0; c < dv; ++c) u_out[c] += e * v[j * dv + c];
        }
        m = m_new;
    }
    *m_out = m;
    *l_out = l;
    return 0;
}

/* ------------------------------------------------------------------------- */
/* forward                                                                   */
/* ------------------------------------------------------------------------- */

typedef struct {
    const void *q, *k, *v;
    int dtype;
    long BH, N, d;
    double scale;
    int causal;
    const int64_t* bh_list;
    long n_bh;
    double *o, *lse;
    head_t* heads; /* n_bh heads widened to fp64 */
    const int64_t* rows;
    long nrows;
    long block_q, block_k;
} fwd_ctx;

static void load_head_item(void* vctx, long item, double* scratch) {
    (void)scratch;
    fwd_ctx* c = (fwd_ctx*)vctx;
    long bh = c->bh_list ? (long)c->bh_list[item] : item;
    if (load_head(&c->heads[item], c->q, c->k, c->v, NULL, c->dtype, bh, c->N, c->d) != 0)
        c->heads[item].q = NULL;
}

static int load_heads(fwd_ctx* c, int nthreads) {
    c->heads = (head_t*)calloc((size_t)c->n_bh, sizeof(head_t));
    if (!c->heads) return -2;
    int rc = parallel_for(load_head_item, c, c->n_bh, 0, nthreads);
    for (long t = 0; t < c->n_bh && rc == 0; ++t) if (!c->heads[t].q) rc = -2;
    return rc;
}

static void free_heads(fwd_ctx* c) {
    if (!c->heads) return;
    for (long t = 0; t < c->n_bh; ++t) free_head(&c->heads[t]);
    free(c->heads);
    c->heads = NULL;
}

/* item = t * N + i : head slot t, query row i */
static void fwd_row_item(void* vctx, long item, double* scratch) {
    fwd_ctx* c = (fwd_ctx*)vctx;
    long t = item / c->N, i = item % c->N;
    double* s = scratch;
    double* p = scratch + c->N;
    double orow[1024];
    double lse = attend_row(&c->heads[t], i, c->N, c->d, c->scale, c->causal, s, p, orow, NULL, NULL);
    if (c->o) memcpy(c->o + (t * c->N + i) * c->d, orow, (size_t)c->d * sizeof(double));
    if (c->lse) c->lse[t * c->N + i] = lse;
}

static int check_common(const void* q, const void* k, const void* v, int dtype,
                        long BH, long N, long d) {
    if (!q || !k || !v) return -1;
    if (dtype != ORACLE_F64 && dtype != ORACLE_BF16) return -1;
    if (BH < 1 || N < 1 || d < 1 || d > 1024) return -1;
    return 0;
}

int oracle_fwd(const void* q, const void* k, const void* v, int dtype,
               long BH, long N, long d, double scale, int causal,
               const int64_t* bh_list, long n_bh,
               double* o, double* lse, int nthreads) {
    if (check_common(q, k, v, dtype, BH, N, d)) return -1;
    if (!bh_list) n_bh = BH;
    if (n_bh < 1) return -1;
    for (long t = 0; bh_list && t < n_bh; ++t) if (bh_list[t] < 0 || bh_list[t] >= BH) return -1;
    fwd_ctx c = { q, k, v, dtype, BH, N, d, scale, causal, bh_list, n_bh, o, lse,
                  NULL, NULL, 0, 0, 0 };
    int rc = load_heads(&c, nthreads);
    if (rc == 0) rc = parallel_for(fwd_row_item, &c, n_bh * N, (size_t)(2 * N), nthreads);
    free_heads(&c);
    return rc;
}

/* item = bh * nrows + r */
static void fwd_sel_item(void* vctx, long item, double* scratch) {
    fwd_ctx* c = (fwd_ctx*)vctx;
    long bh = item / c->nrows;
    long i = (long)c->rows[item];
    double* s = scratch;
    double* p = scratch + c->N;
    double orow[1024];
    double lse = attend_row(&c->heads[bh], i, c->N, c->d, c->scale, c->causal, s, p, orow, NULL, NULL);
    if (c->o) memcpy(c->o + item * c->d, orow, (size_t)c->d * sizeof(double));
    if (c->lse) c->lse[item] = lse;
}

int oracle_fwd_rows(const void* q, const void* k, const void* v, int dtype,
                    long BH, long N, long d, double scale, int causal,
                    const int64_t* rows, long nrows,
                    double* o_rows, double* lse_rows, int nthreads) {
    if (check_common(q, k, v, dtype, BH, N, d) || !rows || nrows < 1) return -1;
    for (long t = 0; t < BH * nrows; ++t) if (rows[t] < 0 || rows[t] >= N) return -1;
    fwd_ctx c = { q, k, v, dtype, BH, N, d, scale, causal, NULL, BH, o_rows, lse_rows,
                  NULL, rows, nrows, 0, 0 };
    int rc = load_heads(&c, nthreads);
    if (rc == 0) rc = parallel_for(fwd_sel_item, &c, BH * nrows, (size_t)(2 * N), nthreads);
    free_heads(&c);
    return rc;
}

/* ------------------------------------------------------------------------- */
/* forward in the tiled order (online recurrence), one query block per item  */
/* ------------------------------------------------------------------------- */

/* item = bh * n_qblocks + qb.  For every row of the query block the key/value
 * blocks are visited in order; per block: block row max, new running max,
 * correction factor alpha = exp(m_old - m_new), l <- alpha l + rowsum(exp(s - m_new)),
 * u <- alpha u + exp(s - m_new) V_j.  After the last block O = u / l and
 * lse = m + log l. */
static void fwd_block_item(void* vctx, long item, double* scratch) {
    fwd_ctx* c = (fwd_ctx*)vctx;
    long nqb = (c->N + c->block_q - 1) / c->block_q;
    long bh = item / nqb, qb = item % nqb;
    const head_t* h = &c->heads[bh];
    long d = c->d, N = c->N;
    long i0 = qb * c->block_q;
    long i1 = i0 + c->block_q < N ? i0 + c->block_q : N;
    double* u = scratch; /* d doubles */
    for (long i = i0; i < i1; ++i) {
        double m = -INFINITY, l = 0.0;
        for (long cc = 0; cc < d; ++cc) u[cc] = 0.0;
        for (long j0 = 0; j0 < N; j0 += c->block_k) {
            long j1 = j0 + c->block_k < N ? j0 + c->block_k : N;
            double sblk[4096];
            long nb = j1 - j0;
            double mb = -INFINITY;
            for (long j = j0; j < j1; ++j) {
                double sj = (c->causal && j > i) ? -INFINITY
                                                 : c->scale * dot(h->q + i * d, h->k + j * d, d);
                sblk[j - j0] = sj;
                if (sj > mb) mb = sj;
            }
            double m_new = m > mb ? m : mb;
            double alpha = (m == -INFINITY) ? 0.0 : exp(m - m_new);
            double ref = (m_new == -INFINITY) ? 0.0 : m_new;
            l *= alpha;
            for (long cc = 0; cc < d; ++cc) u[cc] *= alpha;
            for (long t = 0; t < nb; ++t) {
                double e = exp(sblk[t] - ref);
                l += e;
                const double* vj = h->v + (j0 + t) * d;
                for (long cc = 0; cc < d; ++cc) u[cc] += e * vj[cc];
            }
            m = m_new;
        }
        if (c->o) for (long cc = 0; cc < d; ++cc) c->o[(bh * N + i) * d + cc] = u[cc] / l;
        if (c->lse) c->lse[bh * N + i] = m + log(l);
    }
}

int oracle_fwd_blockwise(const void* q, const void* k, const void* v, int dtype,
                         long BH, long N, long d, double scale, int causal,
                         long block_q, long block_k,
                         double* o, double* lse, int nthreads) {
    if (check_common(q, k, v, dtype, BH, N, d)) return -1;
    if (block_q < 1 || block_k < 1 || block_k > 4096) return -1;
    fwd_ctx c = { q, k, v, dtype, BH, N, d, scale, causal, NULL, BH, o, lse,
                  NULL, NULL, 0, block_q, block_k };
    int rc = load_heads(&c, nthreads);
    long nqb = (N + block_q - 1) / block_q;
    if (rc == 0) rc = parallel_for(fwd_block_item, &c, BH * nqb, (size_t)d, nthreads);
    free_heads(&c);
    return rc;
}

/* ------------------------------------------------------------------------- */
/* backward                                                                  */
/* ------------------------------------------------------------------------- */

typedef struct {
    const head_t* h;
    long N, d;
    double scale;
    int causal;
    /* per-row statistics of the oracle's own forward */
    double* m;  /* row max        [N] */
    double* l;  /* row sum        [N] */
    double* D;  /* rowsum(dO*O)   [N] */
    double *o, *lse, *dq, *dk, *dv; /* this head's slices */
} bwd_head_ctx;

/* Row pass for query row i: scores, P, O, lse, D_i = dO_i . O_i,
 * dP_ij = dO_i . V_j, dS_ij = P_ij (dP_ij - D_i), dQ_i = scale sum_j dS_ij K_j. */
static void bwd_row_item(void* vctx, long i, double* scratch) {
    bwd_head_ctx* c = (bwd_head_ctx*)vctx;
    long N = c->N, d = c->d;
    double* s = scratch;
    double* p = scratch + N;
    double* orow = scratch + 2 * N;
    double m, l;
    double lse = attend_row(c->h, i, N, d, c->scale, c->causal, s, p, orow, &m, &l);
    const double* doi = c->h->dout + i * d;
    double Di = dot(doi, orow, d);
    c->m[i] = m;
    c->l[i] = l;
    c->D[i] = Di;
    if (c->o) memcpy(c->o + i * d, orow, (size_t)d * sizeof(double));
    if (c->lse) c->lse[i] = lse;
    double* dqi = c->dq + i * d;
    for (long cc = 0; cc < d; ++cc) dqi[cc] = 0.0;
    long nk = n_keys(i, N, c->causal);
    for (long j = 0; j < nk; ++j) {
        double dP = dot(doi, c->h->v + j * d, d);
        double dS = p[j] * (dP - Di);
        const double* kj = c->h->k + j * d;
        for (long cc = 0; cc < d; ++cc) dqi[cc] += c->scale * dS * kj[cc];
    }
}

/* Column pass for key row j: every query row i that sees key j contributes
 * dV_j += P_ij dO_i and dK_j += scale dS_ij Q_i, with P_ij = exp(s_ij - m_i) / l_i
 * (the softmax of row i, from that row's max and sum). */
static void bwd_col_item(void* vctx, long j, double* scratch) {
    (void)scratch;
    bwd_head_ctx* c = (bwd_head_ctx*)vctx;
    long N = c->N, d = c->d;
    double* dkj = c->dk + j * d;
    double* dvj = c->dv + j * d;
    for (long cc = 0; cc < d; ++cc) { dkj[cc] = 0.0; dvj[cc] = 0.0; }
    const double* kj = c->h->k + j * d;
    const double* vj = c->h->v + j * d;
    long i0 = c->causal ? j : 0;
    for (long i = i0; i < N; ++i) {
        const double* qi = c->h->q + i * d;
        const double* doi = c->h->dout + i * d;
        double sij = c->scale * dot(qi, kj, d);
        double Pij = exp(sij - c->m[i]) / c->l[i];
        double dP = dot(doi, vj, d);
        double dS = Pij * (dP - c->D[i]);
        for (long cc = 0; cc < d; ++cc) {
            dvj[cc] += Pij * doi[cc];
            dkj[cc] += c->scale * dS * qi[cc];
        }
    }
}

int oracle_bwd(const void* q, const void* k, const void* v, const void* dout, int dtype,
               long BH, long N, long d, double scale, int causal,
               const int64_t* bh_list, long n_bh,
               double* dq, double* dk, double* dv,
               double* o_out, double* lse_out, int nthreads) {
    if (check_common(q, k, v, dtype, BH, N, d) || !dout || !dq || !dk || !dv) return -1;
    if (!bh_list) n_bh = BH;
    if (n_bh < 1) return -1;
    for (long t = 0; bh_list && t < n_bh; ++t) if (bh_list[t] < 0 || bh_list[t] >= BH) return -1;
    double* stats = (double*)malloc((size_t)(3 * N) * sizeof(double));
    if (!stats) return -2;
    int rc = 0;
    for (long t = 0; t < n_bh && rc == 0; ++t) {
        long bh = bh_list ? (long)bh_list[t] : t;
        head_t h;
        rc = load_head(&h, q, k, v, dout, dtype, bh, N, d);
        if (rc) break;
        size_t off = (size_t)t * (size_t)N * (size_t)d;
        bwd_head_ctx c = { &h, N, d, scale, causal, stats, stats + N, stats + 2 * N,
                           o_out ? o_out + off : NULL, lse_out ? lse_out + (size_t)t * N : NULL,
                           dq + off, dk + off, dv + off };
        rc = parallel_for(bwd_row_item, &c, N, (size_t)(2 * N + d), nthreads);
        if (rc == 0) rc = parallel_for(bwd_col_item, &c, N, 0, nthreads);
        free_head(&h);
    }
    free(stats);
    return rc;
}

/* ------------------------------------------------------------------------- */
/* backward for selected rows                                                */
/* ------------------------------------------------------------------------- */

typedef struct {
    bwd_head_ctx* c;
    const int64_t* rows; /* row indices of this head */
} sel_ctx;

/* Statistics of query row i only: m_i, l_i and D_i = dO_i . O_i. */
static void stat_row_item(void* vctx, long item, double* scratch) {
    sel_ctx* sc = (sel_ctx*)vctx;
    bwd_head_ctx* c = sc->c;
    long i = (long)sc->rows[item];
    double* s = scratch;
    double* p = scratch + c->N;
    double* orow = scratch + 2 * c->N;
    double m, l;
    attend_row(c->h, i, c->N, c->d, c->scale, c->causal, s, p, orow, &m, &l);
    c->m[i] = m;
    c->l[i] = l;
    c->D[i] = dot(c->h->dout + i * c->d, orow, c->d);
}

static void sel_row_item(void* vctx, long item, double* scratch) {
    sel_ctx* sc = (sel_ctx*)vctx;
    bwd_row_item(sc->c, (long)sc->rows[item], scratch);
}

static void sel_col_item(void* vctx, long item, double* scratch) {
    sel_ctx* sc = (sel_ctx*)vctx;
    bwd_col_item(sc->c, (long)sc->rows[item], scratch);
}

int oracle_bwd_rows(const void* q, const void* k, const void* v, const void* dout, int dtype,
                    long BH, long N, long d, double scale, int causal,
                    const int64_t* qrows, long nq, const int64_t* krows, long nk,
                    double* dq_rows, double* dk_rows, double* dv_rows, int nthreads) {
    if (check_common(q, k, v, dtype, BH, N, d) || !dout) return -1;
    if (nq < 0 || nk < 0 || nq + nk < 1) return -1;
    if (nq > 0 && (!qrows || !dq_rows)) return -1;
    if (nk > 0 && (!krows || !dk_rows || !dv_rows)) return -1;
    for (long t = 0; t < BH * nq; ++t) if (qrows[t] < 0 || qrows[t] >= N) return -1;
    for (long t = 0; t < BH * nk; ++t) if (krows[t] < 0 || krows[t] >= N) return -1;
    size_t nd = (size_t)N * (size_t)d;
    double* stats = (double*)malloc((size_t)(3 * N) * sizeof(double));
    double* full = (double*)malloc(3 * nd * sizeof(double)); /* dq, dk, dv of one head */
    int64_t* need = (int64_t*)malloc((size_t)N * sizeof(int64_t));
    if (!stats || !full || !need) { free(stats); free(full); free(need); return -2; }
    int rc = 0;
    for (long bh = 0; bh < BH && rc == 0; ++bh) {
        head_t h;
        rc = load_head(&h, q, k, v, dout, dtype, bh, N, d);
        if (rc) break;
        bwd_head_ctx c = { &h, N, d, scale, causal, stats, stats + N, stats + 2 * N,
                           NULL, NULL, full, full + nd, full + 2 * nd };
        /* the column pass of key row j reads the statistics of every query row
         * that sees key j: all rows, or rows i >= j when causal */
        long first = N;
        for (long t = 0; t < nk; ++t) if (krows[bh * nk + t] < first) first = (long)krows[bh * nk + t];
        if (nk > 0 && !causal) first = 0;
        long n_need = 0;
        for (long i = first; i < N; ++i) need[n_need++] = i;
        if (n_need > 0) {
            sel_ctx st = { &c, need };
            rc = parallel_for(stat_row_item, &st, n_need, (size_t)(2 * N + d), nthreads);
        }
        if (rc == 0 && nq > 0) {
            sel_ctx sq = { &c, qrows + bh * nq };
            rc = parallel_for(sel_row_item, &sq, nq, (size_t)(2 * N + d), nthreads);
            for (long t = 0; rc == 0 && t < nq; ++t)
                memcpy(dq_rows + (bh * nq + t) * d, c.dq + qrows[bh * nq + t] * d,
                       (size_t)d * sizeof(double));
        }
        if (rc == 0 && nk > 0) {
            sel_ctx sk = { &c, krows + bh * nk };
            rc = parallel_for(sel_col_item, &sk, nk, 0, nthreads);
            for (long t = 0; rc == 0 && t < nk; ++t) {
                memcpy(dk_rows + (bh * nk + t) * d, c.dk + krows[bh * nk + t] * d,
                       (size_t)d * sizeof(double));
                memcpy(dv_rows + (bh * nk + t) * d, c.dv + krows[bh * nk + t] * d,
                       (size_t)d * sizeof(double));
            }
        }
        free_head(&h);
    }
    free(stats);
    free(full);
    free(need);
    return rc;
}
