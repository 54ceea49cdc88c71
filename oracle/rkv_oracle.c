/*
 * rkv_oracle.c -- plain fp64 CPU oracle of the R-KV decode-time KV-cache
 * compression step.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file: it exists so that tests/, the smoke check and the CPU
 * baseline leg of bench.py can compare the CUDA library against a slow,
 * obviously correct restatement of the method.  It shares no code, header,
 * table or constant with the CUDA library.
 *
 * Sources (the pages the method is taken from):
 *   [notes]      R-KV review (yoonschallenge.tistory.com/1236), opening notes:
 *                B_budget / B_buffer; the newest 8 tokens always stay, the
 *                others are scored, the best that fit the budget are kept,
 *                the rest evicted, and 128 more tokens are generated.
 *   [scheme]     same page, summary table, row "Decoding-time compression
 *                scheme": merge cache and buffer, always keep some recent
 *                observation tokens, prune the rest by score; buffer 128,
 *                observation tokens 8.
 *   [importance] same table, row "importance": attention weight the recent
 *                observation tokens give to each past key; under GQA the
 *                query heads sharing one KV head are max-pooled.
 *   [redundancy] same table, row "redundancy": cosine similarity between key
 *                vectors of the same head; a key similar to many others is
 *                redundant; the beta most recent of the similar tokens are
 *                protected.
 *   [selection]  same table, row "final selection criterion": higher
 *                importance raises the score, higher redundancy lowers it,
 *                lambda = 0.1.  The formula itself was lost from the page; the
 *                plainest form consistent with the row is
 *                Z = lambda * I - (1 - lambda) * R.
 *   [cause3]     same page, question 2, cause 3: the steps of one compression
 *                round (attention importance, key normalisation, all-pairs
 *                cosine similarity, a softmax of the redundancy, combine,
 *                top-k, copy the kept KV).
 *   [snapkv]     same page, summary table: SnapKV, the attention-only method
 *                R-KV is compared with; its importance is pooled over
 *                neighbouring positions.
 *
 * Readings of points the pages leave open (each is stated where it is used):
 *   R1  importance: mean over the n_obs observation queries of the softmax
 *       probability, max over the query heads of the GQA group.
 *   R2  softmax domain: all N keys of the merged cache, scale 1/sqrt(d),
 *       causal among the observation tokens (query q sees keys
 *       j <= N - n_obs + q).
 *   R3  redundancy domain: all N keys except the key itself; mean = sum/(N-1).
 *   R4  "similar" means S_ij > tau (strict).  Token i is protected iff fewer
 *       than beta tokens newer than i are similar to it; a protected token
 *       drops its above-tau similarities from its redundancy sum.
 *   R5  zero-norm key: norms are clamped to eps = 1e-12, so S = 0.
 *   R6  by default no softmax over redundancy (the cause-3 list names one,
 *       but the redundancy is a mean cosine similarity; identical keys give
 *       R = 1).  The softmax is variant R10.
 *   R7  ties in Z: the larger (more recent) index wins.
 *   R8  kept indices are returned in ascending order; the n_obs observation
 *       tokens are always the last n_obs of them.
 *   R9  n_cached <= budget: nothing is evicted (identity).
 *   R10 variant, redundancy softmax: R'_i = exp(R_i) / sum_{j<C} exp(R_j)
 *       over the C = N - n_obs candidates (temperature 1); observation
 *       tokens are not candidates.
 *   R11 variant, importance pooling: I'_i = max of I_j over the candidates j
 *       with |j - i| <= (w-1)/2 for an odd window w, the window cut at the
 *       candidates' ends; applied to I after the max over query heads.
 *
 * Layouts (row-major, contiguous, fp64):
 *   K  [P, N, d]          keys of the merged cache (budget rows, then buffer)
 *   Q  [P, G, n_obs, d]   observation queries; query head g of problem p
 *                         belongs to the KV head of problem p
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_EPS 1e-12

/* ------------------------------------------------------------------ */
/* small helpers                                                        */
/* ------------------------------------------------------------------ */

static double dot_d(const double* a, const double* b, int d) {
    double s = 0.0;
    for (int t = 0; t < d; ++t) s += a[t] * b[t];
    return s;
}

/* ||k|| clamped below by eps (reading R5). */
static double clamped_norm(const double* k, int d) {
    double n = sqrt(dot_d(k, k, d));
    return n > ORACLE_EPS ? n : ORACLE_EPS;
}

/* ------------------------------------------------------------------ */
/* cosine similarity [redundancy], [cause3: key normalisation +        */
/* all-pairs cosine similarity]                                         */
/* ------------------------------------------------------------------ */

/* S[i*N + j] = (k_i . k_j) / (max(|k_i|,eps) * max(|k_j|,eps)) for all i, j
 * of one problem (the diagonal is filled with the same formula). */
void rkv_oracle_cosine(const double* K, int N, int d, double* S) {
    double* nrm = (double*)malloc(sizeof(double) * (size_t)(N > 0 ? N : 1));
    for (int i = 0; i < N; ++i) nrm[i] = clamped_norm(K + (size_t)i * d, d);
    for (int i = 0; i < N; ++i)
        for (int j = 0; j < N; ++j)
            S[(size_t)i * N + j] =
                dot_d(K + (size_t)i * d, K + (size_t)j * d, d) / (nrm[i] * nrm[j]);
    free(nrm);
}

/* ------------------------------------------------------------------ */
/* attention of the observation queries [importance], readings R1, R2   */
/* ------------------------------------------------------------------ */

/* p[(g*n_obs + q)*N + j]: softmax probability that observation query q of
 * query head g gives key j; keys j > N - n_obs + q are masked (p = 0). */
void rkv_oracle_attention(const double* K, const double* Q, int N, int d, int G,
                          int n_obs, double* p) {
    const double scale = 1.0 / sqrt((double)d);
    for (int g = 0; g < G; ++g) {
        for (int q = 0; q < n_obs; ++q) {
            const double* qv = Q + ((size_t)g * n_obs + q) * d;
            double* row = p + ((size_t)g * n_obs + q) * N;
            const int last = N - n_obs + q; /* causal: keys 0..last */
            double mx = -INFINITY;
            for (int j = 0; j < N; ++j) {
                if (j <= last) {
                    row[j] = dot_d(qv, K + (size_t)j * d, d) * scale;
                    if (row[j] > mx) mx = row[j];
                } else {
                    row[j] = 0.0;
                }
            }
            double den = 0.0;
            for (int j = 0; j <= last && j < N; ++j) {
                row[j] = exp(row[j] - mx);
                den += row[j];
            }
            for (int j = 0; j <= last && j < N; ++j) row[j] /= den;
        }
    }
}

/* ------------------------------------------------------------------ */
/* per-problem score                                                     */
/* ------------------------------------------------------------------ */

/* Scores of one problem.  Outputs (length N each):
 *   I[i]       importance (R1, R2)
 *   R[i]       redundancy (R3, R4, R5); 0 for observation tokens
 *   Z[i]       lambda*I - (1-lambda)*R for candidates, +inf for the n_obs
 *              observation tokens (always kept, [scheme])
 *   sum[i]     sum_{j != i} S_ij
 *   sim[i]     sum_{j != i, S_ij > tau} S_ij
 *   newer[i]   #{ j > i : S_ij > tau }
 *   border[i]  1 if some j != i has |S_ij - tau| < border_eps (the kept-set
 *              comparison excuses such tokens: their protection flag or sim
 *              can flip under rounding)
 */
static void score_one(const double* K, const double* Q, int N, int d, int G, int n_obs,
                      double lambda, int beta, double tau, double border_eps,
                      double* I, double* R, double* Z, double* sum, double* sim,
                      int32_t* newer, uint8_t* border, double* scratch_p) {
    const int C = N - n_obs;
    /* importance [importance]: p over keys, mean over queries, max over heads */
    rkv_oracle_attention(K, Q, N, d, G, n_obs, scratch_p);
    for (int i = 0; i < N; ++i) {
        double best = -INFINITY;
        for (int g = 0; g < G; ++g) {
            double m = 0.0;
            for (int q = 0; q < n_obs; ++q) m += scratch_p[((size_t)g * n_obs + q) * N + i];
            m /= (double)n_obs;
            if (m > best) best = m;
        }
        I[i] = best;
    }
    /* redundancy [redundancy] + [cause3] */
    double* nrm = scratch_p + (size_t)G * n_obs * N; /* N doubles after p */
    for (int i = 0; i < N; ++i) nrm[i] = clamped_norm(K + (size_t)i * d, d);
    for (int i = 0; i < N; ++i) {
        double s_all = 0.0, s_sim = 0.0;
        int n_newer = 0;
        uint8_t bd = 0;
        for (int j = 0; j < N; ++j) {
            if (j == i) continue;
            const double s = dot_d(K + (size_t)i * d, K + (size_t)j * d, d) / (nrm[i] * nrm[j]);
            s_all += s;
            if (s > tau) {
                s_sim += s;
                if (j > i) n_newer += 1;
            }
            if (fabs(s - tau) < border_eps) bd = 1;
        }
        sum[i] = s_all;
        sim[i] = s_sim;
        newer[i] = n_newer;
        border[i] = bd;
        if (i < C) {
            const int protect = n_newer < beta; /* reading R4 */
            R[i] = (s_all - (protect ? s_sim : 0.0)) / (double)(N - 1);
            Z[i] = lambda * I[i] - (1.0 - lambda) * R[i];
        } else {
            R[i] = 0.0;
            Z[i] = INFINITY;
        }
    }
}

/* ------------------------------------------------------------------ */
/* a tiny worker pool over problems (plain pthreads)                    */
/* ------------------------------------------------------------------ */

typedef struct {
    void (*fn)(void* ctx, int64_t p, double* scratch);
    void* ctx;
    int64_t P;
    int64_t next;
    size_t scratch_doubles;
    pthread_mutex_t mu;
} pool_t;

static void* pool_worker(void* arg) {
    pool_t* pl = (pool_t*)arg;
    double* scratch = (double*)malloc(sizeof(double) * (pl->scratch_doubles ? pl->scratch_doubles : 1));
    for (;;) {
        pthread_mutex_lock(&pl->mu);
        const int64_t p = pl->next++;
        pthread_mutex_unlock(&pl->mu);
        if (p >= pl->P) break;
        pl->fn(pl->ctx, p, scratch);
    }
    free(scratch);
    return NULL;
}

static void run_pool(void (*fn)(void*, int64_t, double*), void* ctx, int64_t P,
                     size_t scratch_doubles, int nthreads) {
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 512) nthreads = 512;
    if ((int64_t)nthreads > P) nthreads = (int)(P > 0 ? P : 1);
    pool_t pl;
    pl.fn = fn;
    pl.ctx = ctx;
    pl.P = P;
    pl.next = 0;
    pl.scratch_doubles = scratch_doubles;
    pthread_mutex_init(&pl.mu, NULL);
    if (nthreads == 1) {
        pool_worker(&pl);
    } else {
        pthread_t th[512];
        for (int t = 0; t < nthreads; ++t) pthread_create(&th[t], NULL, pool_worker, &pl);
        for (int t = 0; t < nthreads; ++t) pthread_join(th[t], NULL);
    }
    pthread_mutex_destroy(&pl.mu);
}

typedef struct {
    const double *K, *Q;
    int N, d, G, n_obs, beta;
    double lambda, tau, border_eps;
    double *I, *R, *Z, *sum, *sim;
    int32_t* newer;
    uint8_t* border;
} score_ctx;

static void score_task(void* c, int64_t p, double* scratch) {
    score_ctx* s = (score_ctx*)c;
    const size_t nd = (size_t)s->N * s->d, n = (size_t)s->N;
    score_one(s->K + p * nd, s->Q + (size_t)p * s->G * s->n_obs * s->d, s->N, s->d, s->G,
              s->n_obs, s->lambda, s->beta, s->tau, s->border_eps, s->I + p * n,
              s->R + p * n, s->Z + p * n, s->sum + p * n, s->sim + p * n,
              s->newer + p * n, s->border + p * n, scratch);
}

/* Scores for P independent problems (one problem = one (layer, sequence,
 * KV head)).  Returns 0, or -1 for invalid sizes. */
int rkv_oracle_score(const double* K, const double* Q, int64_t P, int N, int d, int G,
                     int n_obs, double lambda, int beta, double tau, double border_eps,
                     double* I, double* R, double* Z, double* sum, double* sim,
                     int32_t* newer, uint8_t* border, int nthreads) {
    if (P < 0 || N < 2 || d < 1 || G < 1 || n_obs < 0 || n_obs > N) return -1;
    score_ctx c = {K, Q, N, d, G, n_obs, beta, lambda, tau, border_eps,
                   I, R, Z, sum, sim, newer, border};
    run_pool(score_task, &c, P, (size_t)G * n_obs * N + N, nthreads);
    return 0;
}

/* ------------------------------------------------------------------ */
/* top-k selection [notes], [scheme], [cause3: top-k], readings R7, R8  */
/* ------------------------------------------------------------------ */

typedef struct {
    double z;
    int32_t i;
} zi_t;

/* larger Z first; equal Z: larger index first (reading R7) */
static int cmp_zi_desc(const void* a, const void* b) {
    const zi_t* x = (const zi_t*)a;
    const zi_t* y = (const zi_t*)b;
    if (x->z > y->z) return -1;
    if (x->z < y->z) return 1;
    return (x->i > y->i) ? -1 : (x->i < y->i) ? 1 : 0;
}

static int cmp_i32_asc(const void* a, const void* b) {
    const int32_t x = *(const int32_t*)a, y = *(const int32_t*)b;
    return (x > y) - (x < y);
}

/* idx[P, budget]: for each problem, the budget - n_obs candidates
 * (indices 0 .. N-n_obs-1) with the largest Z, plus the n_obs observation
 * tokens N-n_obs .. N-1, in ascending order.  N <= budget keeps 0..N-1 and
 * fills the rest of the row with -1 (reading R9).  Returns 0, or -1. */
int rkv_oracle_select(const double* Z, int64_t P, int N, int n_obs, int budget, int32_t* idx) {
    if (P < 0 || N < 1 || n_obs < 0 || n_obs > budget || n_obs > N || budget < 1) return -1;
    const int C = N - n_obs;
    zi_t* buf = (zi_t*)malloc(sizeof(zi_t) * (size_t)(C > 0 ? C : 1));
    for (int64_t p = 0; p < P; ++p) {
        int32_t* out = idx + p * budget;
        if (N <= budget) {
            for (int r = 0; r < budget; ++r) out[r] = r < N ? r : -1;
            continue;
        }
        const double* z = Z + p * (int64_t)N;
        for (int i = 0; i < C; ++i) {
            buf[i].z = z[i];
            buf[i].i = i;
        }
        qsort(buf, (size_t)C, sizeof(zi_t), cmp_zi_desc);
        const int k = budget - n_obs;
        for (int r = 0; r < k; ++r) out[r] = buf[r].i;
        qsort(out, (size_t)k, sizeof(int32_t), cmp_i32_asc);
        for (int r = 0; r < n_obs; ++r) out[k + r] = C + r;
    }
    free(buf);
    return 0;
}

/* ------------------------------------------------------------------ */
/* scoring variants [cause3: redundancy softmax] [snapkv: pooling]     */
/* ------------------------------------------------------------------ */

/* From one call's base scores I, R [P, N], the variant scores: I_out = I
 * pooled over a window of w positions (R11; w = 1 leaves I as it is), R_out =
 * the softmax of R over the candidates (R10) when softmax != 0 (else R), and
 * Z = lambda * I_out - (1 - lambda) * R_out.  Observation tokens keep I,
 * get R = 0 and Z = +inf.  Returns 0, or -1 for invalid sizes. */
int rkv_oracle_variant(const double* I, const double* R, int64_t P, int N, int n_obs,
                       double lambda, int softmax, int window, double* I_out, double* R_out,
                       double* Z) {
    if (P < 0 || N < 1 || n_obs < 0 || n_obs >= N || window < 1 || window % 2 == 0) return -1;
    const int C = N - n_obs, h = (window - 1) / 2;
    for (int64_t p = 0; p < P; ++p) {
        const double* ip = I + p * (int64_t)N;
        const double* rp = R + p * (int64_t)N;
        double* io = I_out + p * (int64_t)N;
        double* ro = R_out + p * (int64_t)N;
        double* z = Z + p * (int64_t)N;
        double m = -INFINITY, total = 0.0;
        if (softmax) {
            for (int j = 0; j < C; ++j) m = rp[j] > m ? rp[j] : m;
            for (int j = 0; j < C; ++j) total += exp(rp[j] - m);
        }
        for (int i = 0; i < C; ++i) {
            const int lo = i - h < 0 ? 0 : i - h, hi = i + h > C - 1 ? C - 1 : i + h;
            double best = ip[lo];
            for (int j = lo + 1; j <= hi; ++j) best = ip[j] > best ? ip[j] : best;
            io[i] = best;
            ro[i] = softmax ? exp(rp[i] - m) / total : rp[i];
            z[i] = lambda * io[i] - (1.0 - lambda) * ro[i];
        }
        for (int i = C; i < N; ++i) {
            io[i] = ip[i];
            ro[i] = 0.0;
            z[i] = INFINITY;
        }
    }
    return 0;
}

/* ------------------------------------------------------------------ */
/* copy of the kept rows [cause3: copy the selected KV to the new cache] */
/* ------------------------------------------------------------------ */

/* out[p, r, :] = src[p, idx[p, r], :] for r < budget with idx >= 0.  Rows are
 * moved as raw bytes (row_bytes each), so any element type is copied
 * exactly.  src and out are [P, n_cap, row] arrays; out may not alias src. */
void rkv_oracle_gather_bytes(const uint8_t* src, int64_t P, int n_cap, int64_t row_bytes,
                             const int32_t* idx, int budget, uint8_t* out) {
    for (int64_t p = 0; p < P; ++p)
        for (int r = 0; r < budget; ++r) {
            const int32_t s = idx[p * budget + r];
            if (s < 0) continue;
            memcpy(out + ((size_t)p * n_cap + r) * row_bytes,
                   src + ((size_t)p * n_cap + s) * row_bytes, (size_t)row_bytes);
        }
}
