/*
 * oracle.c -- plain fp64 CPU oracle for exact causal softmax attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call, link or
 * load this file: only the tests, the package smoke check and the benchmark's
 * CPU-baseline leg use it.  It shares no code, header, table or constant with
 * the CUDA library; the two only ever see the same seeded input arrays.
 *
 * What it computes (DISTFLASHATTN, paperlayer.ai summary of arXiv 2310.03294):
 *   - §3.1: the attention each worker computes is ordinary exact attention of
 *     its query tokens against key/value blocks (FlashAttention's result, no
 *     approximation), and the pseudocode of App. D returns the output together
 *     with its log-sum-exp;
 *   - §3.2: a query only attends to its causal prefix; helpers return a partial
 *     output plus softmax statistics which the owner rescales and merges (the
 *     online-normalizer rule of "Online normalizer calculation for softmax");
 *   - §1/§3.3: the backward reuses the saved output and log-sum-exp, and this
 *     rematerialisation changes no numbers, i.e. the backward is the exact
 *     gradient of the same attention.
 *
 * The pages print no formulas; the readings taken here are the textbook ones:
 *   s_ij  = scale * <q_i, k_j>            visible iff !causal or kv_pos(j) <= q_pos(i)
 *   lse_i = ln sum_j exp(s_ij)            (natural log; -inf for a row with no visible key)
 *   P_ij  = exp(s_ij - lse_i),  O_i = sum_j P_ij v_j   (O_i = 0 for an empty row)
 *   dV_j  = sum_i P_ij dO_i
 *   dP_ij = <dO_i, v_j>
 *   Delta_i = sum_j P_ij dP_ij            (the explicit definition, not dO.O)
 *   dS_ij = P_ij (dP_ij - Delta_i)
 *   dQ_i  = scale sum_j dS_ij k_j,   dK_j = scale sum_i dS_ij q_i
 * The local sliding window of App. F (a worker attends only to its own chunk
 * and the neighbouring ones before it) is read as: key position kp is visible
 * from query position qp iff kp <= qp and floor(kp / C) >= floor(qp / C) - (w - 1)
 * for chunk length C and a window of w chunks (oracle_fwd_local/_bwd_local).
 * A worker's backward step for one (query chunk, key chunk) pair (§3.3) uses
 * the rows' global lse_i and Delta_i and gives the pair's share of dQ (for the
 * query chunk) and of dK, dV (for the key chunk); summed over the pairs these
 * are the full gradients (oracle_chunk_bwd).
 * Grouped-query attention (GQA paper, cited on the DISTFLASHATTN page): query
 * head h reads key/value head h / (H / H_kv); dK/dV sum over the group.
 *
 * Every score row is built in full and normalised with its exact maximum: no
 * blocking, no online softmax, no fused passes.  Layouts: Q/O/dQ/dO are
 * [B, Lq, H, D], K/V/dK/dV are [B, Lkv, H_kv, D], lse is [B, H, Lq], all dense
 * row-major fp64.  Positions: q_pos(i) = q_offset + i, kv_pos(j) = kv_offset + j.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

typedef struct {
    int64_t B, H, Hkv, Lq, Lkv, D, q_offset, kv_offset;
    int causal;
    double scale;
    int64_t win_c, win_w;   /* local window: chunk length and chunks per window (0: none) */
} dims_t;

static inline const double* qrow(const double* q, const dims_t* d, int64_t b, int64_t i, int64_t h) {
    return q + ((b * d->Lq + i) * d->H + h) * d->D;
}
static inline const double* kvrow(const double* k, const dims_t* d, int64_t b, int64_t j, int64_t g) {
    return k + ((b * d->Lkv + j) * d->Hkv + g) * d->D;
}
/* Causal visibility; with a local window (DISTFLASHATTN App. F: a worker
 * attends only to its own and the neighbouring chunks) a key must also lie in
 * the query's chunk or one of the win_w - 1 chunks before it. */
static inline int visible(const dims_t* d, int64_t i, int64_t j) {
    const int64_t qp = d->q_offset + i, kp = d->kv_offset + j;
    if (!d->causal) return 1;
    if (kp > qp) return 0;
    if (d->win_w > 0 && kp / d->win_c < qp / d->win_c - (d->win_w - 1)) return 0;
    return 1;
}

/* One full score row s[0..Lkv) for query (b, h, i); masked keys get -inf.
 * Returns lse_i = max + ln(sum exp(s - max)), or -inf if no key is visible. */
static double score_row(const double* q, const double* k, const dims_t* d,
                        int64_t b, int64_t h, int64_t i, double* s) {
    const int64_t g = h / (d->H / d->Hkv);
    const double* qi = qrow(q, d, b, i, h);
    double m = -INFINITY;
    for (int64_t j = 0; j < d->Lkv; ++j) {
        if (!visible(d, i, j)) { s[j] = -INFINITY; continue; }
        const double* kj = kvrow(k, d, b, j, g);
        double acc = 0.0;
        for (int64_t e = 0; e < d->D; ++e) acc += qi[e] * kj[e];
        s[j] = d->scale * acc;
        if (s[j] > m) m = s[j];
    }
    if (m == -INFINITY) return -INFINITY;
    double sum = 0.0;
    for (int64_t j = 0; j < d->Lkv; ++j)
        if (s[j] != -INFINITY) sum += exp(s[j] - m);
    return m + log(sum);
}

/* P row from a score row and its lse (0 where masked or the row is empty). */
static void prob_row(const dims_t* d, const double* s, double lse, double* p) {
    for (int64_t j = 0; j < d->Lkv; ++j)
        p[j] = (lse == -INFINITY || s[j] == -INFINITY) ? 0.0 : exp(s[j] - lse);
}

/* Forward for one query row: O_i = sum_j P_ij v_j, lse_i. */
static void fwd_one(const double* q, const double* k, const double* v, const dims_t* d,
                    int64_t b, int64_t h, int64_t i, double* s, double* o, double* lse) {
    const int64_t g = h / (d->H / d->Hkv);
    double l = score_row(q, k, d, b, h, i, s);
    prob_row(d, s, l, s);                     /* s now holds P */
    for (int64_t e = 0; e < d->D; ++e) o[e] = 0.0;
    for (int64_t j = 0; j < d->Lkv; ++j) {
        if (s[j] == 0.0) continue;
        const double* vj = kvrow(v, d, b, j, g);
        for (int64_t e = 0; e < d->D; ++e) o[e] += s[j] * vj[e];
    }
    *lse = l;
}

static int check_dims(const dims_t* d) {
    if (d->B < 0 || d->H <= 0 || d->Hkv <= 0 || d->Lq < 0 || d->Lkv < 0 || d->D <= 0) return 1;
    if (d->H % d->Hkv != 0) return 1;
    return 0;
}

static void set_threads(int nthreads) {
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
}

int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Full forward over every (b, h, i). */
static int fwd_all(const double* q, const double* k, const double* v, dims_t d,
                   double* O, double* lse, int nthreads) {
    const int64_t B = d.B, H = d.H, Lq = d.Lq, Lkv = d.Lkv, D = d.D;
    if (check_dims(&d)) return 1;
    set_threads(nthreads);
    const int64_t total = B * H * Lq;
    int err = 0;
#pragma omp parallel
    {
        double* s = (double*)malloc(sizeof(double) * (size_t)(Lkv > 0 ? Lkv : 1));
        if (!s) {
#pragma omp atomic write
            err = 2;
        } else {
#pragma omp for schedule(dynamic, 16)
            for (int64_t t = 0; t < total; ++t) {
                int64_t i = t % Lq, h = (t / Lq) % H, b = t / (Lq * H);
                fwd_one(q, k, v, &d, b, h, i, s, O + ((b * Lq + i) * H + h) * D,
                        lse + (b * H + h) * Lq + i);
            }
            free(s);
        }
    }
    return err;
}

int oracle_fwd(const double* q, const double* k, const double* v,
               int64_t B, int64_t H, int64_t Hkv, int64_t Lq, int64_t Lkv, int64_t D,
               int64_t q_offset, int64_t kv_offset, int causal, double scale,
               double* O, double* lse, int nthreads) {
    dims_t d = {B, H, Hkv, Lq, Lkv, D, q_offset, kv_offset, causal, scale, 0, 0};
    return fwd_all(q, k, v, d, O, lse, nthreads);
}

/* Causal forward restricted to a local window of win_w chunks of win_c tokens. */
int oracle_fwd_local(const double* q, const double* k, const double* v,
                     int64_t B, int64_t H, int64_t Hkv, int64_t Lq, int64_t Lkv, int64_t D,
                     int64_t q_offset, int64_t kv_offset, double scale, int64_t win_c, int64_t win_w,
                     double* O, double* lse, int nthreads) {
    if (win_c <= 0 || win_w <= 0) return 1;
    dims_t d = {B, H, Hkv, Lq, Lkv, D, q_offset, kv_offset, 1, scale, win_c, win_w};
    return fwd_all(q, k, v, d, O, lse, nthreads);
}

/* Forward on selected rows: rows is [n, 3] of (b, h, i); O_rows [n, D], lse_rows [n]. */
int oracle_fwd_rows(const double* q, const double* k, const double* v,
                    int64_t B, int64_t H, int64_t Hkv, int64_t Lq, int64_t Lkv, int64_t D,
                    int64_t q_offset, int64_t kv_offset, int causal, double scale,
                    const int64_t* rows, int64_t n, double* O_rows, double* lse_rows, int nthreads) {
    dims_t d = {B, H, Hkv, Lq, Lkv, D, q_offset, kv_offset, causal, scale};
    if (check_dims(&d)) return 1;
    for (int64_t r = 0; r < n; ++r)
        if (rows[3 * r] < 0 || rows[3 * r] >= B || rows[3 * r + 1] < 0 || rows[3 * r + 1] >= H ||
            rows[3 * r + 2] < 0 || rows[3 * r + 2] >= Lq) return 1;
    set_threads(nthreads);
    int err = 0;
#pragma omp parallel
    {
        double* s = (double*)malloc(sizeof(double) * (size_t)(Lkv > 0 ? Lkv : 1));
        if (!s) {
#pragma omp atomic write
            err = 2;
        } else {
#pragma omp for schedule(dynamic, 1)
            for (int64_t r = 0; r < n; ++r)
                fwd_one(q, k, v, &d, rows[3 * r], rows[3 * r + 1], rows[3 * r + 2], s,
                        O_rows + r * D, lse_rows + r);
            free(s);
        }
    }
    return err;
}

/* Backward quantities of one query row: P row (in p), dP row (in dp), Delta, dS row (in dp). */
static void bwd_row(const double* q, const double* k, const double* v, const double* dO,
                    const dims_t* d, int64_t b, int64_t h, int64_t i, double* p, double* dp) {
    const int64_t g = h / (d->H / d->Hkv);
    double l = score_row(q, k, d, b, h, i, p);
    prob_row(d, p, l, p);
    const double* doi = qrow(dO, d, b, i, h);
    double delta = 0.0;
    for (int64_t j = 0; j < d->Lkv; ++j) {
        if (p[j] == 0.0) { dp[j] = 0.0; continue; }
        const double* vj = kvrow(v, d, b, j, g);
        double acc = 0.0;
        for (int64_t e = 0; e < d->D; ++e) acc += doi[e] * vj[e];
        dp[j] = acc;
        delta += p[j] * acc;
    }
    for (int64_t j = 0; j < d->Lkv; ++j) dp[j] = p[j] * (dp[j] - delta);   /* dS */
}

/* Full backward.  dK/dV are accumulated per thread and reduced at the end. */
static int bwd_all(const double* q, const double* k, const double* v, const double* dO, dims_t d,
                   double* dQ, double* dK, double* dV, int nthreads) {
    const int64_t B = d.B, H = d.H, Hkv = d.Hkv, Lq = d.Lq, Lkv = d.Lkv, D = d.D;
    const double scale = d.scale;
    if (check_dims(&d)) return 1;
    set_threads(nthreads);
    const int64_t kvn = B * Lkv * Hkv * D;
    memset(dK, 0, sizeof(double) * (size_t)kvn);
    memset(dV, 0, sizeof(double) * (size_t)kvn);
    const int64_t total = B * H * Lq;
    const int64_t G = H / Hkv;
    int err = 0;
#pragma omp parallel
    {
        double* p = (double*)malloc(sizeof(double) * (size_t)(Lkv > 0 ? Lkv : 1));
        double* ds = (double*)malloc(sizeof(double) * (size_t)(Lkv > 0 ? Lkv : 1));
        double* lk = (double*)calloc((size_t)(kvn > 0 ? kvn : 1), sizeof(double));
        double* lv = (double*)calloc((size_t)(kvn > 0 ? kvn : 1), sizeof(double));
        if (!p || !ds || !lk || !lv) {
#pragma omp atomic write
            err = 2;
        } else {
#pragma omp for schedule(dynamic, 16)
            for (int64_t t = 0; t < total; ++t) {
                int64_t i = t % Lq, h = (t / Lq) % H, b = t / (Lq * H), g = h / G;
                bwd_row(q, k, v, dO, &d, b, h, i, p, ds);
                const double* qi = qrow(q, &d, b, i, h);
                const double* doi = qrow(dO, &d, b, i, h);
                double* dqi = dQ + ((b * Lq + i) * H + h) * D;
                for (int64_t e = 0; e < D; ++e) dqi[e] = 0.0;
                for (int64_t j = 0; j < Lkv; ++j) {
                    if (p[j] == 0.0 && ds[j] == 0.0) continue;
                    const double* kj = kvrow(k, &d, b, j, g);
                    double* lkj = lk + ((b * Lkv + j) * Hkv + g) * D;
                    double* lvj = lv + ((b * Lkv + j) * Hkv + g) * D;
                    for (int64_t e = 0; e < D; ++e) {
                        dqi[e] += scale * ds[j] * kj[e];
                        lkj[e] += scale * ds[j] * qi[e];
                        lvj[e] += p[j] * doi[e];
                    }
                }
            }
#pragma omp critical
            {
                for (int64_t x = 0; x < kvn; ++x) { dK[x] += lk[x]; dV[x] += lv[x]; }
            }
        }
        free(p); free(ds); free(lk); free(lv);
    }
    return err;
}

int oracle_bwd(const double* q, const double* k, const double* v, const double* dO,
               int64_t B, int64_t H, int64_t Hkv, int64_t Lq, int64_t Lkv, int64_t D,
               int64_t q_offset, int64_t kv_offset, int causal, double scale,
               double* dQ, double* dK, double* dV, int nthreads) {
    dims_t d = {B, H, Hkv, Lq, Lkv, D, q_offset, kv_offset, causal, scale, 0, 0};
    return bwd_all(q, k, v, dO, d, dQ, dK, dV, nthreads);
}

/* Backward of oracle_fwd_local. */
int oracle_bwd_local(const double* q, const double* k, const double* v, const double* dO,
                     int64_t B, int64_t H, int64_t Hkv, int64_t Lq, int64_t Lkv, int64_t D,
                     int64_t q_offset, int64_t kv_offset, double scale, int64_t win_c, int64_t win_w,
                     double* dQ, double* dK, double* dV, int nthreads) {
    if (win_c <= 0 || win_w <= 0) return 1;
    dims_t d = {B, H, Hkv, Lq, Lkv, D, q_offset, kv_offset, 1, scale, win_c, win_w};
    return bwd_all(q, k, v, dO, d, dQ, dK, dV, nthreads);
}

/* dQ on selected query rows (row-local): rows [n,3] of (b, h, i); dQ_rows [n, D]. */
int oracle_dq_rows(const double* q, const double* k, const double* v, const double* dO,
                   int64_t B, int64_t H, int64_t Hkv, int64_t Lq, int64_t Lkv, int64_t D,
                   int64_t q_offset, int64_t kv_offset, int causal, double scale,
                   const int64_t* rows, int64_t n, double* dQ_rows, int nthreads) {
    dims_t d = {B, H, Hkv, Lq, Lkv, D, q_offset, kv_offset, causal, scale};
    if (check_dims(&d)) return 1;
    for (int64_t r = 0; r < n; ++r)
        if (rows[3 * r] < 0 || rows[3 * r] >= B || rows[3 * r + 1] < 0 || rows[3 * r + 1] >= H ||
            rows[3 * r + 2] < 0 || rows[3 * r + 2] >= Lq) return 1;
    set_threads(nthreads);
    const int64_t G = H / Hkv;
    int err = 0;
#pragma omp parallel
    {
        double* p = (double*)malloc(sizeof(double) * (size_t)(Lkv > 0 ? Lkv : 1));
        double* ds = (double*)malloc(sizeof(double) * (size_t)(Lkv > 0 ? Lkv : 1));
        if (!p || !ds) {
#pragma omp atomic write
            err = 2;
        } else {
#pragma omp for schedule(dynamic, 1)
            for (int64_t r = 0; r < n; ++r) {
                int64_t b = rows[3 * r], h = rows[3 * r + 1], i = rows[3 * r + 2], g = h / G;
                bwd_row(q, k, v, dO, &d, b, h, i, p, ds);
                double* out = dQ_rows + r * D;
                for (int64_t e = 0; e < D; ++e) out[e] = 0.0;
                for (int64_t j = 0; j < Lkv; ++j) {
                    if (ds[j] == 0.0) continue;
                    const double* kj = kvrow(k, &d, b, j, g);
                    for (int64_t e = 0; e < D; ++e) out[e] += scale * ds[j] * kj[e];
                }
            }
        }
        free(p); free(ds);
    }
    return err;
}

/* dK/dV on selected key rows: krows [n,3] of (b, g, j); dK_rows/dV_rows [n, D].
 * Each selected key sums over every query row of every head in its group. */
int oracle_dkv_rows(const double* q, const double* k, const double* v, const double* dO,
                    int64_t B, int64_t H, int64_t Hkv, int64_t Lq, int64_t Lkv, int64_t D,
                    int64_t q_offset, int64_t kv_offset, int causal, double scale,
                    const int64_t* krows, int64_t n, double* dK_rows, double* dV_rows, int nthreads) {
    dims_t d = {B, H, Hkv, Lq, Lkv, D, q_offset, kv_offset, causal, scale};
    if (check_dims(&d)) return 1;
    for (int64_t r = 0; r < n; ++r)
        if (krows[3 * r] < 0 || krows[3 * r] >= B || krows[3 * r + 1] < 0 || krows[3 * r + 1] >= Hkv ||
            krows[3 * r + 2] < 0 || krows[3 * r + 2] >= Lkv) return 1;
    set_threads(nthreads);
    const int64_t G = H / Hkv;
    memset(dK_rows, 0, sizeof(double) * (size_t)(n * D));
    memset(dV_rows, 0, sizeof(double) * (size_t)(n * D));
    /* Work unit: one (b, h, i) query row; it contributes to every selected key of
     * its batch and group.  Per-thread partial sums, reduced at the end. */
    const int64_t total = B * H * Lq;
    int err = 0;
#pragma omp parallel
    {
        double* p = (double*)malloc(sizeof(double) * (size_t)(Lkv > 0 ? Lkv : 1));
        double* ds = (double*)malloc(sizeof(double) * (size_t)(Lkv > 0 ? Lkv : 1));
        double* lk = (double*)calloc((size_t)(n * D > 0 ? n * D : 1), sizeof(double));
        double* lv = (double*)calloc((size_t)(n * D > 0 ? n * D : 1), sizeof(double));
        if (!p || !ds || !lk || !lv) {
#pragma omp atomic write
            err = 2;
        } else {
#pragma omp for schedule(dynamic, 4)
            for (int64_t t = 0; t < total; ++t) {
                int64_t i = t % Lq, h = (t / Lq) % H, b = t / (Lq * H), g = h / G;
                /* Skip rows that see none of the selected keys. */
                int any = 0;
                for (int64_t r = 0; r < n && !any; ++r)
                    any = krows[3 * r] == b && krows[3 * r + 1] == g && visible(&d, i, krows[3 * r + 2]);
                if (!any) continue;
                bwd_row(q, k, v, dO, &d, b, h, i, p, ds);
                const double* qi = qrow(q, &d, b, i, h);
                const double* doi = qrow(dO, &d, b, i, h);
                for (int64_t r = 0; r < n; ++r) {
                    if (krows[3 * r] != b || krows[3 * r + 1] != g) continue;
                    int64_t j = krows[3 * r + 2];
                    for (int64_t e = 0; e < D; ++e) {
                        lk[r * D + e] += scale * ds[j] * qi[e];
                        lv[r * D + e] += p[j] * doi[e];
                    }
                }
            }
#pragma omp critical
            {
                for (int64_t x = 0; x < n * D; ++x) { dK_rows[x] += lk[x]; dV_rows[x] += lv[x]; }
            }
        }
        free(p); free(ds); free(lk); free(lv);
    }
    return err;
}

/* Rescale-and-merge of two partial results over the same query rows
 * (DISTFLASHATTN §3.2: helpers return partial output plus softmax statistics
 * for the owner to rescale).  For one row with partials (O_a, lse_a), (O_b, lse_b):
 *   lse = ln(exp(lse_a) + exp(lse_b)),  O = exp(lse_a - lse) O_a + exp(lse_b - lse) O_b.
 * A partial with lse = -inf has weight 0; both -inf gives O = 0, lse = -inf.
 * O_* are [B, L, H, D]; lse_* are [B, H, L]. */
int oracle_merge(const double* Oa, const double* lse_a, const double* Ob, const double* lse_b,
                 int64_t B, int64_t H, int64_t L, int64_t D, double* O, double* lse) {
    if (B < 0 || H <= 0 || L < 0 || D <= 0) return 1;
    for (int64_t b = 0; b < B; ++b)
        for (int64_t h = 0; h < H; ++h)
            for (int64_t i = 0; i < L; ++i) {
                double la = lse_a[(b * H + h) * L + i], lb = lse_b[(b * H + h) * L + i];
                double m = la > lb ? la : lb, l, wa, wb;
                if (m == -INFINITY) { l = -INFINITY; wa = 0.0; wb = 0.0; }
                else {
                    l = m + log(exp(la - m) + exp(lb - m));
                    wa = exp(la - l);
                    wb = exp(lb - l);
                }
                const double* oa = Oa + ((b * L + i) * H + h) * D;
                const double* ob = Ob + ((b * L + i) * H + h) * D;
                double* o = O + ((b * L + i) * H + h) * D;
                for (int64_t e = 0; e < D; ++e) o[e] = wa * oa[e] + wb * ob[e];
                lse[(b * H + h) * L + i] = l;
            }
    return 0;
}

/* Delta_i = sum_j P_ij dP_ij over every visible key of row (b, h, i)
 * (the explicit definition; equal to <dO_i, O_i>).  delta is [B, H, Lq]. */
int oracle_delta(const double* q, const double* k, const double* v, const double* dO,
                 int64_t B, int64_t H, int64_t Hkv, int64_t Lq, int64_t Lkv, int64_t D,
                 int64_t q_offset, int64_t kv_offset, int causal, double scale,
                 double* delta, int nthreads) {
    dims_t d = {B, H, Hkv, Lq, Lkv, D, q_offset, kv_offset, causal, scale};
    if (check_dims(&d)) return 1;
    set_threads(nthreads);
    const int64_t total = B * H * Lq;
    const int64_t G = H / Hkv;
    int err = 0;
#pragma omp parallel
    {
        double* p = (double*)malloc(sizeof(double) * (size_t)(Lkv > 0 ? Lkv : 1));
        if (!p) {
#pragma omp atomic write
            err = 2;
        } else {
#pragma omp for schedule(dynamic, 16)
            for (int64_t t = 0; t < total; ++t) {
                int64_t i = t % Lq, h = (t / Lq) % H, b = t / (Lq * H), g = h / G;
                double l = score_row(q, k, &d, b, h, i, p);
                prob_row(&d, p, l, p);
                const double* doi = qrow(dO, &d, b, i, h);
                double acc = 0.0;
                for (int64_t j = 0; j < Lkv; ++j) {
                    if (p[j] == 0.0) continue;
                    const double* vj = kvrow(v, &d, b, j, g);
                    double dp = 0.0;
                    for (int64_t e = 0; e < D; ++e) dp += doi[e] * vj[e];
                    acc += p[j] * dp;
                }
                delta[(b * H + h) * Lq + i] = acc;
            }
        }
        free(p);
    }
    return err;
}

/* Backward of one (query chunk, key chunk) pair -- the per-worker backward
 * step of DISTFLASHATTN §3.3 (the helper's partial gradients, computed from
 * the owner's saved output statistics).  The rows' lse_i and Delta_i are the
 * global ones (over the whole key sequence), given as inputs [B, H, Lq].  For
 * the pair's visible (i, j):
 *   P_ij = exp(s_ij - lse_i),  dS_ij = P_ij (<dO_i, v_j> - Delta_i)
 *   dQ_i = scale sum_j dS_ij k_j,  dK_j = scale sum_i dS_ij q_i,  dV_j = sum_i P_ij dO_i
 * restricted to this chunk's keys (dQ) and queries (dK, dV).  Summed over the
 * key chunks (dQ) or query chunks (dK, dV) they are the full gradients.
 * Outputs are overwritten.  A row with lse_i = -inf contributes nothing. */
int oracle_chunk_bwd(const double* q, const double* k, const double* v, const double* dO,
                     const double* lse, const double* delta,
                     int64_t B, int64_t H, int64_t Hkv, int64_t Lq, int64_t Lkv, int64_t D,
                     int64_t q_offset, int64_t kv_offset, int causal, double scale,
                     double* dQ, double* dK, double* dV, int nthreads) {
    dims_t d = {B, H, Hkv, Lq, Lkv, D, q_offset, kv_offset, causal, scale};
    if (check_dims(&d)) return 1;
    set_threads(nthreads);
    const int64_t kvn = B * Lkv * Hkv * D;
    memset(dK, 0, sizeof(double) * (size_t)kvn);
    memset(dV, 0, sizeof(double) * (size_t)kvn);
    const int64_t total = B * H * Lq;
    const int64_t G = H / Hkv;
    int err = 0;
#pragma omp parallel
    {
        double* lk = (double*)calloc((size_t)(kvn > 0 ? kvn : 1), sizeof(double));
        double* lv = (double*)calloc((size_t)(kvn > 0 ? kvn : 1), sizeof(double));
        if (!lk || !lv) {
#pragma omp atomic write
            err = 2;
        } else {
#pragma omp for schedule(dynamic, 16)
            for (int64_t t = 0; t < total; ++t) {
                int64_t i = t % Lq, h = (t / Lq) % H, b = t / (Lq * H), g = h / G;
                const double* qi = qrow(q, &d, b, i, h);
                const double* doi = qrow(dO, &d, b, i, h);
                const double li = lse[(b * H + h) * Lq + i], di = delta[(b * H + h) * Lq + i];
                double* dqi = dQ + ((b * Lq + i) * H + h) * D;
                for (int64_t e = 0; e < D; ++e) dqi[e] = 0.0;
                if (li == -INFINITY) continue;
                for (int64_t j = 0; j < Lkv; ++j) {
                    if (!visible(&d, i, j)) continue;
                    const double* kj = kvrow(k, &d, b, j, g);
                    const double* vj = kvrow(v, &d, b, j, g);
                    double s = 0.0, dp = 0.0;
                    for (int64_t e = 0; e < D; ++e) { s += qi[e] * kj[e]; dp += doi[e] * vj[e]; }
                    const double p = exp(scale * s - li);
                    const double ds = p * (dp - di);
                    double* lkj = lk + ((b * Lkv + j) * Hkv + g) * D;
                    double* lvj = lv + ((b * Lkv + j) * Hkv + g) * D;
                    for (int64_t e = 0; e < D; ++e) {
                        dqi[e] += scale * ds * kj[e];
                        lkj[e] += scale * ds * qi[e];
                        lvj[e] += p * doi[e];
                    }
                }
            }
#pragma omp critical
            {
                for (int64_t x = 0; x < kvn; ++x) { dK[x] += lk[x]; dV[x] += lv[x]; }
            }
        }
        free(lk); free(lv);
    }
    return err;
}
