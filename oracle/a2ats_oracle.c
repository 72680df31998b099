/*
 * a2ats_oracle.c -- plain fp64 CPU oracle of the A2ATS hot path.
 *
 * TEST INFRASTRUCTURE ONLY (see a2ats_oracle.h).  Written for a reader who
 * checks each routine against the pages by eye: straight loops, fp64, no
 * blocking, no reordering beyond what each definition states.
 */
#include "a2ats_oracle.h"

#include <math.h>
#include <pthread.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------ */
/* Windowed RoPE.  "A2ATS-adapted" page, paper-fidelity section, "Windowed   */
/* RoPE (Eq. 11-12)": a key within the trailing window is rotated at its     */
/* own position p; every other key takes one common rotation (Eq. 12 leaves  */
/* them unrotated, i.e. far_offset = 0).  The v0.39.0 page, "How it works"    */
/* step 4: window <= 0 -> every key far; window >= length -> every key exact. */
/* ------------------------------------------------------------------------ */
void orc_rope_row(const double* x, double* y, int64_t d, double pos, double base,
                  int interleaved) {
    int64_t half = d / 2;
    for (int64_t i = 0; i < half; i++) {
        double theta = pos * pow(base, -2.0 * (double)i / (double)d);
        double c = cos(theta), s = sin(theta);
        int64_t a = interleaved ? 2 * i : i;
        int64_t b = interleaved ? 2 * i + 1 : i + half;
        double xa = x[a], xb = x[b];
        y[a] = xa * c - xb * s;
        y[b] = xa * s + xb * c;
    }
}

void orc_windowed_rope(const double* x, double* y, int64_t rows, int64_t d,
                       const int64_t* p, const int64_t* t, int64_t window,
                       double far_offset, double base, int interleaved) {
    for (int64_t r = 0; r < rows; r++) {
        int64_t dist = t[r] - p[r];
        int near = window > 0 && dist >= 0 && dist < window;
        double pos = near ? (double)p[r] : far_offset;
        orc_rope_row(x + r * d, y + r * d, d, pos, base, interleaved);
    }
}

/* ------------------------------------------------------------------------ */
/* Query second moment.  API page, a2ats_query_second_moment: H = E[q^T q]   */
/* over the M calibration queries (paper Eq. 10), with `ridge` added to     */
/* each diagonal entry to keep H positive definite.  Not mean-centred.      */
/* ------------------------------------------------------------------------ */
void orc_query_second_moment(const double* q, int64_t M, int64_t d, double ridge,
                             double* h) {
    for (int64_t a = 0; a < d; a++) {
        for (int64_t b = 0; b < d; b++) {
            double s = 0.0;
            for (int64_t m = 0; m < M; m++) s += q[m * d + a] * q[m * d + b];
            h[a * d + b] = (M > 0 ? s / (double)M : 0.0) + (a == b ? ridge : 0.0);
        }
    }
}

/* ------------------------------------------------------------------------ */
/* Cholesky factor.  API page, a2ats_cholesky_factor: lower-triangular L     */
/* with H = L L^T (paper Eq. 15).  Textbook Cholesky-Banachiewicz.           */
/* ------------------------------------------------------------------------ */
int orc_cholesky(const double* h, int64_t d, double* l) {
    memset(l, 0, sizeof(double) * (size_t)(d * d));
    for (int64_t i = 0; i < d; i++) {
        for (int64_t j = 0; j <= i; j++) {
            double s = h[i * d + j];
            for (int64_t k = 0; k < j; k++) s -= l[i * d + k] * l[j * d + k];
            if (i == j) {
                if (!(s > 0.0)) return (int)(i + 1);
                l[i * d + i] = sqrt(s);
            } else {
                l[i * d + j] = s / l[j * d + j];
            }
        }
    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Row-parallel helper: run fn(ctx, begin, end) over [0, n) on nthreads.     */
/* ------------------------------------------------------------------------ */
typedef void (*row_fn)(void* ctx, int64_t r0, int64_t r1);
typedef struct { row_fn fn; void* ctx; int64_t r0, r1; } row_job;

static void* run_job(void* arg) {
    row_job* j = (row_job*)arg;
    j->fn(j->ctx, j->r0, j->r1);
    return NULL;
}

static void parallel_rows(row_fn fn, void* ctx, int64_t n, int nthreads) {
    if (nthreads <= 1 || n < 2) { fn(ctx, 0, n); return; }
    if (nthreads > 256) nthreads = 256;
    pthread_t tid[256];
    row_job jobs[256];
    int64_t per = (n + nthreads - 1) / nthreads;
    int started = 0;
    for (int t = 0; t < nthreads; t++) {
        int64_t r0 = t * per, r1 = r0 + per < n ? r0 + per : n;
        if (r0 >= r1) break;
        jobs[t] = (row_job){fn, ctx, r0, r1};
        if (pthread_create(&tid[t], NULL, run_job, &jobs[t]) != 0) {
            run_job(&jobs[t]);
            tid[t] = 0;
        }
        started = t + 1;
    }
    for (int t = 0; t < started; t++)
        if (tid[t]) pthread_join(tid[t], NULL);
}

/* Keep the two smallest values; ties keep the lower index (first seen). */
static void keep_best2(double v, int32_t j, double* b1, int32_t* j1, double* b2) {
    if (v < *b1) { *b2 = *b1; *b1 = v; *j1 = j; }
    else if (v < *b2) { *b2 = v; }
}

/* ------------------------------------------------------------------------ */
/* H-weighted assignment, literal form.  API page,                          */
/* a2ats_h_weighted_assignment: f'(k; C) = argmin_j (k - c_j) H (k - c_j)^T  */
/* (paper Eq. 14).                                                           */
/* ------------------------------------------------------------------------ */
typedef struct {
    const double *x, *c, *h; int64_t d, K;
    int32_t* code; double *d1, *d2;
} quad_ctx;

static void quad_rows(void* vctx, int64_t r0, int64_t r1) {
    quad_ctx* q = (quad_ctx*)vctx;
    int64_t d = q->d;
    double* diff = (double*)malloc(sizeof(double) * (size_t)d);
    for (int64_t r = r0; r < r1; r++) {
        const double* x = q->x + r * d;
        double b1 = INFINITY, b2 = INFINITY; int32_t j1 = 0;
        for (int64_t j = 0; j < q->K; j++) {
            const double* cj = q->c + j * d;
            for (int64_t a = 0; a < d; a++) diff[a] = x[a] - cj[a];
            double v = 0.0;
            for (int64_t a = 0; a < d; a++) {
                double row = 0.0;
                for (int64_t b = 0; b < d; b++) row += q->h[a * d + b] * diff[b];
                v += diff[a] * row;
            }
            keep_best2(v, (int32_t)j, &b1, &j1, &b2);
        }
        q->code[r] = j1; q->d1[r] = b1; q->d2[r] = b2;
    }
    free(diff);
}

void orc_assign_quadratic(const double* x, int64_t n, int64_t d, const double* c,
                          int64_t K, const double* h, int32_t* code, double* d1,
                          double* d2, int nthreads) {
    quad_ctx ctx = {x, c, h, d, K, code, d1, d2};
    parallel_rows(quad_rows, &ctx, n, nthreads);
}

/* ------------------------------------------------------------------------ */
/* H-weighted assignment through the Cholesky identity.  API page,          */
/* a2ats_h_weighted_assignment and a2ats_cholesky_factor (Eq. 16-18): with   */
/* H = L L^T the quadratic form is |kL - c_jL|^2, a plain Euclidean          */
/* distance between z = kL and the transformed centroid c'_j = c_jL.         */
/* ------------------------------------------------------------------------ */
typedef struct {
    const double *x, *cp; int64_t d, K; const double* l;
    int32_t* code; double *d1, *d2;
} chol_ctx;

static void times_l(const double* v, const double* l, int64_t d, double* out) {
    /* out_b = sum_a v_a L_ab (row vector times L); L == NULL is the identity */
    for (int64_t b = 0; b < d; b++) {
        if (!l) { out[b] = v[b]; continue; }
        double s = 0.0;
        for (int64_t a = 0; a < d; a++) s += v[a] * l[a * d + b];
        out[b] = s;
    }
}

static void chol_rows(void* vctx, int64_t r0, int64_t r1) {
    chol_ctx* q = (chol_ctx*)vctx;
    int64_t d = q->d;
    double* z = (double*)malloc(sizeof(double) * (size_t)d);
    for (int64_t r = r0; r < r1; r++) {
        times_l(q->x + r * d, q->l, d, z);
        double b1 = INFINITY, b2 = INFINITY; int32_t j1 = 0;
        for (int64_t j = 0; j < q->K; j++) {
            const double* cj = q->cp + j * d;
            double v = 0.0;
            for (int64_t b = 0; b < d; b++) { double e = z[b] - cj[b]; v += e * e; }
            keep_best2(v, (int32_t)j, &b1, &j1, &b2);
        }
        q->code[r] = j1; q->d1[r] = b1; q->d2[r] = b2;
    }
    free(z);
}

void orc_assign_cholesky(const double* x, int64_t n, int64_t d, const double* c,
                         int64_t K, const double* l, int32_t* code, double* d1,
                         double* d2, int nthreads) {
    double* cp = (double*)malloc(sizeof(double) * (size_t)(K * d));
    for (int64_t j = 0; j < K; j++) times_l(c + j * d, l, d, cp + j * d);
    chol_ctx ctx = {x, cp, d, K, l, code, d1, d2};
    parallel_rows(chol_rows, &ctx, n, nthreads);
    free(cp);
}

/* ------------------------------------------------------------------------ */
/* Cosine-blend assignment.  API page, a2ats_query_aware_assignment:        */
/* score(c) = beta * (-|x - c|^2 normalised) + (1 - beta) * cos(query, c),   */
/* the error normalised per row by its largest value over the codebook;      */
/* argmax over c.  beta = 1 is plain nearest-centroid VQ (v0.39.0 page,      */
/* honesty point 3), taken here as the argmin of the distance itself.        */
/* ------------------------------------------------------------------------ */
typedef struct {
    const double *x, *c, *q; int64_t d, K, q_stride; double beta;
    const double* cnorm;
    int32_t* code; double *s1, *s2;
} blend_ctx;

static void blend_rows(void* vctx, int64_t r0, int64_t r1) {
    blend_ctx* p = (blend_ctx*)vctx;
    int64_t d = p->d, K = p->K;
    double* e = (double*)malloc(sizeof(double) * (size_t)K);
    for (int64_t r = r0; r < r1; r++) {
        const double* x = p->x + r * d;
        for (int64_t j = 0; j < K; j++) {
            double v = 0.0;
            for (int64_t a = 0; a < d; a++) { double t = x[a] - p->c[j * d + a]; v += t * t; }
            e[j] = v;
        }
        if (p->beta == 1.0) {
            double b1 = INFINITY, b2 = INFINITY; int32_t j1 = 0;
            for (int64_t j = 0; j < K; j++) keep_best2(e[j], (int32_t)j, &b1, &j1, &b2);
            p->code[r] = j1; p->s1[r] = b1; p->s2[r] = b2;
            continue;
        }
        double m = 0.0;
        for (int64_t j = 0; j < K; j++) if (e[j] > m) m = e[j];
        const double* q = p->q + r * p->q_stride;
        double qn = 0.0;
        for (int64_t a = 0; a < d; a++) qn += q[a] * q[a];
        qn = sqrt(qn);
        double b1 = -INFINITY, b2 = -INFINITY; int32_t j1 = 0;
        for (int64_t j = 0; j < K; j++) {
            double err = m > 0.0 ? e[j] / m : 0.0;
            double cosv = 0.0;
            if (qn > 0.0 && p->cnorm[j] > 0.0) {
                double dot = 0.0;
                for (int64_t a = 0; a < d; a++) dot += q[a] * p->c[j * d + a];
                cosv = dot / (qn * p->cnorm[j]);
            }
            double s = -p->beta * err + (1.0 - p->beta) * cosv;
            if (s > b1) { b2 = b1; b1 = s; j1 = (int32_t)j; }
            else if (s > b2) { b2 = s; }
        }
        p->code[r] = j1; p->s1[r] = b1; p->s2[r] = b2;
    }
    free(e);
}

void orc_assign_blend(const double* x, int64_t n, int64_t d, const double* c, int64_t K,
                      const double* q, int64_t q_stride, double beta, int32_t* code,
                      double* s1, double* s2, int nthreads) {
    double* cnorm = (double*)malloc(sizeof(double) * (size_t)K);
    for (int64_t j = 0; j < K; j++) {
        double v = 0.0;
        for (int64_t a = 0; a < d; a++) v += c[j * d + a] * c[j * d + a];
        cnorm[j] = sqrt(v);
    }
    blend_ctx ctx = {x, c, q, d, K, q_stride, beta, cnorm, code, s1, s2};
    parallel_rows(blend_rows, &ctx, n, nthreads);
    free(cnorm);
}

/* ------------------------------------------------------------------------ */
/* Retrieval split.  API page, a2ats_select_retrieval_set: the retrieval    */
/* set holds the ceil(retrieval_fraction * N) keys whose cosine with the    */
/* query is largest; with the bulk it partitions 0..N-1.                    */
/* Here: a full sort by (score descending, index ascending).                 */
/* ------------------------------------------------------------------------ */
typedef struct { double s; int32_t i; } scored;

static int by_score_then_index(const void* a, const void* b) {
    const scored* x = (const scored*)a;
    const scored* y = (const scored*)b;
    if (x->s > y->s) return -1;
    if (x->s < y->s) return 1;
    return (x->i > y->i) - (x->i < y->i);
}

static int by_value(const void* a, const void* b) {
    int32_t x = *(const int32_t*)a, y = *(const int32_t*)b;
    return (x > y) - (x < y);
}

int64_t orc_select_retrieval_set(const double* keys, int64_t n, int64_t d,
                                 const double* q, double fraction, int32_t* perm,
                                 double* scores, double* kth) {
    double qn = 0.0;
    for (int64_t a = 0; a < d; a++) qn += q[a] * q[a];
    qn = sqrt(qn);
    scored* s = (scored*)malloc(sizeof(scored) * (size_t)(n > 0 ? n : 1));
    for (int64_t i = 0; i < n; i++) {
        double dot = 0.0, kn = 0.0;
        for (int64_t a = 0; a < d; a++) {
            dot += keys[i * d + a] * q[a];
            kn += keys[i * d + a] * keys[i * d + a];
        }
        kn = sqrt(kn);
        double v = (kn > 0.0 && qn > 0.0) ? dot / (kn * qn) : 0.0;
        s[i].s = v; s[i].i = (int32_t)i;
        if (scores) scores[i] = v;
    }
    int64_t count = (int64_t)ceil(fraction * (double)n);
    if (count > n) count = n;
    if (count < 0) count = 0;
    qsort(s, (size_t)n, sizeof(scored), by_score_then_index);
    for (int64_t i = 0; i < n; i++) perm[i] = s[i].i;
    if (kth) *kth = count > 0 ? s[count - 1].s : INFINITY;
    qsort(perm, (size_t)count, sizeof(int32_t), by_value);
    qsort(perm + count, (size_t)(n - count), sizeof(int32_t), by_value);
    free(s);
    return count;
}

/* ------------------------------------------------------------------------ */
/* Code-based attention-score estimation and top-K token retrieval.         */
/* "A2ATS-adapted" page, paper-fidelity section, "Windowed RoPE (Eq.         */
/* 11-12)": far keys stay in the unrotated frame and the constant far        */
/* relative position b rides on the query, u_ij = q_i R_b k_j^T; keys inside */
/* the window keep exact RoPE.  The paper's abstract: the attention score    */
/* is approximated through the vector-quantised keys so that the top-K       */
/* tokens are retrieved.  Reading: with q the decode query before RoPE and   */
/* t its position,                                                           */
/*   near row j (0 <= t - j < window):  u_j = RoPE(q, t) . RoPE(k_j, j)       */
/*   far row j:                         u_j = RoPE(q, b) . c_{code_j}         */
/* (a code outside [0, K) scores 0), and the retrieved set is the top        */
/* ceil(fraction n) rows by (u desc, index asc), both halves of perm in      */
/* ascending order as the split writes them.                                 */
/* ------------------------------------------------------------------------ */
int64_t orc_code_attention_topk(const double* keys, int64_t n, int64_t d, int64_t t,
                                const int32_t* codes, const double* codebook, int64_t K,
                                const double* q, int64_t window, double far_b, double base,
                                int interleaved, double fraction, int32_t* perm,
                                double* scores, double* kth) {
    double* qn = (double*)malloc(sizeof(double) * (size_t)d);
    double* qf = (double*)malloc(sizeof(double) * (size_t)d);
    double* kr = (double*)malloc(sizeof(double) * (size_t)d);
    orc_rope_row(q, qn, d, (double)t, base, interleaved);
    orc_rope_row(q, qf, d, far_b, base, interleaved);
    scored* s = (scored*)malloc(sizeof(scored) * (size_t)(n > 0 ? n : 1));
    for (int64_t j = 0; j < n; j++) {
        int64_t dist = t - j;
        int near = window > 0 && dist >= 0 && dist < window;
        double u = 0.0;
        if (near) {
            orc_rope_row(keys + j * d, kr, d, (double)j, base, interleaved);
            for (int64_t a = 0; a < d; a++) u += qn[a] * kr[a];
        } else if (codes[j] >= 0 && codes[j] < K) {
            const double* c = codebook + (int64_t)codes[j] * d;
            for (int64_t a = 0; a < d; a++) u += qf[a] * c[a];
        }
        s[j].s = u;
        s[j].i = (int32_t)j;
        if (scores) scores[j] = u;
    }
    int64_t count = (int64_t)ceil(fraction * (double)n);
    if (count > n) count = n;
    if (count < 0) count = 0;
    qsort(s, (size_t)n, sizeof(scored), by_score_then_index);
    for (int64_t i = 0; i < n; i++) perm[i] = s[i].i;
    if (kth) *kth = count > 0 ? s[count - 1].s : INFINITY;
    qsort(perm, (size_t)count, sizeof(int32_t), by_value);
    qsort(perm + count, (size_t)(n - count), sizeof(int32_t), by_value);
    free(s);
    free(kr);
    free(qf);
    free(qn);
    return count;
}

/* ------------------------------------------------------------------------ */
/* Dequantisation.  v0.39.0 page, "How it works", step 3: a key is          */
/* reconstructed from its assigned centroid, k ~ c_{code}.  Row j of out is */
/* codebook row codes[j] (zeros for a code outside [0, K)).                 */
/* ------------------------------------------------------------------------ */
void orc_dequantize(const int32_t* codes, int64_t n, const double* codebook, int64_t K,
                    int64_t d, double* out) {
    for (int64_t j = 0; j < n; j++) {
        int32_t c = codes[j];
        for (int64_t a = 0; a < d; a++)
            out[j * d + a] = (c >= 0 && c < K) ? codebook[(int64_t)c * d + a] : 0.0;
    }
}

/* ------------------------------------------------------------------------ */
/* The change of variables of the Cholesky route.  API page,                */
/* a2ats_cholesky_factor: with H = L L^T, (k - c) H (k - c)^T equals         */
/* |z_k - z_c|^2 for z = k L, so k-means in z is the H-weighted objective.  */
/* orc_cholesky_rows maps rows to z; orc_cholesky_solve_rows maps z-space   */
/* rows (the centroids k-means finds there) back: c with c L = z, by back   */
/* substitution from the last column (L lower triangular, so column b of    */
/* c L only involves c_a for a >= b).                                       */
/* ------------------------------------------------------------------------ */
void orc_cholesky_rows(const double* x, int64_t n, int64_t d, const double* l, double* z) {
    for (int64_t i = 0; i < n; i++) times_l(x + i * d, l, d, z + i * d);
}

void orc_cholesky_solve_rows(const double* z, int64_t n, int64_t d, const double* l,
                             double* c) {
    for (int64_t i = 0; i < n; i++) {
        const double* zi = z + i * d;
        double* ci = c + i * d;
        for (int64_t b = d - 1; b >= 0; b--) {
            double s = zi[b];
            for (int64_t a = b + 1; a < d; a++) s -= ci[a] * l[a * d + b];
            ci[b] = s / l[b * d + b];
        }
    }
}

/* ------------------------------------------------------------------------ */
/* Codebook calibration in z space.  API page, a2ats_cholesky_factor: once */
/* every row is multiplied by the factor (z = k L, H = L L^T), ordinary     */
/* squared distances between the z rows are the H-weighted ones, so the    */
/* codebook is trained by ordinary k-means++ on the z rows and taken back  */
/* by c = c_z L^-1.  Reading: k-means++ seeding, each centre               */
/* drawn with probability proportional to the squared distance D^2 to the    */
/* nearest centre chosen so far (the first uniformly), with the uniform      */
/* draws u[0..K) given as input: centre k is the first point whose running   */
/* sum of D^2 exceeds u[k] * (sum of D^2), or point floor(u[k] n) when every */
/* D^2 is 0 (the first centre: point floor(u[0] n)); then `iters` Lloyd      */
/* rounds: assign each point to its nearest centre (ties to the lower       */
/* index), move each centre to the mean of its points (a centre without     */
/* points stays).  objective[r] is the sum of squared distances after the   */
/* assignment of round r (r = iters: the final assignment, whose codes are   */
/* returned).                                                               */
/* ------------------------------------------------------------------------ */
static double sq_dist(const double* a, const double* b, int64_t d) {
    double s = 0.0;
    for (int64_t i = 0; i < d; i++) {
        double t = a[i] - b[i];
        s += t * t;
    }
    return s;
}

static double assign_all(const double* z, int64_t n, int64_t d, const double* c, int64_t K,
                         int32_t* codes) {
    double total = 0.0;
    for (int64_t i = 0; i < n; i++) {
        double best = INFINITY;
        int32_t bj = 0;
        for (int64_t j = 0; j < K; j++) {
            double v = sq_dist(z + i * d, c + j * d, d);
            if (v < best) {
                best = v;
                bj = (int32_t)j;
            }
        }
        codes[i] = bj;
        total += best;
    }
    return total;
}

void orc_kmeanspp(const double* z, int64_t n, int64_t d, int64_t K, const double* u,
                  int64_t iters, double* centroids, int32_t* codes, double* objective) {
    if (n <= 0 || K <= 0) return; /* no points to seed from */
    double* d2 = (double*)malloc(sizeof(double) * (size_t)n);
    int64_t first = (int64_t)floor(u[0] * (double)n);
    if (first >= n) first = n - 1;
    if (first < 0) first = 0;
    memcpy(centroids, z + first * d, sizeof(double) * (size_t)d);
    for (int64_t i = 0; i < n; i++) d2[i] = sq_dist(z + i * d, centroids, d);
    for (int64_t k = 1; k < K; k++) {
        double total = 0.0;
        for (int64_t i = 0; i < n; i++) total += d2[i];
        int64_t pick;
        if (total > 0.0) {
            double target = u[k] * total, run = 0.0;
            pick = n - 1;
            for (int64_t i = 0; i < n; i++) {
                run += d2[i];
                if (run > target) {
                    pick = i;
                    break;
                }
            }
        } else {
            pick = (int64_t)floor(u[k] * (double)n);
            if (pick >= n) pick = n - 1;
            if (pick < 0) pick = 0;
        }
        memcpy(centroids + k * d, z + pick * d, sizeof(double) * (size_t)d);
        for (int64_t i = 0; i < n; i++) {
            double v = sq_dist(z + i * d, centroids + k * d, d);
            if (v < d2[i]) d2[i] = v;
        }
    }
    double* sum = (double*)malloc(sizeof(double) * (size_t)(K * d));
    int64_t* cnt = (int64_t*)malloc(sizeof(int64_t) * (size_t)K);
    for (int64_t r = 0; r < iters; r++) {
        objective[r] = assign_all(z, n, d, centroids, K, codes);
        memset(sum, 0, sizeof(double) * (size_t)(K * d));
        memset(cnt, 0, sizeof(int64_t) * (size_t)K);
        for (int64_t i = 0; i < n; i++) {
            cnt[codes[i]]++;
            for (int64_t a = 0; a < d; a++) sum[codes[i] * d + a] += z[i * d + a];
        }
        for (int64_t j = 0; j < K; j++)
            if (cnt[j] > 0)
                for (int64_t a = 0; a < d; a++) centroids[j * d + a] = sum[j * d + a] / (double)cnt[j];
    }
    objective[iters] = assign_all(z, n, d, centroids, K, codes);
    free(cnt);
    free(sum);
    free(d2);
}
