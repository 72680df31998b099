/*
 * a2ats_oracle.h -- plain fp64 CPU oracle of the A2ATS hot path.
 *
 * TEST INFRASTRUCTURE ONLY.  This is the slow, obviously-correct reference the
 * CUDA library is checked against.  Only the tests, the package's smoke check
 * and the CPU-baseline leg of the benchmark may load it; the product path never
 * does.  It shares no code, header, table or constant with the CUDA library.
 *
 * Every array is fp64, row-major, host memory owned by the caller.  Inputs in
 * bf16 / fp16 / fp32 are decoded to fp64 exactly by the caller before the call.
 * Routines that take `nthreads` split independent rows over that many POSIX
 * threads; the result does not depend on the thread count.
 *
 * Sources (the veloxquant-mlx A2ATS pages):
 *  - "A2ATS-adapted" algorithm page (deploy-preview), section "For contributors
 *    -- paper fidelity": windowed RoPE (paper Eq. 11-12), query-aware VQ
 *    (Eq. 13-18);
 *  - API page "veloxquant_mlx.quantizers.a2ats module": the five functions
 *    a2ats_query_second_moment, a2ats_cholesky_factor,
 *    a2ats_h_weighted_assignment, a2ats_query_aware_assignment,
 *    a2ats_select_retrieval_set;
 *  - v0.39.0 algorithm page, "How it works" step 4 (window degradation rules).
 */
#ifndef A2ATS_ORACLE_H
#define A2ATS_ORACLE_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* RoPE of one row at position `pos`: pair i (of d/2) is (i, i+d/2) when
 * interleaved == 0, (2i, 2i+1) otherwise; angle pos * base^(-2i/d). */
void orc_rope_row(const double* x, double* y, int64_t d, double pos, double base,
                  int interleaved);

/* Windowed RoPE of `rows` rows.  Row r sits at position p[r] in a sequence whose
 * decode position is t[r]; it is rotated at p[r] when 0 <= t-p < window and at
 * far_offset otherwise (window <= 0: every row is far). */
void orc_windowed_rope(const double* x, double* y, int64_t rows, int64_t d,
                       const int64_t* p, const int64_t* t, int64_t window,
                       double far_offset, double base, int interleaved);

/* H = (1/M) sum_m q_m^T q_m + ridge * I   (paper Eq. 10).  q [M, d] -> h [d, d]. */
void orc_query_second_moment(const double* q, int64_t M, int64_t d, double ridge,
                             double* h);

/* Cholesky-Banachiewicz, H = L L^T (paper Eq. 15).  Returns 0, or j (1-based)
 * when the leading minor of order j is not positive definite. */
int orc_cholesky(const double* h, int64_t d, double* l);

/* argmin_j (x - c_j) H (x - c_j)^T evaluated literally, O(K d^2) per row
 * (paper Eq. 14).  d1/d2: the best two values (d2 = +inf when K = 1). */
void orc_assign_quadratic(const double* x, int64_t n, int64_t d, const double* c,
                          int64_t K, const double* h, int32_t* code, double* d1,
                          double* d2, int nthreads);

/* The same argmin through the Cholesky identity (Eq. 16-18): z = xL, c'_j = c_jL,
 * distance sum_b (z_b - c'_jb)^2.  L == NULL means the identity (plain VQ). */
void orc_assign_cholesky(const double* x, int64_t n, int64_t d, const double* c,
                         int64_t K, const double* l, int32_t* code, double* d1,
                         double* d2, int nthreads);

/* Cosine blend: e_j = |x - c_j|^2, m = max_j e_j,
 * s_j = -beta e_j / m + (1 - beta) cos(q, c_j), code = argmax_j s_j.
 * q_stride == 0: one query shared by all rows; q_stride == d: row r uses
 * q + r*d.  beta == 1 is the plain nearest-centroid rule (s1/s2 then hold
 * the two smallest distances). */
void orc_assign_blend(const double* x, int64_t n, int64_t d, const double* c, int64_t K,
                      const double* q, int64_t q_stride, double beta, int32_t* code,
                      double* s1, double* s2, int nthreads);

/* Retrieval split: s_i = cos(k_i, q) (0 when a norm is 0); the top
 * ceil(fraction * n) rows by (s desc, index asc) form the retrieval set.
 * perm[0:count] = retrieval indices ascending, perm[count:n] = bulk ascending.
 * scores[n] receives s_i; kth receives the smallest retained score (or +inf
 * when count == 0).  Returns count. */
int64_t orc_select_retrieval_set(const double* keys, int64_t n, int64_t d,
                                 const double* q, double fraction, int32_t* perm,
                                 double* scores, double* kth);

/* Code-based attention scores and the top ceil(fraction n) tokens of one
 * (b, h): near rows (0 <= t - j < window) score RoPE(q, t) . RoPE(k_j, j),
 * far rows RoPE(q, far_b) . codebook[codes[j]] (0 for a code outside
 * [0, K)).  keys [n, d] pre-RoPE, codebook [K, d], q [d] pre-RoPE.  perm,
 * scores and kth as orc_select_retrieval_set.  Returns the count. */
int64_t orc_code_attention_topk(const double* keys, int64_t n, int64_t d, int64_t t,
                                const int32_t* codes, const double* codebook, int64_t K,
                                const double* q, int64_t window, double far_b, double base,
                                int interleaved, double fraction, int32_t* perm,
                                double* scores, double* kth);

/* Row j of out [n, d] = codebook [K, d] row codes[j]; zeros for a code
 * outside [0, K). */
void orc_dequantize(const int32_t* codes, int64_t n, const double* codebook, int64_t K,
                    int64_t d, double* out);

/* z [n, d] = x L (row vectors times L [d, d]); c [n, d] with c L = z for a
 * lower-triangular L with nonzero diagonal. */
void orc_cholesky_rows(const double* x, int64_t n, int64_t d, const double* l, double* z);
void orc_cholesky_solve_rows(const double* z, int64_t n, int64_t d, const double* l,
                             double* c);

/* k-means++ seeding with the given uniform draws u [K], then `iters` Lloyd
 * rounds, on points z [n, d]; centroids [K, d], the final codes [n] and
 * objective [iters + 1] (sum of squared distances after each assignment). */
void orc_kmeanspp(const double* z, int64_t n, int64_t d, int64_t K, const double* u,
                  int64_t iters, double* centroids, int32_t* codes, double* objective);

#ifdef __cplusplus
}
#endif
#endif
