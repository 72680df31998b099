/*
 * a2ats.h -- C ABI of the GB300 (sm_103a) library for the data-parallel hot path
 * of A2ATS-style retrieval-based KV-cache compression: windowed RoPE, query
 * second moment and its Cholesky factor, H-weighted and cosine-blend codebook
 * assignment, and the retrieval-set split; and the steps around it:
 * code-based attention scores with top-token retrieval, dequantisation and
 * byte accounting, sub-vector (product) VQ of keys and values, and codebook
 * calibration by k-means++ in Cholesky space.
 *
 * Sources.  The operations follow the veloxquant-mlx documentation of its
 * "A2ATS-adapted" method (after He et al., "A2ATS: Retrieval-Based KV Cache
 * Reduction via Windowed Rotary Position Embedding and Query-Aware Vector
 * Quantization", ACL 2025 Findings):
 *   [API]  "veloxquant_mlx.quantizers.a2ats module" (readthedocs API page):
 *          the five functions a2ats_query_second_moment, a2ats_cholesky_factor,
 *          a2ats_h_weighted_assignment, a2ats_query_aware_assignment,
 *          a2ats_select_retrieval_set;
 *   [ALG]  "A2ATS-adapted" algorithm page (deploy-preview build), section
 *          "For contributors -- paper fidelity": windowed RoPE (Eq. 11-12),
 *          query-aware VQ (Eq. 13-18), per-step re-rotation;
 *   [V039] the v0.39.0 algorithm page, "How it works" (steps 1-5),
 *          configuration and "Byte accounting";
 *   [ABS]  the paper's abstract (attention scores approximated through the
 *          quantised keys to retrieve the top tokens).
 *
 * Conventions shared by every call
 * --------------------------------
 * - Every array argument is DEVICE memory owned by the caller; the library
 *   keeps no pointer after the call returns and allocates no device memory.
 *   Calls that need scratch take a caller-owned `workspace` of at least the
 *   size the matching *_workspace_size() function returns.
 * - Work is enqueued on `stream` (a cudaStream_t; NULL = the legacy default
 *   stream) and runs asynchronously: a call returns after enqueueing.
 * - Keys are laid out [B, H, Ncap, d] row-major: B sequences, H heads,
 *   Ncap cached rows of width d per (sequence, head).  Sequence b holds
 *   len[b] valid rows (len: device int32 [B]; NULL means every row is
 *   valid).  Row j of sequence b is at position j; its decode position is
 *   t = len[b] - 1.  Rows j >= len[b] are neither read nor written.
 * - Codebooks are [H, K, d] in the same dtype as the keys, shared by the
 *   batch.  H and L matrices are [H, d, d] fp32 row-major.
 * - Pointers to key, query, codebook and output arrays must be 16-byte
 *   aligned; d must be a multiple of 8 with 8 <= d <= 256.
 * - Return value: A2ATS_OK, or a negative a2ats_status found on the host
 *   before anything is enqueued (bad argument, shape, dtype, alignment,
 *   workspace), or A2ATS_ERR_CUDA when a launch fails
 *   (a2ats_last_error() then gives CUDA's message).
 * - Results are deterministic: the same inputs give the same bits.
 */
#ifndef A2ATS_H
#define A2ATS_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    A2ATS_OK = 0,
    A2ATS_ERR_INVALID_ARG = -1, /* a parameter out of its range, or a NULL array */
    A2ATS_ERR_SHAPE = -2,       /* sizes the kernels do not support */
    A2ATS_ERR_DTYPE = -3,       /* dtype code not in a2ats_dtype */
    A2ATS_ERR_ALIGN = -4,       /* an array not 16-byte aligned */
    A2ATS_ERR_CUDA = -5,        /* a kernel launch failed */
    A2ATS_ERR_WORKSPACE = -6,   /* workspace NULL or smaller than required */
    A2ATS_ERR_CAPACITY = -7     /* shape beyond a fixed library-owned scratch array */
} a2ats_status;

typedef enum { A2ATS_F32 = 0, A2ATS_BF16 = 1, A2ATS_F16 = 2 } a2ats_dtype;

/* Which rows an assignment call visits (routing of [V039] step 2). */
typedef enum {
    A2ATS_ROWS_ALL = 0,       /* rows 0 .. len-1 */
    A2ATS_ROWS_RETRIEVAL = 1, /* rows perm[0 .. count-1] of a retrieval split */
    A2ATS_ROWS_BULK = 2,      /* rows perm[count .. len-1] of a retrieval split */
    A2ATS_ROWS_LAST = 3       /* the decode row t = len-1 only (the key just appended) */
} a2ats_rows;

/* Windowed RoPE ([ALG] Eq. 11-12; [V039] step 4).  Row p with decode
 * position t is rotated at its own position p when 0 <= t - p < window, and
 * at the one shared position far_offset otherwise.  far_offset = 0 leaves far
 * keys unrotated, which is the paper's Eq. 12.  window <= 0: every row is far;
 * window >= len: every row is exact.  Pair i of d/2 is (i, i + d/2) when
 * interleaved = 0 and (2i, 2i+1) otherwise; its angle is
 * position * rope_base^(-2i/d).  Positions must stay below 2^24. */
typedef struct {
    int32_t window;
    int32_t far_offset;
    double rope_base;
    int32_t interleaved;
} a2ats_rope_params;

/* --------------------------------------------------------------------------
 * a2ats_windowed_rope -- [ALG] "Windowed RoPE (Eq. 11-12)" and "Per-step
 * re-rotation": re-rotate every cached key against the current decode
 * position.
 *   k_in   [B, H, Ncap, d] in in_dtype (pre-RoPE keys)
 *   k_out  [B, H, Ncap, d] in out_dtype; may alias k_in when the dtypes match
 * Arithmetic is fp32; the fp32 output is within 1e-6 relative of the exact
 * rotation, a bf16/fp16 output is the fp32 result rounded to nearest even.
 * ------------------------------------------------------------------------ */
int a2ats_windowed_rope(const void* k_in, int32_t in_dtype, void* k_out, int32_t out_dtype,
                        int64_t B, int64_t H, int64_t Ncap, int64_t d, const int32_t* len,
                        const a2ats_rope_params* rope, void* stream);

/* --------------------------------------------------------------------------
 * a2ats_append_rows -- the cache step of a decode ([V039] "How it works": every
 * call stores the incoming keys, pre-RoPE, and the whole cache is re-rotated
 * against the new position): row len[b] of every (b, h) receives
 * rows[b, h, :], then len[b] += 1.
 *   cache [B, H, Ncap, d] in dtype;  rows [B, H, d] in dtype;
 *   len   [B] int32 device, read and updated in place (required).
 * A sequence already holding Ncap rows is left unchanged (len stays Ncap).
 * ------------------------------------------------------------------------ */
int a2ats_append_rows(void* cache, int32_t dtype, int64_t B, int64_t H, int64_t Ncap, int64_t d,
                      int32_t* len, const void* rows, void* stream);

/* --------------------------------------------------------------------------
 * a2ats_query_second_moment -- [API] a2ats_query_second_moment (paper Eq. 10):
 *   H_h = (1/M) Q_h^T Q_h + ridge * I, not mean-centred.
 *   queries [H, M, d] in dtype;  h_out [H, d, d] fp32, exactly symmetric.
 * ridge >= 0 (the page's default is 1e-4).  M >= 1.
 * ------------------------------------------------------------------------ */
size_t a2ats_query_second_moment_workspace_size(int64_t H, int64_t M, int64_t d);
int a2ats_query_second_moment(const void* queries, int32_t dtype, int64_t H, int64_t M,
                              int64_t d, double ridge, float* h_out, void* workspace,
                              size_t workspace_bytes, void* stream);

/* --------------------------------------------------------------------------
 * a2ats_cholesky_factor -- [API] a2ats_cholesky_factor (paper Eq. 15):
 * lower-triangular L with H = L L^T, per head.
 *   h [H, d, d] fp32 (symmetric positive definite);  l_out [H, d, d] fp32
 *   (zeros above the diagonal);  info [H] int32: 0, or j >= 1 when the
 *   leading minor of order j of that head is not positive definite (L of that
 *   head is then unspecified).  A non-PD input is reported, never trapped.
 * ------------------------------------------------------------------------ */
int a2ats_cholesky_factor(const float* h, int64_t H, int64_t d, float* l_out, int32_t* info,
                          void* stream);

/* --------------------------------------------------------------------------
 * a2ats_h_weighted_assign -- [API] a2ats_h_weighted_assignment (paper
 * Eq. 14 through the Eq. 15-18 Cholesky identity):
 *   code = argmin_j (k~ - c_j) H (k~ - c_j)^T = argmin_j |k~ L - c_j L|^2,
 * ties to the lowest j.
 *   x        [B, H, Ncap, d] in dtype: k~ itself, or pre-RoPE keys when
 *            fused_rope != NULL (windowed RoPE is then applied on the fly)
 *   codebook [H, K, d] in dtype (untransformed centroids)
 *   L        [H, d, d] fp32 Cholesky factor; only its lower triangle (with
 *            the diagonal) is read, entries above the diagonal are ignored;
 *            NULL = identity, which is plain nearest-centroid VQ ([V039]
 *            step 2, bulk rows)
 *   rows     which rows to assign; RETRIEVAL / BULK read perm [B, H, Ncap]
 *            and count [B, H] as written by a2ats_select_retrieval_set;
 *            LAST assigns the decode row t = len-1 of each (b, h)
 *   codes    [B, H, Ncap] int32; only the visited rows are written
 * Exactness: the code equals the exact argmin except possibly on rows whose
 * two best distances differ by less than 1e-5 of the second best.
 * ------------------------------------------------------------------------ */
size_t a2ats_h_weighted_assign_workspace_size(int64_t B, int64_t H, int64_t Ncap, int64_t d,
                                              int64_t K);
int a2ats_h_weighted_assign(const void* x, int32_t dtype, int64_t B, int64_t H, int64_t Ncap,
                            int64_t d, const int32_t* len, const void* codebook, int64_t K,
                            const float* L, const a2ats_rope_params* fused_rope,
                            int32_t rows, const int32_t* perm, const int32_t* count,
                            int32_t* codes, void* workspace, size_t workspace_bytes,
                            void* stream);

/* --------------------------------------------------------------------------
 * a2ats_h_weighted_assign_reuse -- a2ats_h_weighted_assign without the
 * codebook side (no counterpart on the pages: the codebook and L are
 * per-layer calibration artifacts, [ALG] "Optional: query-aware
 * calibration", and the Eq. 16-18 route assigns against pre-transformed
 * centroids, so a decode loop needs their transform once per layer).
 * It takes the lower-triangle copy of L, c L, |c L|^2 / 2, c L L^T and their
 * 16-bit planes and tables from the workspace, where the last
 * a2ats_h_weighted_assign call on it left them.  The caller guarantees that
 * that call had the same codebook and L contents, dtype, B, H, Ncap, d, K,
 * fused_rope and rows, and that nothing but a2ats_h_weighted_assign_reuse
 * calls has used the workspace since; otherwise the codes are unspecified
 * (no error is detected).  Arguments, results and errors are otherwise those
 * of a2ats_h_weighted_assign (codebook and L are only checked, not read).
 * ------------------------------------------------------------------------ */
int a2ats_h_weighted_assign_reuse(const void* x, int32_t dtype, int64_t B, int64_t H,
                                  int64_t Ncap, int64_t d, const int32_t* len,
                                  const void* codebook, int64_t K, const float* L,
                                  const a2ats_rope_params* fused_rope, int32_t rows,
                                  const int32_t* perm, const int32_t* count, int32_t* codes,
                                  void* workspace, size_t workspace_bytes, void* stream);

/* --------------------------------------------------------------------------
 * a2ats_query_aware_assign -- [API] a2ats_query_aware_assignment (cosine
 * blend):  e_j = |x - c_j|^2,  m = max_j e_j,
 *   score_j = -beta * e_j / m + (1 - beta) * cos(query, c_j),
 *   code = argmax_j score_j (ties to the lowest j);  e_j / m is 0 when m = 0
 *   and a cosine with a zero-norm vector is 0.  beta = 1 is exactly plain
 *   nearest-centroid VQ (argmin_j e_j).
 *   query  [B, H, d] in dtype, one query per (sequence, head); NULL = the
 *          proxy query of [V039] honesty point 1: the key at the decode
 *          position t after windowed RoPE (the same proxy the retrieval split
 *          uses; with fused_rope == NULL, x at t as given).
 *   beta in [0, 1]; other arguments as a2ats_h_weighted_assign.
 * Exactness: the exact argmax except possibly on rows whose two best scores
 * differ by less than 1e-5.
 * ------------------------------------------------------------------------ */
size_t a2ats_query_aware_assign_workspace_size(int64_t B, int64_t H, int64_t Ncap, int64_t d,
                                               int64_t K);
int a2ats_query_aware_assign(const void* x, int32_t dtype, int64_t B, int64_t H, int64_t Ncap,
                             int64_t d, const int32_t* len, const void* codebook, int64_t K,
                             const void* query, double beta,
                             const a2ats_rope_params* fused_rope, int32_t rows,
                             const int32_t* perm, const int32_t* count, int32_t* codes,
                             void* workspace, size_t workspace_bytes, void* stream);

/* --------------------------------------------------------------------------
 * a2ats_query_aware_assign_reuse -- a2ats_query_aware_assign without the
 * codebook side (no counterpart on the pages: the codebook is a per-layer
 * artifact, and a decode loop that assigns its new keys at every step needs
 * the decoded centroids and their norms once).  It takes the decoded fp32
 * centroids, |c|^2 / 2 and |c| (for beta = 1 also the contraction's planes
 * and tables) from the workspace, where the last a2ats_query_aware_assign
 * call on it left them.  The caller guarantees that that call had the same
 * codebook contents, dtype, B, H, Ncap, d, K, beta (1 or not), fused_rope
 * and rows, and that nothing but a2ats_query_aware_assign_reuse calls has
 * used the workspace since; otherwise the codes are unspecified (no error is
 * detected).  Arguments, results and errors are otherwise those of
 * a2ats_query_aware_assign (codebook is only checked, not read).
 * ------------------------------------------------------------------------ */
int a2ats_query_aware_assign_reuse(const void* x, int32_t dtype, int64_t B, int64_t H,
                                   int64_t Ncap, int64_t d, const int32_t* len,
                                   const void* codebook, int64_t K, const void* query,
                                   double beta, const a2ats_rope_params* fused_rope, int32_t rows,
                                   const int32_t* perm, const int32_t* count, int32_t* codes,
                                   void* workspace, size_t workspace_bytes, void* stream);

/* --------------------------------------------------------------------------
 * a2ats_select_retrieval_set -- [API] a2ats_select_retrieval_set: per
 * (sequence, head), score s_i = cos(k~_i, query) (0 when a norm is 0) and
 * keep the top n_r = ceil(fraction * len) rows, ordered by (score desc,
 * index asc), with fraction * len evaluated in IEEE double.
 *   keys   [B, H, Ncap, d] in dtype: k~, or pre-RoPE keys with fused_rope
 *   query  [B, H, d] in dtype; NULL = the proxy query: the key at the decode
 *          position t as it stands after windowed RoPE
 *   fraction in [0, 1] (the page's default is 0.2)
 *   perm   [B, H, Ncap] int32: perm[0:n_r] the retrieval rows ascending,
 *          perm[n_r:len] the bulk rows ascending (disjoint, covering 0..len-1)
 *   count  [B, H] int32: n_r
 * Exactness: the exact set except possibly for rows whose score is within
 * 1e-5 of the n_r-th largest score; the set size is always exactly n_r.
 * ------------------------------------------------------------------------ */
size_t a2ats_select_retrieval_set_workspace_size(int64_t B, int64_t H, int64_t Ncap, int64_t d);
int a2ats_select_retrieval_set(const void* keys, int32_t dtype, int64_t B, int64_t H,
                               int64_t Ncap, int64_t d, const int32_t* len, const void* query,
                               double fraction, const a2ats_rope_params* fused_rope,
                               int32_t* perm, int32_t* count, void* workspace,
                               size_t workspace_bytes, void* stream);

/* --------------------------------------------------------------------------
 * a2ats_select_retrieval_set_rotated -- a2ats_windowed_rope and
 * a2ats_select_retrieval_set (fused_rope = rope) in one pass over the keys
 * (no counterpart on the pages: it fuses two of their steps, the per-step
 * re-rotation of [ALG] "Per-step re-rotation" and the split of [API]
 * a2ats_select_retrieval_set, so the pre-RoPE cache is read once).
 *   keys   [B, H, Ncap, d] pre-RoPE, in dtype
 *   rope   required; k_out [B, H, Ncap, d] in out_dtype receives exactly what
 *          a2ats_windowed_rope(keys, ..., rope) writes (rows j < len[b]);
 *          k_out must not be keys
 *   query, fraction, perm, count, workspace: as a2ats_select_retrieval_set,
 *          and perm / count are exactly what it writes with fused_rope = rope
 * Errors: those of both calls; the workspace size is
 * a2ats_select_retrieval_set_workspace_size.
 * ------------------------------------------------------------------------ */
int a2ats_select_retrieval_set_rotated(const void* keys, int32_t dtype, int64_t B, int64_t H,
                                       int64_t Ncap, int64_t d, const int32_t* len,
                                       const void* query, double fraction,
                                       const a2ats_rope_params* rope, void* k_out,
                                       int32_t out_dtype, int32_t* perm, int32_t* count,
                                       void* workspace, size_t workspace_bytes, void* stream);

/* --------------------------------------------------------------------------
 * a2ats_rope_split_plain_assign -- a2ats_select_retrieval_set_rotated
 * (out_dtype = dtype) and plain VQ over every row,
 * a2ats_h_weighted_assign(keys, codebook, L = NULL, fused_rope = rope,
 * rows = A2ATS_ROWS_ALL), in one call (no counterpart on the pages: it joins
 * the per-step re-rotation of [ALG] "Per-step re-rotation", the split of
 * [API] a2ats_select_retrieval_set and the bulk rule of [V039] step 2, the
 * nearest centroid, so that with far_offset = 0 one pass over the stored
 * keys outside the RoPE window copies them to k_out, scores them and
 * assigns them).
 *   keys, dtype, B, H, Ncap, d, len, query, fraction, rope: as
 *          a2ats_select_retrieval_set_rotated (rope required)
 *   codebook [H, K, d] in dtype; K in [1, 2^24]
 *   k_out  [B, H, Ncap, d] in dtype: the windowed-RoPE keys (rows j < len[b],
 *          exactly what a2ats_windowed_rope writes); must not be keys
 *   perm, count: the split, as a2ats_select_retrieval_set writes it
 *   codes  [B, H, Ncap] int32: the nearest centroid of every row j < len[b]
 *          (the exactness of a2ats_h_weighted_assign)
 *   reuse  nonzero: the codebook side (decoded centroids, norms, planes,
 *          tables) is taken from the workspace as the previous call of this
 *          function on it, with the same codebook, shapes and rope, left it
 *   split_done  a cudaEvent_t, or NULL: recorded on the stream as soon as
 *          k_out, perm and count are complete (before the codes are), so a
 *          second stream can start on the split while this call finishes
 *   split_stream  a cudaStream_t other than stream, or NULL: with split_done
 *          given, the split itself runs there (split_done is recorded on
 *          stream once the scores are written, split_stream waits for it,
 *          and split_done is recorded again on split_stream after the
 *          split), so the RoPE-window rows' assignment on stream runs beside
 *          it; stream waits for split_done before the call returns, so every
 *          output is complete in stream order as without it.  INVALID_ARG
 *          when given without split_done or equal to stream
 *   workspace  a2ats_rope_split_plain_assign_workspace_size(B, H, Ncap, d, K)
 *          bytes of device memory, owned by the caller
 * The scores of this call may differ from those of
 * a2ats_select_retrieval_set in the last bits (another order of fp32
 * additions), so the split is exact except on the near-ties that call
 * exempts too.
 * Errors: those of both calls; WORKSPACE when workspace is NULL or short.
 * ------------------------------------------------------------------------ */
size_t a2ats_rope_split_plain_assign_workspace_size(int64_t B, int64_t H, int64_t Ncap,
                                                    int64_t d, int64_t K);
int a2ats_rope_split_plain_assign(const void* keys, int32_t dtype, int64_t B, int64_t H,
                                  int64_t Ncap, int64_t d, const int32_t* len, const void* query,
                                  double fraction, const a2ats_rope_params* rope,
                                  const void* codebook, int64_t K, void* k_out, int32_t* perm,
                                  int32_t* count, int32_t* codes, int32_t reuse,
                                  void* split_done, void* split_stream, void* workspace,
                                  size_t workspace_bytes, void* stream);

/* --------------------------------------------------------------------------
 * a2ats_code_attention_topk -- the attention score of the decode query with
 * every cached key, far keys through their codes, and the top tokens by it:
 * deploy-preview "A2ATS-adapted" page, paper-fidelity section, "Windowed
 * RoPE (Eq. 11-12)" (far keys unrotated, the far relative position b on the
 * query, u_ij = q_i R_b k_j^T, the page's a2ats_apply_far_query_rope half;
 * keys inside the window with exact RoPE), and the paper's abstract (top-K
 * tokens retrieved by the approximate attention score).  The pages give no
 * function for it.  With t = len[b] - 1:
 *   near row j (0 <= t - j < window):  u_j = RoPE(q, t) . RoPE(keys_j, j)
 *   far row j:                         u_j = RoPE(q, far_b) . codebook[codes_j]
 * (0 for a code outside [0, K)).
 *   keys     [B, H, Ncap, d] pre-RoPE, in dtype (only the window rows are read)
 *   codes    [B, H, Ncap] int32 (e.g. from the assignment of k~)
 *   codebook [H, K, d] in dtype; K in [1, 2^24]
 *   query    [B, H, d] in dtype, the decode query before RoPE
 *   rope     required: window and RoPE base / pairing (far_offset unused)
 *   far_b    the far relative position, |far_b| < 2^24 (the page's default 2048)
 *   fraction in [0, 1]: the top ceil(fraction len) rows are retrieved
 *   scores   [B, H, Ncap] fp32: u_j for rows j < len[b]
 *   perm, count: as a2ats_select_retrieval_set writes them, ranked by u
 *   workspace  a2ats_code_attention_topk_workspace_size(B, H, Ncap, d, K)
 *            bytes of device memory, owned by the caller
 * Scores are fp32 (table entries and near dots summed in fp32); the set is
 * exact except possibly for rows whose score is within 1e-5 of the largest
 * score's magnitude from the threshold.
 * Errors: SHAPE, DTYPE, ALIGN as the other calls; INVALID_ARG for a NULL
 * rope, fraction outside [0, 1], |far_b| >= 2^24 or a NULL array when
 * Ncap > 0; WORKSPACE when workspace is NULL or short.
 * ------------------------------------------------------------------------ */
size_t a2ats_code_attention_topk_workspace_size(int64_t B, int64_t H, int64_t Ncap, int64_t d,
                                                int64_t K);
int a2ats_code_attention_topk(const void* keys, int32_t dtype, int64_t B, int64_t H, int64_t Ncap,
                              int64_t d, const int32_t* len, const int32_t* codes,
                              const void* codebook, int64_t K, const void* query,
                              const a2ats_rope_params* rope, int32_t far_b, double fraction,
                              float* scores, int32_t* perm, int32_t* count, void* workspace,
                              size_t workspace_bytes, void* stream);

/* --------------------------------------------------------------------------
 * a2ats_dequantize -- v0.39.0 page, "How it works", step 3: each key is
 * reconstructed from its assigned centroid.  out[b, h, j] = codebook[h,
 * codes[b, h, j]] for rows j < len[b] (zeros for a code outside [0, K));
 * rows past len[b] are not written.
 *   codes    [B, H, Ncap] int32 device
 *   codebook [H, K, d] device, in dtype; K in [1, 2^24]
 *   len      [B] int32 device, or NULL for Ncap everywhere
 *   out      [B, H, Ncap, d] device, in dtype; must not be the codebook
 * Errors: DTYPE, SHAPE (d a multiple of 8 in [8, 256]), ALIGN, INVALID_ARG
 * for a NULL array when B*H*Ncap > 0 or out == codebook.
 * ------------------------------------------------------------------------ */
int a2ats_dequantize(const int32_t* codes, const void* codebook, int32_t dtype, int64_t B,
                     int64_t H, int64_t Ncap, int64_t d, int64_t K, const int32_t* len, void* out,
                     void* stream);

/* --------------------------------------------------------------------------
 * a2ats_byte_accounting -- v0.39.0 page, "Byte accounting" and "What you
 * get with the defaults": the storage of `tokens` keys and `tokens` values
 * of width d as codes of codebook_bits bits, one per sub_dim numbers (both
 * follow the cache's one a2ats_sub_dim / a2ats_codebook_bits; the
 * full-width VQ here has sub_dim = d and codebook_bits = log2 K).  Host
 * only; no device memory.
 *   compressed_key_bytes = compressed_value_bytes = tokens (d / sub_dim)
 *                          codebook_bits / 8
 *   fp16_key_bytes       = fp16_value_bytes = tokens d 2
 *   compression_ratio    = (fp16 keys + values) / (compressed keys + values)
 *                        = 16 sub_dim / codebook_bits (also for tokens = 0:
 *                          the settings alone decide it)
 *   codebook_bytes       = 2^codebook_bits sub_dim 2: one table of fp16
 *                          entries, the page's "Table size"
 *   assigned_avg_bits    = codebook_bits / sub_dim
 * Errors: INVALID_ARG for a NULL out, sub_dim < 1 or codebook_bits outside
 * [1, 24]; SHAPE for tokens < 0, d < 1 or d not a multiple of sub_dim.
 * ------------------------------------------------------------------------ */
typedef struct {
    double compressed_key_bytes;
    double compressed_value_bytes;
    double fp16_key_bytes;
    double fp16_value_bytes;
    double compression_ratio;
    double codebook_bytes;
    double assigned_avg_bits;
} a2ats_cache_bytes;
int a2ats_byte_accounting(int64_t tokens, int64_t d, int64_t sub_dim, int32_t codebook_bits,
                          a2ats_cache_bytes* out);

/* --------------------------------------------------------------------------
 * a2ats_cholesky_rows -- the change of variables of [API]
 * a2ats_cholesky_factor: z = x L for every row, so that the H-weighted
 * distance (x - c) H (x - c)^T with H = L L^T is |z_x - z_c|^2 and
 * ordinary k-means on the z rows trains an H-weighted codebook.
 *   x  [H, n, d] device, in dtype (e.g. calibration keys of one layer, head
 *      by head)
 *   L  [H, d, d] fp32 device; only the lower triangle (with the diagonal) is
 *      read
 *   z  [H, n, d] fp32 device output; must not be x
 * Each element is a compensated fp32 dot product (twice-fp32 accumulation)
 * rounded once.  n < 2^24; d a multiple of 8 in [8, 256].
 * Errors: DTYPE, SHAPE, ALIGN, INVALID_ARG for a NULL array when H*n > 0 or
 * z == x, WORKSPACE.
 * ------------------------------------------------------------------------ */
size_t a2ats_cholesky_rows_workspace_size(int64_t H, int64_t n, int64_t d);
int a2ats_cholesky_rows(const void* x, int32_t dtype, int64_t H, int64_t n, int64_t d,
                        const float* L, float* z, void* workspace, size_t workspace_bytes,
                        void* stream);

/* --------------------------------------------------------------------------
 * a2ats_cholesky_solve_rows -- back from z space ([API]
 * a2ats_cholesky_factor): c with c L = zc for every row, so that centroids
 * found by k-means on z = x L become a key-space codebook for
 * a2ats_h_weighted_assign with the same L.
 *   zc [H, rows, d] fp32 device; c [H, rows, d] fp32 device output (may be
 *   zc itself)
 *   L  [H, d, d] fp32 device, lower triangular with a nonzero diagonal (a
 *      Cholesky factor); only the lower triangle is read
 * Back substitution from the last column in fp64, rounded to fp32.
 * rows <= 2^24, H*rows <= 2^30; d a multiple of 8 in [8, 256].
 * Errors: SHAPE, ALIGN, INVALID_ARG for a NULL array when H*rows > 0.
 * ------------------------------------------------------------------------ */
int a2ats_cholesky_solve_rows(const float* zc, int64_t H, int64_t rows, int64_t d, const float* L,
                              float* c, void* stream);

/* --------------------------------------------------------------------------
 * a2ats_kmeanspp -- codebook calibration by k-means++ in z space ([API]
 * a2ats_cholesky_factor: k-means++ on z = k L builds the H-weighted
 * codebook), head by head.
 *   Seeding: centre 0 is row floor(u[h, 0] n); centre k is the first row
 *   whose running sum of D^2 (the squared distance to the nearest centre
 *   chosen so far) exceeds u[h, k] times the sum of D^2 over all rows, or
 *   row floor(u[h, k] n) when every D^2 is 0 (row indices clamped to
 *   [0, n)).  D^2 and its running sums are fp64.
 *   Then `iters` Lloyd rounds: each row takes its nearest centroid (ties to
 *   the lower index; the exact assignment of a2ats_h_weighted_assign with
 *   L = NULL), each centroid moves to the fp64 mean of its rows (rounded to
 *   fp32) and a centroid without rows stays; a last assignment follows.
 *   z          [H, n, d] fp32 device (e.g. from a2ats_cholesky_rows); 1 <= n
 *              < 2^24; d a multiple of 8 in [8, 256]
 *   u          [H, K] fp64 device: the uniform draws, in [0, 1)
 *   iters      Lloyd rounds, in [0, 2^20]
 *   centroids  [H, K, d] fp32 device output: the z-space codebook after the
 *              last mean step (the seeds when iters = 0); K in [1, 2^24]
 *   codes      [H, n] int32 device output: the last assignment
 *   objective  [H, iters + 1] fp64 device output: the sum over rows of the
 *              squared distance to the assigned centroid, after each
 *              assignment (entry iters belongs to the returned codes)
 * z, centroids and codes must not overlap.  The rows must be finite with
 * squares that do not overflow fp32.
 * Errors: SHAPE (also n = 0 with H > 0), INVALID_ARG for a NULL array,
 * iters out of range or overlapping arrays, ALIGN (z, centroids, codes
 * 16-byte; u, objective 8-byte), WORKSPACE.
 * ------------------------------------------------------------------------ */
size_t a2ats_kmeanspp_workspace_size(int64_t H, int64_t n, int64_t d, int64_t K);
int a2ats_kmeanspp(const float* z, int64_t H, int64_t n, int64_t d, int64_t K, const double* u,
                   int32_t iters, float* centroids, int32_t* codes, double* objective,
                   void* workspace, size_t workspace_bytes, void* stream);

/* --------------------------------------------------------------------------
 * a2ats_subvector_assign -- sub-vector (product) VQ, the v0.39.0 page's
 * configuration (a2ats_sub_dim, a2ats_codebook_bits) with "How it works"
 * steps 2 and 5: every token row j < len[b] of width d is G = d / sub_dim
 * sub-vectors x_g = x[j, g sub_dim .. (g + 1) sub_dim), each coded by
 *   code[b, h, j, g] = argmin_k |x_g L - c_k L|^2   (H-weighted rule, [API]
 *                      a2ats_h_weighted_assignment, Eq. 14-18)
 * on the retrieval tokens (perm[b, h, :count[b, h]]) when L is given, and by
 *   code[b, h, j, g] = argmin_k |x_g - c_k|^2       (plain VQ)
 * on every other token; ties go to the lowest k.
 *   x        [B, H, Ncap, d] device, in dtype (for keys: k~ after windowed
 *            RoPE, which pairs elements of different sub-vectors and so runs
 *            on the whole row first; for values: the values)
 *   codebook [H, K, sub_dim] device, in dtype: one table per head
 *   L        [H, sub_dim, sub_dim] fp32 device (lower triangle read), or
 *            NULL: plain VQ for every token
 *   perm, count  the token split as a2ats_select_retrieval_set writes it, or
 *            both NULL: with L given, every token takes the H-weighted rule
 *   codes    [B, H, Ncap, G] int32 device output; rows past len[b] are not
 *            written
 * sub_dim is 8 or 16 and divides d; K * sub_dim <= 8192.  The distance of a
 * sub_dim-wide difference is a direct fp32 sum (relative error below
 * (sub_dim + 2) 2^-24), so a code can differ from the exact argmin only
 * where the two best distances are that close.
 * Errors: DTYPE, SHAPE, INVALID_ARG for a NULL array when B*H*Ncap > 0 or
 * only one of perm / count, ALIGN, WORKSPACE.
 * ------------------------------------------------------------------------ */
size_t a2ats_subvector_assign_workspace_size(int64_t B, int64_t H, int64_t Ncap, int64_t d,
                                             int64_t sub_dim, int64_t K);
int a2ats_subvector_assign(const void* x, int32_t dtype, int64_t B, int64_t H, int64_t Ncap,
                           int64_t d, const int32_t* len, int64_t sub_dim, const void* codebook,
                           int64_t K, const float* L, const int32_t* perm, const int32_t* count,
                           int32_t* codes, void* workspace, size_t workspace_bytes,
                           void* stream);

/* --------------------------------------------------------------------------
 * a2ats_subvector_query_aware_assign -- sub-vector VQ with the cosine blend
 * of [API] a2ats_query_aware_assignment on the retrieval tokens: the rule
 * the v0.39.0 page's wrapper takes when no calibrated H (a2ats_query_h) is
 * given, with a2ats_beta.  For sub-vector g of a retrieval token j < len[b]
 * (perm[b, h, :count[b, h]], or every token when perm and count are NULL):
 *   e_k = |x_g - c_k|^2,  m = max_k e_k,
 *   score_k = -beta e_k / m + (1 - beta) cos(q_g, c_k),
 *   code = argmax_k score_k (ties to the lowest k),
 * with q_g the query's slice g (elements g sub_dim .. (g + 1) sub_dim);
 * e_k / m is 0 when m = 0 and a cosine with a zero-norm vector is 0.  Every
 * other token, and every token when beta = 1, takes plain VQ (argmin_k e_k).
 *   query  [B, H, d] device in dtype, one query per (sequence, head); NULL =
 *          the row of x at t = len[b] - 1 (for keys: the proxy query k~_t)
 *   beta in [0, 1]; other arguments as a2ats_subvector_assign.
 * A code can differ from the exact argmax only where the two best scores
 * are within about 10^-5 of each other (fp32 distances and cosines).
 * Errors: as a2ats_subvector_assign, and INVALID_ARG for beta outside
 * [0, 1].
 * ------------------------------------------------------------------------ */
size_t a2ats_subvector_query_aware_assign_workspace_size(int64_t B, int64_t H, int64_t Ncap,
                                                         int64_t d, int64_t sub_dim, int64_t K);
int a2ats_subvector_query_aware_assign(const void* x, int32_t dtype, int64_t B, int64_t H,
                                       int64_t Ncap, int64_t d, const int32_t* len,
                                       int64_t sub_dim, const void* codebook, int64_t K,
                                       const void* query, double beta, const int32_t* perm,
                                       const int32_t* count, int32_t* codes, void* workspace,
                                       size_t workspace_bytes, void* stream);

/* --------------------------------------------------------------------------
 * a2ats_copy_retrieval_rows -- dst[b, h, j] = src[b, h, j] for the retrieval
 * rows j = perm[b, h, i], i < count[b, h], j < len[b] (no counterpart on the
 * pages: it joins the two halves of [V039] step 2's routing when they are
 * computed at the same time, the bulk rule over every row into dst and the
 * retrieval rule into src).
 *   src, dst  [B, H, Ncap] int32 device arrays (e.g. codes)
 *   len       [B] int32 device, or NULL for Ncap everywhere
 *   perm, count as written by a2ats_select_retrieval_set
 * Errors: SHAPE for negative sizes or B*H > 65535; INVALID_ARG for a NULL
 * array when B*H*Ncap > 0.
 * ------------------------------------------------------------------------ */
int a2ats_copy_retrieval_rows(const int32_t* src, int32_t* dst, int64_t B, int64_t H,
                              int64_t Ncap, const int32_t* len, const int32_t* perm,
                              const int32_t* count, void* stream);

/* --------------------------------------------------------------------------
 * a2ats_select_retrieval_set_static -- the same retrieval split as
 * a2ats_select_retrieval_set, for callers that cannot allocate device memory
 * (no counterpart on the pages: this is a packaging variant).  Some callers
 * have every byte of device memory owned by another allocator, or run on
 * paths that must never risk an allocation failure or its latency; they
 * cannot provide a workspace.  This entry point allocates nothing: its
 * scratch is one fixed array compiled into the library, which every GPU that
 * loads the library holds (about 5.3 MB) until the process exits.
 *   Limits: B*H <= 1024 and B*H*Ncap <= 1048576, else A2ATS_ERR_CAPACITY
 *   (before anything is enqueued).  Arguments and results are otherwise those
 *   of a2ats_select_retrieval_set, and the results are identical.
 *   The first call on each device looks up the array's device address with
 *   that device current, and so does the first call after the device's
 *   context was replaced (cudaDeviceReset); make such a call before any
 *   stream capture.  Arguments are validated exactly as
 *   a2ats_select_retrieval_set validates them, and a CUDA failure leaves its
 *   message for a2ats_last_error.
 *   All calls share the one array and it keeps the last call's contents
 *   (every word a call reads is written earlier in the same call): calls
 *   that may overlap on the GPU -- on different streams, or from different
 *   host threads -- race and must be serialised by the caller.
 * ------------------------------------------------------------------------ */
int a2ats_select_retrieval_set_static(const void* keys, int32_t dtype, int64_t B, int64_t H,
                                      int64_t Ncap, int64_t d, const int32_t* len,
                                      const void* query, double fraction,
                                      const a2ats_rope_params* fused_rope, int32_t* perm,
                                      int32_t* count, void* stream);

/* Number of kernels this library has enqueued since it was loaded, over all
 * host threads (diagnostics: lets a caller count the launches of a region). */
uint64_t a2ats_kernel_launches(void);

/* Diagnostics for benchmarks.  With timing on, every assignment call records
 * a pair of CUDA events on its stream around each tensor-core contraction
 * over keys in stored order (the pass that does almost all of the work).
 * a2ats_timed_kernels_ms() waits for the recorded events, returns the summed
 * milliseconds, writes the number of timed launches to *launches (if not
 * NULL) and clears the record.  Timing is off after loading; not for
 * concurrent use from several host threads. */
int a2ats_set_kernel_timing(int32_t enable);
double a2ats_timed_kernels_ms(int64_t* launches);

/* Human-readable name of a status code (static storage). */
const char* a2ats_status_string(int32_t status);

/* CUDA's message for the last A2ATS_ERR_CUDA returned on this host thread
 * (static per-thread storage; "" when there was none). */
const char* a2ats_last_error(void);

#ifdef __cplusplus
}
#endif
#endif /* A2ATS_H */
