// kernels.cuh -- host-side launch functions of the A2ATS kernels.  Each .cu
// file implements the launches for its kernels; api.cu validates arguments,
// lays out the workspace and calls these.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"

namespace a2ats {

// Count of kernels enqueued by this library (see a2ats_kernel_launches).
void note_launches(int n);

// Event pairs around the stored-order contraction (see a2ats_set_kernel_timing).
bool kernel_timing_on();
void timing_begin(cudaStream_t st);
void timing_end(cudaStream_t st);

struct Shape {
    int64_t B, H, Ncap, d;
};

// rope_split.cu ----------------------------------------------------------
cudaError_t launch_windowed_rope(const void* k_in, int in_dt, void* k_out, int out_dt,
                                 const Shape& s, const int32_t* len, const RopeArgs& ra,
                                 cudaStream_t st);

// q_out [B*H, d] fp32 and qnorm [B*H]: the given query (decoded), or the key
// at the decode position after windowed RoPE when query == nullptr.
cudaError_t launch_prepare_query(const void* keys, const void* query, int dt, const Shape& s,
                                 const int32_t* len, const RopeArgs& ra, float* q_out,
                                 float* qnorm, cudaStream_t st);

// scores [B*H*Ncap] fp32 cosine of every valid row with its (b, h) query.
// kout != null: the windowed-RoPE rows are stored too, in out_dt (the same
// values launch_windowed_rope writes); cudaErrorNotSupported when the width
// has no fused form (the caller then runs launch_windowed_rope).
cudaError_t launch_cosine_scores(const void* keys, int dt, const Shape& s, const int32_t* len,
                                 const RopeArgs& ra, const float* q, const float* qnorm,
                                 float* scores, cudaStream_t st, void* kout = nullptr,
                                 int out_dt = -1);

// The query of each (b, h) into q / qnorm (exactly what launch_prepare_query
// writes) and the RoPE window only (rows j in [len - W, len) of each
// (b, h)): kout <- the rotated rows in the keys' dtype, scores <- their
// cosine with the query.  cudaErrorNotSupported when d % 16 != 0.
cudaError_t launch_window_scores(const void* keys, const void* query, int dt, const Shape& s,
                                 const int32_t* len, const RopeArgs& ra, float* q, float* qnorm,
                                 float* scores, void* kout, cudaStream_t st);

// code_attention.cu ------------------------------------------------------
// Code-based attention scores of every row j < len[b]: near rows (t - j <
// window, t = len - 1) RoPE(q, t) . RoPE(k_j, j), far rows
// RoPE(q, far_b) . c[code_j] through the per-(b, h) table lut [B*H, K];
// q_near [B*H, d] receives RoPE(q, t).
cudaError_t launch_code_attention(const void* keys, int dt, const Shape& s, const int32_t* len,
                                  const int32_t* codes, const void* codebook, int64_t K,
                                  const void* query, const RopeArgs& ra, int32_t far_b,
                                  float* q_near, float* lut, float* scores, cudaStream_t st);

// out [B, H, Ncap, d] (the codebook's dtype) <- codebook[h, codes[b, h, j]]
// for rows j < len[b]; zeros for a code outside [0, K).
cudaError_t launch_dequantize(const int32_t* codes, const void* codebook, int dt, const Shape& s,
                              int64_t K, const int32_t* len, void* out, cudaStream_t st);

// row len[b] of each (b, h) <- rows[b, h]; then len[b] += 1 (capped at Ncap)
cudaError_t launch_append_rows(void* cache, int dt, const Shape& s, int32_t* len, const void* rows,
                               cudaStream_t st);

// dst <- src on the retrieval rows of the split (perm[:count], within len).
cudaError_t launch_copy_retrieval_rows(const int32_t* src, int32_t* dst, const Shape& s,
                                       const int32_t* len, const int32_t* perm,
                                       const int32_t* count, cudaStream_t st);
cudaError_t launch_select(const float* scores, const Shape& s, const int32_t* len,
                          double fraction, int32_t* perm, int32_t* count, cudaStream_t st);

// calib.cu ---------------------------------------------------------------
int64_t second_moment_splits(int64_t M, int64_t H);
// partial: [2][splits][H][d][d] (hi and lo planes); status: an int32 the
// tensor-core kernel sets on a timed-out wait (zeroed here first).
cudaError_t launch_second_moment(const void* q, int dt, int64_t H, int64_t M, int64_t d,
                                 double ridge, float* partial, int32_t* status, float* h_out,
                                 cudaStream_t st);
// calib_tc.cu: the slices' partial sums on the tensor cores (16-bit queries,
// d = 128, slices short enough for fp32 accumulators); the same partial
// layout as the SIMT kernel.
bool second_moment_tc_supported(int dt, int64_t H, int64_t M, int64_t d);
cudaError_t launch_second_moment_tc(const void* q, int dt, int64_t H, int64_t M, float* partial,
                                    int32_t* status, cudaStream_t st);

cudaError_t launch_cholesky(const float* h, int64_t H, int64_t d, float* l_out, int32_t* info,
                            cudaStream_t st);

// Lc [H, d, d] = the lower triangle of L (zeros above the diagonal, which
// is all of L the library reads) and Lt [H, d, d] = Lc^T.
cudaError_t launch_factor_prep(const float* L, int64_t H, int64_t d, float* Lc, float* Lt,
                               cudaStream_t st);

// Transformed codebook for the assignment: cp [H, K, d] fp32 = c Lc (c when
// Lc is null) and half_norm [H, K] fp32 = |cp_j|^2 / 2; with Lc and chat
// given, also chat [H, K, d] fp32 = cp Lc^T (Lt = Lc^T).
cudaError_t launch_codebook_transform(const void* c, int dt, int64_t H, int64_t K, int64_t d,
                                      const float* Lc, const float* Lt, float* cp,
                                      float* half_norm, float* chat, cudaStream_t st);

// assign.cu --------------------------------------------------------------
struct RowSel {
    int32_t mode;  // a2ats_rows
    const int32_t* perm;
    const int32_t* count;
};

// Exact z-space assignment (SIMT, compensated fp32): code = argmin_j
// |x~ L - cp_j|^2.  L null = identity.
cudaError_t launch_assign_exact(const void* x, int dt, const Shape& s, const int32_t* len,
                                const RopeArgs& ra, const RowSel& sel, const float* L,
                                const float* cp, const float* half_norm, int64_t K,
                                int32_t* codes, cudaStream_t st);

// Cosine blend (SIMT): q [B*H, d] fp32 per-(b, h) query and its norm.
cudaError_t launch_assign_blend(const void* x, const void* c, int dt, const Shape& s,
                                const int32_t* len, const RopeArgs& ra, const RowSel& sel,
                                const float* q, const float* qnorm, float beta, int64_t K,
                                const float* cnorm, int32_t* codes, cudaStream_t st);

// assign_tc.cu ----------------------------------------------------------
// Centroids per group of the tensor-core pass's certification bound (the
// per-group maxima of |chat_j| and h_j, TcCall::gstat).
constexpr int kTcGroup = 16;

// Tensor-core assignment (argmin_j |x~ L - c_j L|^2, L null = identity) for
// bf16 / fp16 keys with d a multiple of 64.  cp / half_norm must already hold
// c L and |c L|^2 / 2, and with L given chat must hold c L L^T
// (launch_codebook_transform; L is the lower-triangular copy).  Rows inside the RoPE
// window and rows whose top two the contraction cannot separate are decided
// by the exact kernel.
struct TcCall {
    int dt;
    Shape s;
    int64_t K;
    const void* x;
    const void* codebook;
    const float* L;
    RopeArgs ra;
    RowSel sel;
    const int32_t* len;
    const float* cp;
    const float* half_norm;
    int32_t* codes;
    bool prepared;        // the codebook side is already in the workspace
    // workspace
    float* Lt;            // [H, d, d]  L^T
    float* chat;          // [H, K, d]  c L L^T
    float* chat_rot;      // [H, K, d]  the same, rotated by -far_offset
    float* hneg;          // [H, Kpad]  -|c L|^2 / 2, padded to 256 columns (fp16 keys)
    uint16_t* hplanes;    // [H, Kpad, 16] the same as the bf16 operand of one MMA step (bf16 keys)
    uint32_t* head_bits;  // [2, H, 4]
    float* head;          // [2, H, 4]
    float2* gstat;        // [2, H, Kpad / 32] group maxima of |chat_j| and h_j
    float* scale;         // [2, H]
    uint16_t* planes;     // [2, H, 3, K, d]
    uint16_t* compact;    // [2, B*H*Ncap, d] two 16-bit planes of rotated rows
    int32_t* row_map;     // [B*H*Ncap]
    int32_t* ccount;      // [B*H]
    uint8_t* skip;        // [B*H*Ncap]
    int64_t* exact_list;  // [B*H*Ncap]
    unsigned long long* exact_best;  // [B*H*Ncap] (distance bits, index) of listed rows
    int32_t* exact_done;  // [B*H*Ncap] centroid slices finished per listed row
    int32_t* exact_count; // [4]: count, status, longest compact list, unused
    int32_t* head_count;  // [H] listed rows per head (the exact path): exact_count + 4
    int32_t* tile_rot;    // [B*H, ceil(Ncap/128)] nonzero: that 128-row tile of the compact
                          // list holds a rotated row (head_count + H; zeroed with them)
    // optional, for the pass over the stored keys in natural order (rows
    // outside the RoPE window, far_offset = 0): the cosine of each row with
    // score_q of its (b, h) into scores, and a copy of the row into kcopy
    // (null: not taken)
    const float* score_q;   // [B*H, d]
    const float* score_qn;  // [B*H]
    float* scores;          // [B*H*Ncap]
    void* kcopy;            // [B*H*Ncap, d], the keys' dtype
    // optional: launched on the stream right after that pass, before the
    // rotated rows and the exact path
    cudaError_t (*after_natural)(void* ctx, cudaStream_t st);
    void* after_ctx;
};
bool tc_supported(int dt, int64_t d);
cudaError_t launch_assign_tc(const TcCall& c, cudaStream_t st);

// kmeans.cu --------------------------------------------------------------
// k-means++ seeds of z [H, n, d] fp32 with the draws u [H, K] into cent
// [H, K, d]; d2 [H, n] fp64 scratch.
cudaError_t launch_kmeans_seed(const float* z, int64_t H, int64_t n, int64_t d, int64_t K,
                               const double* u, float* cent, double* d2, cudaStream_t st);

// The objective of the assignment codes [H, n] against cent (sum over rows
// of |z_i - cent[code_i]|^2, fp64) into objective[h * obj_stride]; with
// update, each centroid then moves to the mean of its rows (kept when it has
// none).  obj_part [H, K] fp64 scratch.
cudaError_t launch_kmeans_update(const float* z, int64_t H, int64_t n, int64_t d, int64_t K,
                                 const int32_t* codes, float* cent, double* obj_part,
                                 bool update, double* objective, int64_t obj_stride,
                                 cudaStream_t st);

// c [H, rows, d] with c L = zc (back substitution on the lower triangle of L).
cudaError_t launch_cholesky_solve(const float* zc, int64_t H, int64_t rows, int64_t d,
                                  const float* L, float* c, cudaStream_t st);

// subvector.cu -----------------------------------------------------------
// Largest K * sub_dim a sub-vector table may have (both tables sit in
// shared memory).
int64_t subvector_table_limit();

// mark [B*H*Ncap] <- 1 for the tokens perm[:count] of each (b, h), 0 for the
// rest of the split (rows below len only).
cudaError_t launch_mark_retrieval(const int32_t* perm, const int32_t* count, const int32_t* len,
                                  const Shape& s, uint8_t* mark, cudaStream_t st);

// codes [B, H, Ncap, d / sub_dim] of the sub-vectors of x (rows below len):
// nearest entry of tab_plain [H, K, sub_dim], or, where Lc is given and the
// token is marked (every token when mark is null), nearest entry of
// tab_weighted = c Lc after z = x Lc.  sub_dim is 8 or 16.
cudaError_t launch_subvector_assign(const void* x, int dt, const Shape& s, const int32_t* len,
                                    int64_t sub_dim, const float* tab_plain,
                                    const float* tab_weighted, const float* Lc,
                                    const uint8_t* mark, int64_t K, int32_t* codes,
                                    cudaStream_t st);

// codes [B, H, Ncap, d / sub_dim] by the cosine blend on the marked tokens
// (every token when mark is null; none when beta = 1) with the query's
// slice g (query [B*H, d], or the row at t = len - 1 of x when null), plain
// VQ elsewhere; tab [H, K, sub_dim] the decoded table, cnorm [H, K] |c_k|.
cudaError_t launch_subvector_blend(const void* x, int dt, const Shape& s, const int32_t* len,
                                   int64_t sub_dim, const float* tab, const float* cnorm,
                                   const void* query, float beta, const uint8_t* mark, int64_t K,
                                   int32_t* codes, cudaStream_t st);

cudaError_t launch_centroid_norms(const void* c, int dt, int64_t H, int64_t K, int64_t d,
                                  float* cnorm, cudaStream_t st);

}  // namespace a2ats
