// api.cu -- the extern "C" entry points declared in include/a2ats.h.
//
// Each entry point checks its arguments on the host (nothing is enqueued when
// a check fails), carves its workspace, and enqueues the kernels on the
// caller's stream.  The operations follow the API page
// "veloxquant_mlx.quantizers.a2ats module" and the "A2ATS-adapted" algorithm
// pages; see include/a2ats.h for the contract of each call.
#include <math.h>
#include <stdio.h>
#include <string.h>

#include <atomic>
#include <vector>

#include "../../include/a2ats.h"
#include "entry.cuh"
#include "kernels.cuh"

using namespace a2ats;

namespace {
std::atomic<uint64_t> g_launches{0};
}  // namespace

void a2ats::note_launches(int n) { g_launches.fetch_add((uint64_t)n, std::memory_order_relaxed); }

namespace {
struct TimingPool {
    bool on = false;
    std::vector<cudaEvent_t> ev;  // pairs
    size_t used = 0;
};
TimingPool g_timing;
}  // namespace

bool a2ats::kernel_timing_on() { return g_timing.on; }

static cudaEvent_t timing_event() {
    if (g_timing.used == g_timing.ev.size()) {
        cudaEvent_t e;
        if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
        g_timing.ev.push_back(e);
    }
    return g_timing.ev[g_timing.used++];
}

void a2ats::timing_begin(cudaStream_t st) {
    if (!g_timing.on || (g_timing.used & 1)) return;
    cudaEvent_t e = timing_event();
    if (e) cudaEventRecord(e, st);
}

void a2ats::timing_end(cudaStream_t st) {
    if (!g_timing.on || !(g_timing.used & 1)) return;
    cudaEvent_t e = timing_event();
    if (e) cudaEventRecord(e, st);
}

namespace {
thread_local char g_last_error[256] = "";
}  // namespace

int a2ats::cuda_fail(cudaError_t e) {
    snprintf(g_last_error, sizeof(g_last_error), "%s: %s", cudaGetErrorName(e),
             cudaGetErrorString(e));
    return A2ATS_ERR_CUDA;
}

bool a2ats::dtype_ok(int32_t dt) {
    return dt == A2ATS_F32 || dt == A2ATS_BF16 || dt == A2ATS_F16;
}

int a2ats::check_shape(int64_t B, int64_t H, int64_t Ncap, int64_t d) {
    if (B < 0 || H < 0 || Ncap < 0) return A2ATS_ERR_SHAPE;
    if (d < 8 || d > kMaxD || d % 8 != 0) return A2ATS_ERR_SHAPE;
    if (Ncap >= (int64_t(1) << 24)) return A2ATS_ERR_SHAPE;
    if (B > (int64_t(1) << 20) || H > 4096 || B * H > 65535) return A2ATS_ERR_SHAPE;
    return A2ATS_OK;
}

bool a2ats::unit_interval(double v) { return v >= 0.0 && v <= 1.0; }

int a2ats::make_rope(const a2ats_rope_params* p, int64_t d, RopeArgs& ra) {
    memset(&ra, 0, sizeof(ra));
    if (!p) return A2ATS_OK;
    if (!(p->rope_base > 0.0) || !isfinite(p->rope_base)) return A2ATS_ERR_INVALID_ARG;
    if (p->far_offset <= -(1 << 24) || p->far_offset >= (1 << 24)) return A2ATS_ERR_INVALID_ARG;
    if (d % 2 != 0) return A2ATS_ERR_SHAPE;
    ra.enabled = 1;
    ra.window = p->window;
    ra.far_offset = p->far_offset;
    ra.interleaved = p->interleaved ? 1 : 0;
    const double two_pi = 6.283185307179586476925286766559;
    const float a = (float)two_pi;
    const float b = (float)(two_pi - (double)a);
    const float c = (float)(two_pi - (double)a - (double)b);
    ra.two_pi_a = a;
    ra.two_pi_b = b;
    ra.two_pi_c = c;
    ra.inv_2pi = (float)(1.0 / two_pi);
    for (int64_t i = 0; i < d / 2; i++) {
        const double om = pow(p->rope_base, -2.0 * (double)i / (double)d);
        ra.omega_hi[i] = (float)om;
        ra.omega_lo[i] = (float)(om - (double)ra.omega_hi[i]);
    }
    return A2ATS_OK;
}

namespace {

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

// Do the byte ranges [p, p + pb) and [q, q + qb) share a byte?
bool overlap(const void* p, size_t pb, const void* q, size_t qb) {
    const uintptr_t a = (uintptr_t)p, b = (uintptr_t)q;
    return a < b + qb && b < a + pb;
}


// Bump allocator over the caller's workspace (256-byte aligned pieces).
struct Carve {
    char* base;
    size_t used = 0;
    explicit Carve(void* p) : base((char*)p) {}
    template <class T>
    T* take(size_t count) {
        used = (used + 255) & ~size_t(255);
        T* p = base ? (T*)(base + used) : nullptr;
        used += sizeof(T) * count;
        return p;
    }
};

struct AssignWs {
    float* Lc;         // [H, d, d] lower triangle of L
    float* cp;         // [H, K, d] transformed (or decoded) centroids
    float* half_norm;  // [H, K]
    float* cnorm;      // [H, K]
    float* q;          // [B*H, d]
    float* qnorm;      // [B*H]
    TcCall tc;         // buffers of the tensor-core path
};

AssignWs carve_assign(Carve& c, int64_t B, int64_t H, int64_t Ncap, int64_t d, int64_t K) {
    AssignWs w;
    w.Lc = c.take<float>((size_t)(H * d * d));
    w.cp = c.take<float>((size_t)(H * K * d));
    w.half_norm = c.take<float>((size_t)(H * K));
    w.cnorm = c.take<float>((size_t)(H * K));
    w.q = c.take<float>((size_t)(B * H * d));
    w.qnorm = c.take<float>((size_t)(B * H));
    const size_t rows = (size_t)(B * H * Ncap);
    memset(&w.tc, 0, sizeof(w.tc));
    const int64_t kpad = (K + 255) / 256 * 256;
    w.tc.Lt = c.take<float>((size_t)(H * d * d));
    w.tc.chat = c.take<float>((size_t)(H * K * d));
    w.tc.chat_rot = c.take<float>((size_t)(H * K * d));
    w.tc.hneg = c.take<float>((size_t)(H * kpad));
    w.tc.hplanes = c.take<uint16_t>((size_t)(H * kpad * 16));
    w.tc.head_bits = c.take<uint32_t>((size_t)(2 * H * 4));
    w.tc.head = c.take<float>((size_t)(2 * H * 4));
    w.tc.gstat = c.take<float2>((size_t)(2 * H * (kpad / kTcGroup)));
    w.tc.scale = c.take<float>((size_t)(2 * H));
    w.tc.planes = c.take<uint16_t>((size_t)(2 * H * 3 * K * d));
    w.tc.compact = c.take<uint16_t>(2 * rows * (size_t)d);
    w.tc.row_map = c.take<int32_t>(rows);
    w.tc.ccount = c.take<int32_t>((size_t)(B * H));
    w.tc.skip = c.take<uint8_t>(rows);
    w.tc.exact_list = c.take<int64_t>(rows);
    w.tc.exact_best = c.take<unsigned long long>(rows);
    w.tc.exact_done = c.take<int32_t>(rows);
    // the counters, the per-head list lengths and the compact tiles' flags
    // are adjacent: one memset
    w.tc.exact_count = c.take<int32_t>((size_t)(4 + H + B * H * ((Ncap + 127) / 128)));
    w.tc.head_count = w.tc.exact_count + 4;
    w.tc.tile_rot = w.tc.head_count + H;
    return w;
}

// The tensor-core route for bf16 / fp16 keys (d a multiple of 64); cp and
// half_norm must hold c L and |c L|^2 / 2.
cudaError_t assign_on_tensor_cores(AssignWs& w, int32_t dtype, const Shape& sh,
                                   const int32_t* len, const void* x, const void* codebook,
                                   int64_t K, const float* L, const RopeArgs& ra,
                                   const RowSel& sel, int32_t* codes, cudaStream_t s) {
    TcCall& c = w.tc;
    c.dt = dtype;
    c.s = sh;
    c.K = K;
    c.x = x;
    c.codebook = codebook;
    c.L = L;
    c.ra = ra;
    c.sel = sel;
    c.len = len;
    c.cp = w.cp;
    c.half_norm = w.half_norm;
    c.codes = codes;
    return launch_assign_tc(c, s);
}

struct SelectWs {
    float* q;
    float* qnorm;
    float* scores;
};

SelectWs carve_select(Carve& c, int64_t B, int64_t H, int64_t Ncap, int64_t d) {
    SelectWs w;
    w.q = c.take<float>((size_t)(B * H * d));
    w.qnorm = c.take<float>((size_t)(B * H));
    w.scores = c.take<float>((size_t)(B * H * Ncap));
    return w;
}

int check_rows(int32_t rows, const int32_t* perm, const int32_t* count) {
    if (rows != A2ATS_ROWS_ALL && rows != A2ATS_ROWS_RETRIEVAL && rows != A2ATS_ROWS_BULK &&
        rows != A2ATS_ROWS_LAST)
        return A2ATS_ERR_INVALID_ARG;
    if ((rows == A2ATS_ROWS_RETRIEVAL || rows == A2ATS_ROWS_BULK) && (!perm || !count))
        return A2ATS_ERR_INVALID_ARG;
    return A2ATS_OK;
}

int check_assign_common(const void* x, int32_t dtype, int64_t B, int64_t H, int64_t Ncap,
                        int64_t d, const void* codebook, int64_t K, int32_t rows,
                        const int32_t* perm, const int32_t* count, const int32_t* codes) {
    if (!dtype_ok(dtype)) return A2ATS_ERR_DTYPE;
    int st = check_shape(B, H, Ncap, d);
    if (st) return st;
    if (K < 1 || K > (int64_t(1) << 24)) return A2ATS_ERR_SHAPE;
    if ((st = check_rows(rows, perm, count))) return st;
    if (B * H * Ncap == 0) return A2ATS_OK;
    if (!x || !codebook || !codes) return A2ATS_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(codebook) || !aligned16(codes)) return A2ATS_ERR_ALIGN;
    return A2ATS_OK;
}

}  // namespace

extern "C" {

const char* a2ats_status_string(int32_t status) {
    switch (status) {
        case A2ATS_OK: return "A2ATS_OK";
        case A2ATS_ERR_INVALID_ARG: return "A2ATS_ERR_INVALID_ARG";
        case A2ATS_ERR_SHAPE: return "A2ATS_ERR_SHAPE";
        case A2ATS_ERR_DTYPE: return "A2ATS_ERR_DTYPE";
        case A2ATS_ERR_ALIGN: return "A2ATS_ERR_ALIGN";
        case A2ATS_ERR_CUDA: return "A2ATS_ERR_CUDA";
        case A2ATS_ERR_WORKSPACE: return "A2ATS_ERR_WORKSPACE";
        case A2ATS_ERR_CAPACITY: return "A2ATS_ERR_CAPACITY";
        default: return "A2ATS_ERR_UNKNOWN";
    }
}

const char* a2ats_last_error(void) { return g_last_error; }

uint64_t a2ats_kernel_launches(void) { return g_launches.load(std::memory_order_relaxed); }

int a2ats_set_kernel_timing(int32_t enable) {
    g_timing.on = enable != 0;
    g_timing.used = 0;
    return A2ATS_OK;
}

double a2ats_timed_kernels_ms(int64_t* launches) {
    double total = 0.0;
    int64_t n = 0;
    for (size_t i = 0; i + 1 < g_timing.used; i += 2) {
        float ms = 0.f;
        if (cudaEventSynchronize(g_timing.ev[i + 1]) == cudaSuccess &&
            cudaEventElapsedTime(&ms, g_timing.ev[i], g_timing.ev[i + 1]) == cudaSuccess) {
            total += ms;
            n++;
        }
    }
    g_timing.used = 0;
    if (launches) *launches = n;
    return total;
}

int a2ats_windowed_rope(const void* k_in, int32_t in_dtype, void* k_out, int32_t out_dtype,
                        int64_t B, int64_t H, int64_t Ncap, int64_t d, const int32_t* len,
                        const a2ats_rope_params* rope, void* stream) {
    if (!dtype_ok(in_dtype) || !dtype_ok(out_dtype)) return A2ATS_ERR_DTYPE;
    int st = check_shape(B, H, Ncap, d);
    if (st) return st;
    if (!rope) return A2ATS_ERR_INVALID_ARG;
    RopeArgs ra;
    if ((st = make_rope(rope, d, ra))) return st;
    if (B * H * Ncap == 0) return A2ATS_OK;
    if (!k_in || !k_out) return A2ATS_ERR_INVALID_ARG;
    if (!aligned16(k_in) || !aligned16(k_out)) return A2ATS_ERR_ALIGN;
    if (k_in == k_out && in_dtype != out_dtype) return A2ATS_ERR_INVALID_ARG;
    cudaError_t e = launch_windowed_rope(k_in, in_dtype, k_out, out_dtype, Shape{B, H, Ncap, d},
                                         len, ra, (cudaStream_t)stream);
    return e == cudaSuccess ? A2ATS_OK : cuda_fail(e);
}

int a2ats_append_rows(void* cache, int32_t dtype, int64_t B, int64_t H, int64_t Ncap, int64_t d,
                      int32_t* len, const void* rows, void* stream) {
    if (!dtype_ok(dtype)) return A2ATS_ERR_DTYPE;
    int st = check_shape(B, H, Ncap, d);
    if (st) return st;
    if (B * H == 0 || Ncap == 0) return A2ATS_OK;
    if (!cache || !len || !rows) return A2ATS_ERR_INVALID_ARG;
    if (!aligned16(cache) || !aligned16(rows)) return A2ATS_ERR_ALIGN;
    cudaError_t e = launch_append_rows(cache, dtype, Shape{B, H, Ncap, d}, len, rows,
                                       (cudaStream_t)stream);
    return e == cudaSuccess ? A2ATS_OK : cuda_fail(e);
}

size_t a2ats_query_second_moment_workspace_size(int64_t H, int64_t M, int64_t d) {
    if (H < 0 || M < 1 || d < 1) return 0;
    Carve c(nullptr);
    c.take<float>((size_t)(2 * second_moment_splits(M, H) * H * d * d));
    c.take<int32_t>(4);
    return c.used + 256;
}

int a2ats_query_second_moment(const void* queries, int32_t dtype, int64_t H, int64_t M,
                              int64_t d, double ridge, float* h_out, void* workspace,
                              size_t workspace_bytes, void* stream) {
    if (!dtype_ok(dtype)) return A2ATS_ERR_DTYPE;
    if (H < 0 || H > 4096 || M < 1 || M >= (int64_t(1) << 31) || d < 8 || d > kMaxD || d % 8)
        return A2ATS_ERR_SHAPE;
    if (!(ridge >= 0.0) || !isfinite(ridge)) return A2ATS_ERR_INVALID_ARG;
    if (H == 0) return A2ATS_OK;
    if (!queries || !h_out) return A2ATS_ERR_INVALID_ARG;
    if (!aligned16(queries) || !aligned16(h_out)) return A2ATS_ERR_ALIGN;
    if (!workspace || workspace_bytes < a2ats_query_second_moment_workspace_size(H, M, d))
        return A2ATS_ERR_WORKSPACE;
    Carve c(workspace);
    float* partial = c.take<float>((size_t)(2 * second_moment_splits(M, H) * H * d * d));
    int32_t* status = c.take<int32_t>(4);
    cudaError_t e = launch_second_moment(queries, dtype, H, M, d, ridge, partial, status, h_out,
                                         (cudaStream_t)stream);
    return e == cudaSuccess ? A2ATS_OK : cuda_fail(e);
}

int a2ats_cholesky_factor(const float* h, int64_t H, int64_t d, float* l_out, int32_t* info,
                          void* stream) {
    if (H < 0 || H > 4096 || d < 8 || d > kMaxD || d % 8) return A2ATS_ERR_SHAPE;
    if (H == 0) return A2ATS_OK;
    if (!h || !l_out || !info) return A2ATS_ERR_INVALID_ARG;
    if (!aligned16(h) || !aligned16(l_out)) return A2ATS_ERR_ALIGN;
    cudaError_t e = launch_cholesky(h, H, d, l_out, info, (cudaStream_t)stream);
    return e == cudaSuccess ? A2ATS_OK : cuda_fail(e);
}

size_t a2ats_h_weighted_assign_workspace_size(int64_t B, int64_t H, int64_t Ncap, int64_t d,
                                              int64_t K) {
    Carve c(nullptr);
    carve_assign(c, B, H, Ncap, d, K);
    return c.used + 256;
}

namespace {
// The H-weighted assignment; with reuse, the codebook side (the copy of L,
// c L, |c L|^2 / 2, c L L^T, its planes and tables) is taken as an earlier
// call on this workspace left it.
int h_weighted(const void* x, int32_t dtype, int64_t B, int64_t H, int64_t Ncap, int64_t d,
               const int32_t* len, const void* codebook, int64_t K, const float* L,
               const a2ats_rope_params* fused_rope, int32_t rows, const int32_t* perm,
               const int32_t* count, int32_t* codes, void* workspace, size_t workspace_bytes,
               void* stream, bool reuse) {
    int st = check_assign_common(x, dtype, B, H, Ncap, d, codebook, K, rows, perm, count, codes);
    if (st) return st;
    RopeArgs ra;
    if ((st = make_rope(fused_rope, d, ra))) return st;
    if (B * H * Ncap == 0) return A2ATS_OK;
    if (L && !aligned16(L)) return A2ATS_ERR_ALIGN;
    if (!workspace ||
        workspace_bytes < a2ats_h_weighted_assign_workspace_size(B, H, Ncap, d, K))
        return A2ATS_ERR_WORKSPACE;
    Carve c(workspace);
    AssignWs w = carve_assign(c, B, H, Ncap, d, K);
    cudaStream_t s = (cudaStream_t)stream;
    cudaError_t e;
    // only the lower triangle of L is read: every kernel uses the masked copy
    const float* Lc = L ? w.Lc : nullptr;
    const bool tc = tc_supported(dtype, d) && 2 * B * H * Ncap < (int64_t(1) << 30);
    if (!reuse) {
        if (L && (e = launch_factor_prep(L, H, d, w.Lc, w.tc.Lt, s)) != cudaSuccess)
            return cuda_fail(e);
        e = launch_codebook_transform(codebook, dtype, H, K, d, Lc, w.tc.Lt, w.cp, w.half_norm,
                                      tc ? w.tc.chat : nullptr, s);
        if (e != cudaSuccess) return cuda_fail(e);
    }
    const Shape sh{B, H, Ncap, d};
    if (tc) {
        w.tc.prepared = reuse;
        e = assign_on_tensor_cores(w, dtype, sh, len, x, codebook, K, Lc, ra,
                                   RowSel{rows, perm, count}, codes, s);
    } else {
        e = launch_assign_exact(x, dtype, sh, len, ra, RowSel{rows, perm, count}, Lc, w.cp,
                                w.half_norm, K, codes, s);
    }
    return e == cudaSuccess ? A2ATS_OK : cuda_fail(e);
}
}  // namespace

int a2ats_h_weighted_assign(const void* x, int32_t dtype, int64_t B, int64_t H, int64_t Ncap,
                            int64_t d, const int32_t* len, const void* codebook, int64_t K,
                            const float* L, const a2ats_rope_params* fused_rope, int32_t rows,
                            const int32_t* perm, const int32_t* count, int32_t* codes,
                            void* workspace, size_t workspace_bytes, void* stream) {
    return h_weighted(x, dtype, B, H, Ncap, d, len, codebook, K, L, fused_rope, rows, perm, count,
                      codes, workspace, workspace_bytes, stream, false);
}

int a2ats_h_weighted_assign_reuse(const void* x, int32_t dtype, int64_t B, int64_t H,
                                  int64_t Ncap, int64_t d, const int32_t* len,
                                  const void* codebook, int64_t K, const float* L,
                                  const a2ats_rope_params* fused_rope, int32_t rows,
                                  const int32_t* perm, const int32_t* count, int32_t* codes,
                                  void* workspace, size_t workspace_bytes, void* stream) {
    return h_weighted(x, dtype, B, H, Ncap, d, len, codebook, K, L, fused_rope, rows, perm, count,
                      codes, workspace, workspace_bytes, stream, true);
}

size_t a2ats_query_aware_assign_workspace_size(int64_t B, int64_t H, int64_t Ncap, int64_t d,
                                               int64_t K) {
    return a2ats_h_weighted_assign_workspace_size(B, H, Ncap, d, K);
}

namespace {
// The cosine blend; reuse: the codebook side (decoded centroids, their
// norms and |c|^2 / 2, and for beta = 1 the contraction's planes and
// tables) is the one the last call on this workspace left.
int query_aware(const void* x, int32_t dtype, int64_t B, int64_t H, int64_t Ncap, int64_t d,
                const int32_t* len, const void* codebook, int64_t K, const void* query,
                double beta, const a2ats_rope_params* fused_rope, int32_t rows,
                const int32_t* perm, const int32_t* count, int32_t* codes, void* workspace,
                size_t workspace_bytes, void* stream, bool reuse) {
    int st = check_assign_common(x, dtype, B, H, Ncap, d, codebook, K, rows, perm, count, codes);
    if (st) return st;
    if (!unit_interval(beta)) return A2ATS_ERR_INVALID_ARG;
    RopeArgs ra;
    if ((st = make_rope(fused_rope, d, ra))) return st;
    if (B * H * Ncap == 0) return A2ATS_OK;
    if (query && !aligned16(query)) return A2ATS_ERR_ALIGN;
    if (!workspace ||
        workspace_bytes < a2ats_query_aware_assign_workspace_size(B, H, Ncap, d, K))
        return A2ATS_ERR_WORKSPACE;
    Carve c(workspace);
    AssignWs w = carve_assign(c, B, H, Ncap, d, K);
    cudaStream_t s = (cudaStream_t)stream;
    const Shape sh{B, H, Ncap, d};
    // decoded fp32 centroids (and |c|^2 / 2) for either rule
    cudaError_t e = cudaSuccess;
    if (!reuse) {
        e = launch_codebook_transform(codebook, dtype, H, K, d, nullptr, nullptr, w.cp,
                                      w.half_norm, nullptr, s);
        if (e != cudaSuccess) return cuda_fail(e);
    }
    if (beta == 1.0) {
        // beta = 1 is plain nearest-centroid VQ: the same argmin as the
        // H-weighted rule with L = I, so it reduces exactly by construction
        if (tc_supported(dtype, d) && 2 * B * H * Ncap < (int64_t(1) << 30)) {
            w.tc.prepared = reuse;
            e = assign_on_tensor_cores(w, dtype, sh, len, x, codebook, K, nullptr, ra,
                                       RowSel{rows, perm, count}, codes, s);
        } else {
            e = launch_assign_exact(x, dtype, sh, len, ra, RowSel{rows, perm, count}, nullptr,
                                    w.cp, w.half_norm, K, codes, s);
        }
        return e == cudaSuccess ? A2ATS_OK : cuda_fail(e);
    }
    if (!reuse) {
        e = launch_centroid_norms(codebook, dtype, H, K, d, w.cnorm, s);
        if (e != cudaSuccess) return cuda_fail(e);
    }
    // the per-(b, h) query: decoded as given, or the proxy k~ at t
    e = launch_prepare_query(x, query, dtype, sh, len, ra, w.q, w.qnorm, s);
    if (e != cudaSuccess) return cuda_fail(e);
    e = launch_assign_blend(x, w.cp, dtype, sh, len, ra, RowSel{rows, perm, count}, w.q,
                            w.qnorm, (float)beta, K, w.cnorm, codes, s);
    return e == cudaSuccess ? A2ATS_OK : cuda_fail(e);
}
}  // namespace

int a2ats_query_aware_assign(const void* x, int32_t dtype, int64_t B, int64_t H, int64_t Ncap,
                             int64_t d, const int32_t* len, const void* codebook, int64_t K,
                             const void* query, double beta, const a2ats_rope_params* fused_rope,
                             int32_t rows, const int32_t* perm, const int32_t* count,
                             int32_t* codes, void* workspace, size_t workspace_bytes,
                             void* stream) {
    return query_aware(x, dtype, B, H, Ncap, d, len, codebook, K, query, beta, fused_rope, rows,
                       perm, count, codes, workspace, workspace_bytes, stream, false);
}

int a2ats_query_aware_assign_reuse(const void* x, int32_t dtype, int64_t B, int64_t H,
                                   int64_t Ncap, int64_t d, const int32_t* len,
                                   const void* codebook, int64_t K, const void* query,
                                   double beta, const a2ats_rope_params* fused_rope, int32_t rows,
                                   const int32_t* perm, const int32_t* count, int32_t* codes,
                                   void* workspace, size_t workspace_bytes, void* stream) {
    return query_aware(x, dtype, B, H, Ncap, d, len, codebook, K, query, beta, fused_rope, rows,
                       perm, count, codes, workspace, workspace_bytes, stream, true);
}

size_t a2ats_select_retrieval_set_workspace_size(int64_t B, int64_t H, int64_t Ncap, int64_t d) {
    Carve c(nullptr);
    carve_select(c, B, H, Ncap, d);
    return c.used + 256;
}

int a2ats_select_retrieval_set(const void* keys, int32_t dtype, int64_t B, int64_t H,
                               int64_t Ncap, int64_t d, const int32_t* len, const void* query,
                               double fraction, const a2ats_rope_params* fused_rope,
                               int32_t* perm, int32_t* count, void* workspace,
                               size_t workspace_bytes, void* stream) {
    if (!dtype_ok(dtype)) return A2ATS_ERR_DTYPE;
    int st = check_shape(B, H, Ncap, d);
    if (st) return st;
    if (!unit_interval(fraction)) return A2ATS_ERR_INVALID_ARG;
    RopeArgs ra;
    if ((st = make_rope(fused_rope, d, ra))) return st;
    if (B * H == 0) return A2ATS_OK;
    if (!count || (Ncap > 0 && (!keys || !perm))) return A2ATS_ERR_INVALID_ARG;
    if ((keys && !aligned16(keys)) || (query && !aligned16(query)) || (perm && !aligned16(perm)))
        return A2ATS_ERR_ALIGN;
    if (!workspace || workspace_bytes < a2ats_select_retrieval_set_workspace_size(B, H, Ncap, d))
        return A2ATS_ERR_WORKSPACE;
    Carve c(workspace);
    SelectWs w = carve_select(c, B, H, Ncap, d);
    cudaStream_t s = (cudaStream_t)stream;
    const Shape sh{B, H, Ncap, d};
    cudaError_t e = cudaSuccess;
    if (Ncap > 0) {
        e = launch_prepare_query(keys, query, dtype, sh, len, ra, w.q, w.qnorm, s);
        if (e != cudaSuccess) return cuda_fail(e);
        e = launch_cosine_scores(keys, dtype, sh, len, ra, w.q, w.qnorm, w.scores, s);
        if (e != cudaSuccess) return cuda_fail(e);
    }
    e = launch_select(w.scores, sh, len, fraction, perm, count, s);
    return e == cudaSuccess ? A2ATS_OK : cuda_fail(e);
}

int a2ats_select_retrieval_set_rotated(const void* keys, int32_t dtype, int64_t B, int64_t H,
                                       int64_t Ncap, int64_t d, const int32_t* len,
                                       const void* query, double fraction,
                                       const a2ats_rope_params* rope, void* k_out,
                                       int32_t out_dtype, int32_t* perm, int32_t* count,
                                       void* workspace, size_t workspace_bytes, void* stream) {
    if (!dtype_ok(dtype) || !dtype_ok(out_dtype)) return A2ATS_ERR_DTYPE;
    int st = check_shape(B, H, Ncap, d);
    if (st) return st;
    if (!unit_interval(fraction)) return A2ATS_ERR_INVALID_ARG;
    if (!rope) return A2ATS_ERR_INVALID_ARG;
    RopeArgs ra;
    if ((st = make_rope(rope, d, ra))) return st;
    if (B * H == 0) return A2ATS_OK;
    if (!count || (Ncap > 0 && (!keys || !perm || !k_out))) return A2ATS_ERR_INVALID_ARG;
    if ((keys && !aligned16(keys)) || (query && !aligned16(query)) || (perm && !aligned16(perm)) ||
        (k_out && !aligned16(k_out)))
        return A2ATS_ERR_ALIGN;
    // the keys are read again after k_out is written, so they may not share memory
    if (Ncap > 0 && k_out == keys) return A2ATS_ERR_INVALID_ARG;
    if (!workspace || workspace_bytes < a2ats_select_retrieval_set_workspace_size(B, H, Ncap, d))
        return A2ATS_ERR_WORKSPACE;
    Carve c(workspace);
    SelectWs w = carve_select(c, B, H, Ncap, d);
    cudaStream_t s = (cudaStream_t)stream;
    const Shape sh{B, H, Ncap, d};
    cudaError_t e = cudaSuccess;
    if (Ncap > 0) {
        e = launch_prepare_query(keys, query, dtype, sh, len, ra, w.q, w.qnorm, s);
        if (e != cudaSuccess) return cuda_fail(e);
        e = launch_cosine_scores(keys, dtype, sh, len, ra, w.q, w.qnorm, w.scores, s, k_out,
                                 out_dtype);
        if (e == cudaErrorNotSupported) {
            // no fused form for this width: rotate in a pass of its own
            e = launch_cosine_scores(keys, dtype, sh, len, ra, w.q, w.qnorm, w.scores, s);
            if (e == cudaSuccess)
                e = launch_windowed_rope(keys, dtype, k_out, out_dtype, sh, len, ra, s);
        }
        if (e != cudaSuccess) return cuda_fail(e);
    }
    e = launch_select(w.scores, sh, len, fraction, perm, count, s);
    return e == cudaSuccess ? A2ATS_OK : cuda_fail(e);
}

size_t a2ats_rope_split_plain_assign_workspace_size(int64_t B, int64_t H, int64_t Ncap,
                                                    int64_t d, int64_t K) {
    Carve c(nullptr);
    carve_assign(c, B, H, Ncap, d, K);
    carve_select(c, B, H, Ncap, d);
    return c.used + 256;
}

namespace {
// The split, launched between the pass over the stored keys (the last
// scores it needs) and the rest of the assignment; then the caller's event.
struct SplitAfter {
    const float* scores;
    Shape sh;
    const int32_t* len;
    double fraction;
    int32_t* perm;
    int32_t* count;
    cudaEvent_t done;
    cudaStream_t side;  // or null: the split runs on the call's stream
};

// With a side stream the split forks there through `done` (recorded on st
// once the scores are written, waited on by side) and `done` is recorded
// again on side after it; the call's stream joins it at the end.
cudaError_t split_after_natural(void* ctx, cudaStream_t st) {
    const SplitAfter* a = static_cast<const SplitAfter*>(ctx);
    cudaStream_t on = st;
    cudaError_t e = cudaSuccess;
    if (a->side) {
        e = cudaEventRecord(a->done, st);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(a->side, a->done, 0);
        on = a->side;
    }
    if (e == cudaSuccess)
        e = launch_select(a->scores, a->sh, a->len, a->fraction, a->perm, a->count, on);
    if (e == cudaSuccess && a->done) e = cudaEventRecord(a->done, on);
    return e;
}

cudaError_t join_split(const SplitAfter& a, cudaStream_t st, cudaError_t e) {
    if (e == cudaSuccess && a.side) e = cudaStreamWaitEvent(st, a.done, 0);
    return e;
}
}  // namespace

int a2ats_rope_split_plain_assign(const void* keys, int32_t dtype, int64_t B, int64_t H,
                                  int64_t Ncap, int64_t d, const int32_t* len, const void* query,
                                  double fraction, const a2ats_rope_params* rope,
                                  const void* codebook, int64_t K, void* k_out, int32_t* perm,
                                  int32_t* count, int32_t* codes, int32_t reuse,
                                  void* split_done, void* split_stream, void* workspace,
                                  size_t workspace_bytes, void* stream) {
    if (!dtype_ok(dtype)) return A2ATS_ERR_DTYPE;
    int st = check_shape(B, H, Ncap, d);
    if (st) return st;
    if (K < 1 || K > (int64_t(1) << 24)) return A2ATS_ERR_SHAPE;
    if (!unit_interval(fraction)) return A2ATS_ERR_INVALID_ARG;
    if (!rope) return A2ATS_ERR_INVALID_ARG;
    if (split_stream && (!split_done || split_stream == stream)) return A2ATS_ERR_INVALID_ARG;
    RopeArgs ra;
    if ((st = make_rope(rope, d, ra))) return st;
    if (B * H == 0) return A2ATS_OK;
    if (!count || (Ncap > 0 && (!keys || !perm || !k_out || !codebook || !codes)))
        return A2ATS_ERR_INVALID_ARG;
    if ((keys && !aligned16(keys)) || (query && !aligned16(query)) || (perm && !aligned16(perm)) ||
        (k_out && !aligned16(k_out)) || (codebook && !aligned16(codebook)) ||
        (codes && !aligned16(codes)))
        return A2ATS_ERR_ALIGN;
    // the keys are read again after k_out is written, so they may not share memory
    if (Ncap > 0 && k_out == keys) return A2ATS_ERR_INVALID_ARG;
    if (!workspace ||
        workspace_bytes < a2ats_rope_split_plain_assign_workspace_size(B, H, Ncap, d, K))
        return A2ATS_ERR_WORKSPACE;
    Carve c(workspace);
    AssignWs w = carve_assign(c, B, H, Ncap, d, K);
    SelectWs sw = carve_select(c, B, H, Ncap, d);
    cudaStream_t s = (cudaStream_t)stream;
    const Shape sh{B, H, Ncap, d};
    SplitAfter after{sw.scores, sh, len, fraction, perm, count, (cudaEvent_t)split_done,
                     (cudaStream_t)split_stream};
    cudaError_t e;
    if (Ncap == 0) {
        e = join_split(after, s, split_after_natural(&after, s));
        return e == cudaSuccess ? A2ATS_OK : cuda_fail(e);
    }
    const bool tc = tc_supported(dtype, d) && 2 * B * H * Ncap < (int64_t(1) << 30);
    // one pass over the stored keys serves all three when the far rows are
    // the keys themselves (far_offset = 0)
    const bool fused = tc && ra.far_offset == 0;
    if (!fused) {
        e = launch_prepare_query(keys, query, dtype, sh, len, ra, sw.q, sw.qnorm, s);
        if (e != cudaSuccess) return cuda_fail(e);
        // the separate passes: RoPE and scores, the split, then plain VQ
        e = launch_cosine_scores(keys, dtype, sh, len, ra, sw.q, sw.qnorm, sw.scores, s, k_out,
                                 dtype);
        if (e == cudaErrorNotSupported) {
            e = launch_cosine_scores(keys, dtype, sh, len, ra, sw.q, sw.qnorm, sw.scores, s);
            if (e == cudaSuccess) e = launch_windowed_rope(keys, dtype, k_out, dtype, sh, len, ra, s);
        }
        if (e == cudaSuccess) e = split_after_natural(&after, s);
        if (e != cudaSuccess) return cuda_fail(e);
    } else {
        // the query, and the RoPE window: rotated rows and their scores
        e = launch_window_scores(keys, query, dtype, sh, len, ra, sw.q, sw.qnorm, sw.scores, k_out,
                                 s);
        if (e != cudaSuccess) return cuda_fail(e);
    }
    if (!reuse) {
        e = launch_codebook_transform(codebook, dtype, H, K, d, nullptr, w.tc.Lt, w.cp,
                                      w.half_norm, tc ? w.tc.chat : nullptr, s);
        if (e != cudaSuccess) return cuda_fail(e);
    }
    const RowSel all{A2ATS_ROWS_ALL, nullptr, nullptr};
    if (tc) {
        w.tc.prepared = reuse != 0;
        if (fused) {
            w.tc.score_q = sw.q;
            w.tc.score_qn = sw.qnorm;
            w.tc.scores = sw.scores;
            w.tc.kcopy = k_out;
            w.tc.after_natural = split_after_natural;
            w.tc.after_ctx = &after;
        }
        e = assign_on_tensor_cores(w, dtype, sh, len, keys, codebook, K, nullptr, ra, all, codes,
                                   s);
    } else {
        e = launch_assign_exact(keys, dtype, sh, len, ra, all, nullptr, w.cp, w.half_norm, K,
                                codes, s);
    }
    e = join_split(after, s, e);
    return e == cudaSuccess ? A2ATS_OK : cuda_fail(e);
}

size_t a2ats_code_attention_topk_workspace_size(int64_t B, int64_t H, int64_t Ncap, int64_t d,
                                                int64_t K) {
    (void)Ncap;
    if (B < 0 || H < 0 || d < 0 || K < 0) return 0;
    Carve c(nullptr);
    c.take<float>((size_t)(B * H * d));  // RoPE(q, t)
    c.take<float>((size_t)(B * H * K));  // the per-(b, h) table
    return c.used + 256;
}

int a2ats_code_attention_topk(const void* keys, int32_t dtype, int64_t B, int64_t H, int64_t Ncap,
                              int64_t d, const int32_t* len, const int32_t* codes,
                              const void* codebook, int64_t K, const void* query,
                              const a2ats_rope_params* rope, int32_t far_b, double fraction,
                              float* scores, int32_t* perm, int32_t* count, void* workspace,
                              size_t workspace_bytes, void* stream) {
    if (!dtype_ok(dtype)) return A2ATS_ERR_DTYPE;
    int st = check_shape(B, H, Ncap, d);
    if (st) return st;
    if (K < 1 || K > (int64_t(1) << 24)) return A2ATS_ERR_SHAPE;
    if (!unit_interval(fraction)) return A2ATS_ERR_INVALID_ARG;
    if (!rope) return A2ATS_ERR_INVALID_ARG;
    if (far_b <= -(1 << 24) || far_b >= (1 << 24)) return A2ATS_ERR_INVALID_ARG;
    RopeArgs ra;
    if ((st = make_rope(rope, d, ra))) return st;
    if (B * H == 0) return A2ATS_OK;
    if (!count || (Ncap > 0 && (!keys || !codes || !codebook || !query || !scores || !perm)))
        return A2ATS_ERR_INVALID_ARG;
    if ((keys && !aligned16(keys)) || (codes && !aligned16(codes)) ||
        (codebook && !aligned16(codebook)) || (query && !aligned16(query)) ||
        (scores && !aligned16(scores)) || (perm && !aligned16(perm)))
        return A2ATS_ERR_ALIGN;
    if (!workspace ||
        workspace_bytes < a2ats_code_attention_topk_workspace_size(B, H, Ncap, d, K))
        return A2ATS_ERR_WORKSPACE;
    Carve c(workspace);
    float* q_near = c.take<float>((size_t)(B * H * d));
    float* lut = c.take<float>((size_t)(B * H * K));
    cudaStream_t s = (cudaStream_t)stream;
    const Shape sh{B, H, Ncap, d};
    cudaError_t e = launch_code_attention(keys, dtype, sh, len, codes, codebook, K, query, ra,
                                          far_b, q_near, lut, scores, s);
    if (e == cudaSuccess) e = launch_select(scores, sh, len, fraction, perm, count, s);
    return e == cudaSuccess ? A2ATS_OK : cuda_fail(e);
}

int a2ats_dequantize(const int32_t* codes, const void* codebook, int32_t dtype, int64_t B,
                     int64_t H, int64_t Ncap, int64_t d, int64_t K, const int32_t* len, void* out,
                     void* stream) {
    if (!dtype_ok(dtype)) return A2ATS_ERR_DTYPE;
    int st = check_shape(B, H, Ncap, d);
    if (st) return st;
    if (K < 1 || K > (int64_t(1) << 24)) return A2ATS_ERR_SHAPE;
    if (B * H * Ncap == 0) return A2ATS_OK;
    if (!codes || !codebook || !out) return A2ATS_ERR_INVALID_ARG;
    if (!aligned16(codes) || !aligned16(codebook) || !aligned16(out)) return A2ATS_ERR_ALIGN;
    if (out == codebook) return A2ATS_ERR_INVALID_ARG;
    cudaError_t e = launch_dequantize(codes, codebook, dtype, Shape{B, H, Ncap, d}, K, len, out,
                                      (cudaStream_t)stream);
    return e == cudaSuccess ? A2ATS_OK : cuda_fail(e);
}

int a2ats_byte_accounting(int64_t tokens, int64_t d, int64_t sub_dim, int32_t codebook_bits,
                          a2ats_cache_bytes* out) {
    if (!out) return A2ATS_ERR_INVALID_ARG;
    if (tokens < 0 || d < 1) return A2ATS_ERR_SHAPE;
    if (sub_dim < 1 || codebook_bits < 1 || codebook_bits > 24) return A2ATS_ERR_INVALID_ARG;
    if (d % sub_dim != 0) return A2ATS_ERR_SHAPE;
    const double groups = (double)(d / sub_dim);
    out->compressed_key_bytes = (double)tokens * groups * (double)codebook_bits / 8.0;
    out->compressed_value_bytes = out->compressed_key_bytes;
    out->fp16_key_bytes = (double)tokens * (double)d * 2.0;
    out->fp16_value_bytes = out->fp16_key_bytes;
    out->compression_ratio = 16.0 * (double)sub_dim / (double)codebook_bits;
    out->codebook_bytes = (double)(int64_t(1) << codebook_bits) * (double)sub_dim * 2.0;
    out->assigned_avg_bits = (double)codebook_bits / (double)sub_dim;
    return A2ATS_OK;
}

int a2ats_copy_retrieval_rows(const int32_t* src, int32_t* dst, int64_t B, int64_t H,
                              int64_t Ncap, const int32_t* len, const int32_t* perm,
                              const int32_t* count, void* stream) {
    if (B < 0 || H < 0 || Ncap < 0 || Ncap >= (int64_t(1) << 31) || B * H > 65535)
        return A2ATS_ERR_SHAPE;
    if (B * H == 0 || Ncap == 0) return A2ATS_OK;
    if (!src || !dst || !perm || !count) return A2ATS_ERR_INVALID_ARG;
    cudaError_t e = launch_copy_retrieval_rows(src, dst, Shape{B, H, Ncap, 8}, len, perm, count,
                                               (cudaStream_t)stream);
    return e == cudaSuccess ? A2ATS_OK : cuda_fail(e);
}

size_t a2ats_cholesky_rows_workspace_size(int64_t H, int64_t n, int64_t d) {
    if (H < 0 || n < 0 || d < 0) return 0;
    Carve c(nullptr);
    c.take<float>((size_t)(H * d * d));  // lower triangle of L
    c.take<float>((size_t)(H * d * d));  // its transpose
    c.take<float>((size_t)(H * n));      // |z|^2 / 2 (written, not returned)
    return c.used + 256;
}

int a2ats_cholesky_rows(const void* x, int32_t dtype, int64_t H, int64_t n, int64_t d,
                        const float* L, float* z, void* workspace, size_t workspace_bytes,
                        void* stream) {
    if (!dtype_ok(dtype)) return A2ATS_ERR_DTYPE;
    if (H < 0 || H > 4096 || n < 0 || n >= (int64_t(1) << 24) || d < 8 || d > kMaxD || d % 8)
        return A2ATS_ERR_SHAPE;
    if (H * n == 0) return A2ATS_OK;
    if (!x || !L || !z) return A2ATS_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(L) || !aligned16(z)) return A2ATS_ERR_ALIGN;
    if ((const void*)z == x) return A2ATS_ERR_INVALID_ARG;
    if (!workspace || workspace_bytes < a2ats_cholesky_rows_workspace_size(H, n, d))
        return A2ATS_ERR_WORKSPACE;
    Carve c(workspace);
    float* Lc = c.take<float>((size_t)(H * d * d));
    float* Lt = c.take<float>((size_t)(H * d * d));
    float* half_norm = c.take<float>((size_t)(H * n));
    cudaStream_t s = (cudaStream_t)stream;
    cudaError_t e = launch_factor_prep(L, H, d, Lc, Lt, s);
    if (e == cudaSuccess)
        e = launch_codebook_transform(x, dtype, H, n, d, Lc, nullptr, z, half_norm, nullptr, s);
    return e == cudaSuccess ? A2ATS_OK : cuda_fail(e);
}

int a2ats_cholesky_solve_rows(const float* zc, int64_t H, int64_t rows, int64_t d, const float* L,
                              float* c, void* stream) {
    if (H < 0 || H > 4096 || rows < 0 || rows > (int64_t(1) << 24) || d < 8 || d > kMaxD ||
        d % 8 || H * rows > (int64_t(1) << 30))
        return A2ATS_ERR_SHAPE;
    if (H * rows == 0) return A2ATS_OK;
    if (!zc || !L || !c) return A2ATS_ERR_INVALID_ARG;
    if (!aligned16(zc) || !aligned16(L) || !aligned16(c)) return A2ATS_ERR_ALIGN;
    cudaError_t e = launch_cholesky_solve(zc, H, rows, d, L, c, (cudaStream_t)stream);
    return e == cudaSuccess ? A2ATS_OK : cuda_fail(e);
}

size_t a2ats_kmeanspp_workspace_size(int64_t H, int64_t n, int64_t d, int64_t K) {
    if (H < 0 || n < 0 || d < 0 || K < 0) return 0;
    Carve c(nullptr);
    c.take<double>((size_t)(H * n));  // D^2 of the seeding
    c.take<double>((size_t)(H * K));  // per-centroid objectives
    c.take<char>(a2ats_h_weighted_assign_workspace_size(1, H, n, d, K));
    return c.used + 256;
}

int a2ats_kmeanspp(const float* z, int64_t H, int64_t n, int64_t d, int64_t K, const double* u,
                   int32_t iters, float* centroids, int32_t* codes, double* objective,
                   void* workspace, size_t workspace_bytes, void* stream) {
    if (H < 0 || H > 4096 || n < 0 || n >= (int64_t(1) << 24) || d < 8 || d > kMaxD || d % 8)
        return A2ATS_ERR_SHAPE;
    if (K < 1 || K > (int64_t(1) << 24)) return A2ATS_ERR_SHAPE;
    if (iters < 0 || iters > (1 << 20)) return A2ATS_ERR_INVALID_ARG;
    if (H == 0) return A2ATS_OK;
    if (n == 0) return A2ATS_ERR_SHAPE;
    if (!z || !u || !centroids || !codes || !objective) return A2ATS_ERR_INVALID_ARG;
    if (!aligned16(z) || !aligned16(centroids) || !aligned16(codes) || ((uintptr_t)u & 7u) ||
        ((uintptr_t)objective & 7u))
        return A2ATS_ERR_ALIGN;
    const size_t zb = sizeof(float) * (size_t)(H * n * d), cb = sizeof(float) * (size_t)(H * K * d),
                 kb = sizeof(int32_t) * (size_t)(H * n);
    if (overlap(z, zb, centroids, cb) || overlap(z, zb, codes, kb) ||
        overlap(centroids, cb, codes, kb))
        return A2ATS_ERR_INVALID_ARG;
    if (!workspace || workspace_bytes < a2ats_kmeanspp_workspace_size(H, n, d, K))
        return A2ATS_ERR_WORKSPACE;
    Carve c(workspace);
    double* d2 = c.take<double>((size_t)(H * n));
    double* obj_part = c.take<double>((size_t)(H * K));
    const size_t assign_bytes = a2ats_h_weighted_assign_workspace_size(1, H, n, d, K);
    void* assign_ws = c.take<char>(assign_bytes);
    cudaStream_t s = (cudaStream_t)stream;
    cudaError_t e = launch_kmeans_seed(z, H, n, d, K, u, centroids, d2, s);
    if (e != cudaSuccess) return cuda_fail(e);
    for (int32_t r = 0; r <= iters; r++) {
        // nearest centroid of every row (L = identity), then the mean step
        const int st = h_weighted(z, A2ATS_F32, 1, H, n, d, nullptr, centroids, K, nullptr,
                                  nullptr, A2ATS_ROWS_ALL, nullptr, nullptr, codes, assign_ws,
                                  assign_bytes, stream, false);
        if (st) return st;
        e = launch_kmeans_update(z, H, n, d, K, codes, centroids, obj_part, r < iters,
                                 objective + r, (int64_t)iters + 1, s);
        if (e != cudaSuccess) return cuda_fail(e);
    }
    return A2ATS_OK;
}

size_t a2ats_subvector_assign_workspace_size(int64_t B, int64_t H, int64_t Ncap, int64_t d,
                                             int64_t sub_dim, int64_t K) {
    (void)d;
    if (B < 0 || H < 0 || Ncap < 0 || sub_dim < 0 || K < 0) return 0;
    Carve c(nullptr);
    c.take<float>((size_t)(H * sub_dim * sub_dim));  // lower triangle of L
    c.take<float>((size_t)(H * sub_dim * sub_dim));  // its transpose
    c.take<float>((size_t)(H * K * sub_dim));        // decoded table
    c.take<float>((size_t)(H * K * sub_dim));        // table times L
    c.take<float>((size_t)(H * K));                  // half norms (written, not read)
    c.take<uint8_t>((size_t)(B * H * Ncap));         // retrieval marks
    return c.used + 256;
}

int a2ats_subvector_assign(const void* x, int32_t dtype, int64_t B, int64_t H, int64_t Ncap,
                           int64_t d, const int32_t* len, int64_t sub_dim, const void* codebook,
                           int64_t K, const float* L, const int32_t* perm, const int32_t* count,
                           int32_t* codes, void* workspace, size_t workspace_bytes,
                           void* stream) {
    if (!dtype_ok(dtype)) return A2ATS_ERR_DTYPE;
    int st = check_shape(B, H, Ncap, d);
    if (st) return st;
    if ((sub_dim != 8 && sub_dim != 16) || d % sub_dim != 0) return A2ATS_ERR_SHAPE;
    if (K < 1 || K * sub_dim > subvector_table_limit()) return A2ATS_ERR_SHAPE;
    if ((perm == nullptr) != (count == nullptr)) return A2ATS_ERR_INVALID_ARG;
    if (B * H * Ncap == 0) return A2ATS_OK;
    if (!x || !codebook || !codes) return A2ATS_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(codebook) || !aligned16(codes) || (L && !aligned16(L)))
        return A2ATS_ERR_ALIGN;
    if (!workspace ||
        workspace_bytes < a2ats_subvector_assign_workspace_size(B, H, Ncap, d, sub_dim, K))
        return A2ATS_ERR_WORKSPACE;
    Carve c(workspace);
    float* Lc = c.take<float>((size_t)(H * sub_dim * sub_dim));
    float* Lt = c.take<float>((size_t)(H * sub_dim * sub_dim));
    float* plain = c.take<float>((size_t)(H * K * sub_dim));
    float* weighted = c.take<float>((size_t)(H * K * sub_dim));
    float* half_norm = c.take<float>((size_t)(H * K));
    uint8_t* mark = c.take<uint8_t>((size_t)(B * H * Ncap));
    cudaStream_t s = (cudaStream_t)stream;
    const Shape sh{B, H, Ncap, d};
    cudaError_t e = launch_codebook_transform(codebook, dtype, H, K, sub_dim, nullptr, nullptr,
                                              plain, half_norm, nullptr, s);
    if (e == cudaSuccess && L) {
        e = launch_factor_prep(L, H, sub_dim, Lc, Lt, s);
        if (e == cudaSuccess)
            e = launch_codebook_transform(codebook, dtype, H, K, sub_dim, Lc, nullptr, weighted,
                                          half_norm, nullptr, s);
        if (e == cudaSuccess && perm) e = launch_mark_retrieval(perm, count, len, sh, mark, s);
    }
    if (e == cudaSuccess)
        e = launch_subvector_assign(x, dtype, sh, len, sub_dim, plain, L ? weighted : nullptr,
                                    L ? Lc : nullptr, (L && perm) ? mark : nullptr, K, codes, s);
    return e == cudaSuccess ? A2ATS_OK : cuda_fail(e);
}

size_t a2ats_subvector_query_aware_assign_workspace_size(int64_t B, int64_t H, int64_t Ncap,
                                                         int64_t d, int64_t sub_dim, int64_t K) {
    (void)d;
    if (B < 0 || H < 0 || Ncap < 0 || sub_dim < 0 || K < 0) return 0;
    Carve c(nullptr);
    c.take<float>((size_t)(H * K * sub_dim));  // decoded table
    c.take<float>((size_t)(H * K));            // half norms (written, not read)
    c.take<float>((size_t)(H * K));            // |c_k|
    c.take<uint8_t>((size_t)(B * H * Ncap));   // retrieval marks
    return c.used + 256;
}

int a2ats_subvector_query_aware_assign(const void* x, int32_t dtype, int64_t B, int64_t H,
                                       int64_t Ncap, int64_t d, const int32_t* len,
                                       int64_t sub_dim, const void* codebook, int64_t K,
                                       const void* query, double beta, const int32_t* perm,
                                       const int32_t* count, int32_t* codes, void* workspace,
                                       size_t workspace_bytes, void* stream) {
    if (!dtype_ok(dtype)) return A2ATS_ERR_DTYPE;
    int st = check_shape(B, H, Ncap, d);
    if (st) return st;
    if ((sub_dim != 8 && sub_dim != 16) || d % sub_dim != 0) return A2ATS_ERR_SHAPE;
    if (K < 1 || K * sub_dim > subvector_table_limit()) return A2ATS_ERR_SHAPE;
    if (!unit_interval(beta)) return A2ATS_ERR_INVALID_ARG;
    if ((perm == nullptr) != (count == nullptr)) return A2ATS_ERR_INVALID_ARG;
    if (B * H * Ncap == 0) return A2ATS_OK;
    if (!x || !codebook || !codes) return A2ATS_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(codebook) || !aligned16(codes) ||
        (query && !aligned16(query)))
        return A2ATS_ERR_ALIGN;
    if (!workspace || workspace_bytes < a2ats_subvector_query_aware_assign_workspace_size(
                                            B, H, Ncap, d, sub_dim, K))
        return A2ATS_ERR_WORKSPACE;
    Carve c(workspace);
    float* table = c.take<float>((size_t)(H * K * sub_dim));
    float* half_norm = c.take<float>((size_t)(H * K));
    float* cnorm = c.take<float>((size_t)(H * K));
    uint8_t* mark = c.take<uint8_t>((size_t)(B * H * Ncap));
    cudaStream_t s = (cudaStream_t)stream;
    const Shape sh{B, H, Ncap, d};
    cudaError_t e = launch_codebook_transform(codebook, dtype, H, K, sub_dim, nullptr, nullptr,
                                              table, half_norm, nullptr, s);
    if (e == cudaSuccess) e = launch_centroid_norms(codebook, dtype, H, K, sub_dim, cnorm, s);
    if (e == cudaSuccess && perm) e = launch_mark_retrieval(perm, count, len, sh, mark, s);
    if (e == cudaSuccess)
        e = launch_subvector_blend(x, dtype, sh, len, sub_dim, table, cnorm, query, (float)beta,
                                   perm ? mark : nullptr, K, codes, s);
    return e == cudaSuccess ? A2ATS_OK : cuda_fail(e);
}

}  // extern "C"
