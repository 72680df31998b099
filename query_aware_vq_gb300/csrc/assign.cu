// assign.cu -- codebook assignment on the CUDA cores.
//
// API page, a2ats_h_weighted_assignment (paper Eq. 14, computed through the
// Eq. 15-18 Cholesky identity: argmin_j |kL - c_jL|^2) and
// a2ats_query_aware_assignment (the cosine blend).  These kernels evaluate the
// distances directly in z = kL space in fp32: they are the exact path for
// rows the tensor-core contraction cannot decide (near ties) and for shapes it
// does not cover.
#include "kernels.cuh"

namespace a2ats {
namespace {

constexpr int kRB = 32;       // rows per block
constexpr int kCT = 32;       // centroids per shared-memory tile
constexpr int kSlots = 8;     // threads per row
constexpr int kAThreads = kRB * kSlots;

// Row r of the (b, h) row list: its index within the sequence, or -1.
// Entries of a caller's perm outside [0, L) are skipped, never dereferenced.
__device__ __forceinline__ int32_t list_row(const RowSel& sel, int64_t bh, int32_t ncap, int32_t L,
                                            int32_t r) {
    if (sel.mode == 0) return r < L ? r : -1;
    if (sel.mode == 3) return (r == 0 && L > 0) ? L - 1 : -1;
    const int32_t cnt = min(max(sel.count[bh], 0), L);
    int32_t j = -1;
    if (sel.mode == 1) j = r < cnt ? sel.perm[bh * ncap + r] : -1;
    else j = r < L - cnt ? sel.perm[bh * ncap + cnt + r] : -1;
    return (j >= 0 && j < L) ? j : -1;
}

// Load kRB rows of the list into shared memory as fp32, with the windowed
// RoPE applied when enabled.
template <int DT>
__device__ void load_rows(const void* x, int64_t bh, int32_t ncap, int32_t d, int32_t L,
                          const RopeArgs& ra, const int32_t* rows, float* xs, int ld) {
    for (int e = threadIdx.x; e < kRB * d; e += blockDim.x) {
        const int r = e / d, a = e % d;
        xs[r * ld + a] = rows[r] >= 0 ? load1<DT>(x, (bh * ncap + rows[r]) * d + a) : 0.f;
    }
    __syncthreads();
    if (ra.enabled) {
        const int half = d / 2;
        for (int e = threadIdx.x; e < kRB * half; e += blockDim.x) {
            const int r = e / half, i = e % half;
            if (rows[r] < 0) continue;
            const int32_t pos = rope_position(rows[r], L - 1, ra);
            if (pos == 0) continue;
            float s, c;
            rope_angle(pos, ra.omega_hi[i], ra.omega_lo[i], ra, s, c);
            const int a = ra.interleaved ? 2 * i : i;
            const int b = ra.interleaved ? 2 * i + 1 : i + half;
            const float xa = xs[r * ld + a], xb = xs[r * ld + b];
            xs[r * ld + a] = fmaf(xa, c, -__fmul_rn(xb, s));
            xs[r * ld + b] = fmaf(xa, s, __fmul_rn(xb, c));
        }
        __syncthreads();
    }
}

// Better candidate in (distance, index) order: smaller distance, then lower index.
__device__ __forceinline__ bool better_min(float v, int32_t j, float bv, int32_t bj) {
    return v < bv || (v == bv && j < bj);
}

template <int DT>
__global__ void __launch_bounds__(kAThreads)
assign_exact_kernel(const void* __restrict__ x, int32_t H, int32_t ncap, int32_t d,
                    const int32_t* __restrict__ len, const RopeArgs ra, const RowSel sel,
                    const float* __restrict__ L, const float* __restrict__ cp,
                    const float* __restrict__ half_norm, int64_t K, int32_t* __restrict__ codes) {
    extern __shared__ float sm[];
    const int ld = d + 1;
    float* xs = sm;                 // [kRB][d+1] rows (then z)
    float* zs = xs + kRB * ld;      // [kRB][d+1] z = x L
    float* cs = zs + kRB * ld;      // [kCT][d+1] centroid tile
    __shared__ int32_t rows[kRB];
    const int64_t bh = blockIdx.y;
    const int32_t Ls = seq_len(len, (int32_t)(bh / H), ncap);
    const int32_t r0 = blockIdx.x * kRB;
    bool any = false;
    if (threadIdx.x < kRB) {
        rows[threadIdx.x] = list_row(sel, bh, ncap, Ls, r0 + threadIdx.x);
        any = rows[threadIdx.x] >= 0;
    }
    if (!__syncthreads_or(any)) return;  // this slice of the row list is empty
    load_rows<DT>(x, bh, ncap, d, Ls, ra, rows, xs, ld);
    const float* Z = xs;
    if (L) {
        const float* Lh = L + bh % H * (int64_t)d * d;
        for (int e = threadIdx.x; e < kRB * d; e += blockDim.x) {
            const int r = e / d, b = e % d;
            Dot2 acc;
            for (int a = 0; a < d; a++) acc.add_prod(xs[r * ld + a], Lh[(int64_t)a * d + b]);
            zs[r * ld + b] = acc.value();
        }
        __syncthreads();
        Z = zs;
    }
    const int r = threadIdx.x / kSlots, slot = threadIdx.x % kSlots;
    const float* zr = Z + r * ld;
    float best = INFINITY;
    int32_t bj = 0;
    const int64_t h = bh % H;
    for (int64_t j0 = 0; j0 < K; j0 += kCT) {
        const int nc = (int)(K - j0 < (int64_t)(kCT) ? K - j0 : (int64_t)(kCT));
        for (int e = threadIdx.x; e < kCT * d; e += blockDim.x) {
            const int c = e / d, a = e % d;
            cs[c * ld + a] = c < nc ? cp[((h * K) + j0 + c) * d + a] : 0.f;
        }
        __syncthreads();
        for (int c = slot; c < nc; c += kSlots) {
            const float* cc = cs + c * ld;
            float acc[4] = {0.f, 0.f, 0.f, 0.f};
            int a = 0;
            for (; a + 4 <= d; a += 4) {
#pragma unroll
                for (int u = 0; u < 4; u++) {
                    const float t = zr[a + u] - cc[a + u];
                    acc[u] = fmaf(t, t, acc[u]);
                }
            }
            for (; a < d; a++) {
                const float t = zr[a] - cc[a];
                acc[0] = fmaf(t, t, acc[0]);
            }
            const float v = (acc[0] + acc[1]) + (acc[2] + acc[3]);
            const int32_t j = (int32_t)(j0 + c);
            if (better_min(v, j, best, bj)) { best = v; bj = j; }
        }
        __syncthreads();
    }
    for (int m = kSlots / 2; m; m >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, best, m);
        const int32_t oj = __shfl_xor_sync(0xffffffffu, bj, m);
        if (better_min(ov, oj, best, bj)) { best = ov; bj = oj; }
    }
    if (slot == 0 && rows[r] >= 0) codes[bh * ncap + rows[r]] = bj;
    (void)half_norm;
}

// Cosine blend: e_j = |x - c_j|^2, m = max_j e_j,
// s_j = -beta e_j / m + (1 - beta) cos(q, c_j); argmax (lowest j on ties).
template <int DT>
__global__ void __launch_bounds__(kAThreads)
assign_blend_kernel(const void* __restrict__ x, const float* __restrict__ cf, int32_t H,
                    int32_t ncap, int32_t d, const int32_t* __restrict__ len, const RopeArgs ra,
                    const RowSel sel, const float* __restrict__ q, const float* __restrict__ qnorm,
                    float beta, int64_t K, const float* __restrict__ cnorm,
                    int32_t* __restrict__ codes) {
    extern __shared__ float sm[];
    const int ld = d + 1;
    float* xs = sm;                 // [kRB][d+1]
    float* cs = xs + kRB * ld;      // [kCT][d+1]
    float* qs = cs + kCT * ld;      // [d] shared query
    __shared__ int32_t rows[kRB];
    const int64_t bh = blockIdx.y;
    const int64_t h = bh % H;
    const int32_t Ls = seq_len(len, (int32_t)(bh / H), ncap);
    const int32_t r0 = blockIdx.x * kRB;
    bool any = false;
    if (threadIdx.x < kRB) {
        rows[threadIdx.x] = list_row(sel, bh, ncap, Ls, r0 + threadIdx.x);
        any = rows[threadIdx.x] >= 0;
    }
    if (!__syncthreads_or(any)) return;
    load_rows<DT>(x, bh, ncap, d, Ls, ra, rows, xs, ld);
    for (int a = threadIdx.x; a < d; a += blockDim.x) qs[a] = q[bh * d + a];
    const int r = threadIdx.x / kSlots, slot = threadIdx.x % kSlots;
    const float* xr = xs + r * ld;
    const float qn = qnorm[bh];
    __syncthreads();
    const float* qv = qs;
    float emax = 0.f;
    float best = -INFINITY;
    int32_t bj = 0;
    for (int pass = 0; pass < 2; pass++) {
        if (pass == 1) {
            for (int m = kSlots / 2; m; m >>= 1)
                emax = fmaxf(emax, __shfl_xor_sync(0xffffffffu, emax, m));
        }
        for (int64_t j0 = 0; j0 < K; j0 += kCT) {
            const int nc = (int)(K - j0 < (int64_t)(kCT) ? K - j0 : (int64_t)(kCT));
            for (int e = threadIdx.x; e < kCT * d; e += blockDim.x) {
                const int c = e / d, a = e % d;
                cs[c * ld + a] = c < nc ? cf[((h * K) + j0 + c) * d + a] : 0.f;
            }
            __syncthreads();
            for (int c = slot; c < nc; c += kSlots) {
                const float* cc = cs + c * ld;
                float e4[4] = {0.f, 0.f, 0.f, 0.f}, dq = 0.f;
                int a = 0;
                for (; a + 4 <= d; a += 4) {
#pragma unroll
                    for (int u = 0; u < 4; u++) {
                        const float t = xr[a + u] - cc[a + u];
                        e4[u] = fmaf(t, t, e4[u]);
                    }
                }
                for (; a < d; a++) {
                    const float t = xr[a] - cc[a];
                    e4[0] = fmaf(t, t, e4[0]);
                }
                const float e = (e4[0] + e4[1]) + (e4[2] + e4[3]);
                if (pass == 0) {
                    emax = fmaxf(emax, e);
                    continue;
                }
                Dot2 dot;
                for (int aa = 0; aa < d; aa++) dot.add_prod(qv[aa], cc[aa]);
                const int32_t j = (int32_t)(j0 + c);
                const float cn = cnorm[h * K + j];
                const float cosv = (qn > 0.f && cn > 0.f) ? dot.value() / (qn * cn) : 0.f;
                const float err = emax > 0.f ? e / emax : 0.f;
                const float s = fmaf(-beta, err, (1.f - beta) * cosv);
                if (s > best || (s == best && j < bj)) { best = s; bj = j; }
            }
            __syncthreads();
        }
    }
    for (int m = kSlots / 2; m; m >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, best, m);
        const int32_t oj = __shfl_xor_sync(0xffffffffu, bj, m);
        if (ov > best || (ov == best && oj < bj)) { best = ov; bj = oj; }
    }
    if (slot == 0 && rows[r] >= 0) codes[bh * ncap + rows[r]] = bj;
}

size_t exact_smem(int d) { return sizeof(float) * (size_t)((2 * kRB + kCT) * (d + 1)); }
size_t blend_smem(int d) { return sizeof(float) * (size_t)((kRB + kCT) * (d + 1) + d); }

}  // namespace

cudaError_t launch_assign_exact(const void* x, int dt, const Shape& s, const int32_t* len,
                                const RopeArgs& ra, const RowSel& sel, const float* L,
                                const float* cp, const float* half_norm, int64_t K,
                                int32_t* codes, cudaStream_t st) {
    if (s.B * s.H * s.Ncap == 0) return cudaSuccess;
    // the decode-row selection has one row per (b, h)
    dim3 grid(sel.mode == 3 ? 1u : (unsigned)((s.Ncap + kRB - 1) / kRB), (unsigned)(s.B * s.H));
    const size_t smem = exact_smem((int)s.d);
    cudaError_t e = cudaSuccess;
#define A2ATS_LAUNCH_EXACT(DTV)                                                               \
    e = cudaFuncSetAttribute(assign_exact_kernel<DTV>,                                        \
                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);         \
    if (e != cudaSuccess) return e;                                                           \
    assign_exact_kernel<DTV><<<grid, kAThreads, smem, st>>>(x, (int32_t)s.H, (int32_t)s.Ncap, \
                                                            (int32_t)s.d, len, ra, sel, L,    \
                                                            cp, half_norm, K, codes); \
    note_launches(1);
    switch (dt) {
        case kF32: A2ATS_LAUNCH_EXACT(kF32) break;
        case kBF16: A2ATS_LAUNCH_EXACT(kBF16) break;
        default: A2ATS_LAUNCH_EXACT(kF16)
    }
#undef A2ATS_LAUNCH_EXACT
    return cudaGetLastError();
}

cudaError_t launch_assign_blend(const void* x, const void* c, int dt, const Shape& s,
                                const int32_t* len, const RopeArgs& ra, const RowSel& sel,
                                const float* q, const float* qnorm, float beta, int64_t K,
                                const float* cnorm, int32_t* codes, cudaStream_t st) {
    if (s.B * s.H * s.Ncap == 0) return cudaSuccess;
    dim3 grid(sel.mode == 3 ? 1u : (unsigned)((s.Ncap + kRB - 1) / kRB), (unsigned)(s.B * s.H));
    const size_t smem = blend_smem((int)s.d);
    const float* cf = reinterpret_cast<const float*>(c);  // fp32 copy of the codebook
    cudaError_t e = cudaSuccess;
#define A2ATS_LAUNCH_BLEND(DTV)                                                               \
    e = cudaFuncSetAttribute(assign_blend_kernel<DTV>,                                        \
                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);         \
    if (e != cudaSuccess) return e;                                                           \
    assign_blend_kernel<DTV><<<grid, kAThreads, smem, st>>>(x, cf, (int32_t)s.H,              \
                                                            (int32_t)s.Ncap, (int32_t)s.d,    \
                                                            len, ra, sel, q, qnorm, beta, K,  \
                                                            cnorm, codes);            \
    note_launches(1);
    switch (dt) {
        case kF32: A2ATS_LAUNCH_BLEND(kF32) break;
        case kBF16: A2ATS_LAUNCH_BLEND(kBF16) break;
        default: A2ATS_LAUNCH_BLEND(kF16)
    }
#undef A2ATS_LAUNCH_BLEND
    return cudaGetLastError();
}

}  // namespace a2ats
