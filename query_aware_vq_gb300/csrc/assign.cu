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
    float* cosc = qs + d;           // [kCT] cos(query, c_j) of the tile's centroids
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
            if (pass == 1) {
                // the cosine term depends on the centroid only (one query per
                // (b, h)): kSlots threads per centroid, compensated sums
                const int cc_i = threadIdx.x / kSlots, part = threadIdx.x % kSlots;
                Dot2 dq;
                if (cc_i < nc)
                    for (int aa = part; aa < d; aa += kSlots) dq.add_prod(qs[aa], cs[cc_i * ld + aa]);
                for (int m = kSlots / 2; m; m >>= 1) dq.merge(shfl_xor(dq, m));
                if (part == 0 && cc_i < nc) {
                    const float cn = cnorm[h * K + j0 + cc_i];
                    cosc[cc_i] = (qn > 0.f && cn > 0.f) ? dq.value() / (qn * cn) : 0.f;
                }
                __syncthreads();
            }
            // rows of the list that are empty do no work
            for (int c = slot; c < nc && rows[r] >= 0; c += kSlots) {
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
                const int32_t j = (int32_t)(j0 + c);
                const float cosv = cosc[c];
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
// The cosine blend of the decode row alone (rows = LAST): one block per
// (b, h) and one row, so the block's lanes spread over the centroids instead
// of over rows.  8 lanes share a centroid (each 1/8 of its elements, 16-byte
// loads); pass 1 finds e_max = max_j |x - c_j|^2, pass 2 scores every
// centroid.  With K <= kLastCache pass 1 also keeps e_j and q . c_j in
// shared memory and pass 2 reads them back instead of the codebook.  The
// arithmetic is the general kernel's: e_j as a plain fp32 sum of squares,
// q . c_j compensated.
constexpr int64_t kLastCache = 8192;
template <int DT>
__global__ void __launch_bounds__(256)
assign_blend_last_kernel(const void* __restrict__ x, const float* __restrict__ cf, int32_t H,
                         int32_t ncap, int32_t d, const int32_t* __restrict__ len,
                         const RopeArgs ra, const float* __restrict__ q,
                         const float* __restrict__ qnorm, float beta, int64_t K,
                         const float* __restrict__ cnorm, int32_t* __restrict__ codes) {
    __shared__ __align__(16) float xs[kMaxD];
    __shared__ __align__(16) float qs[kMaxD];
    __shared__ float wmax[8];
    __shared__ float wbest[8];
    __shared__ int32_t wj[8];
    extern __shared__ float ecache[];  // [2][K]: e_j, then q . c_j (K <= kLastCache)
    const bool cached = K <= kLastCache;
    const int64_t bh = blockIdx.x;
    const int64_t h = bh % H;
    const int32_t Ls = seq_len(len, (int32_t)(bh / H), ncap);
    if (Ls <= 0) return;
    // the row with its windowed RoPE, and the query
    for (int a = threadIdx.x; a < d; a += blockDim.x) xs[a] = load1<DT>(x, (bh * ncap + Ls - 1) * d + a);
    for (int a = threadIdx.x; a < d; a += blockDim.x) qs[a] = q[bh * d + a];
    __syncthreads();
    if (ra.enabled) {
        const int half = d / 2;
        const int32_t pos = rope_position(Ls - 1, Ls - 1, ra);
        if (pos != 0)
            for (int i = threadIdx.x; i < half; i += blockDim.x) {
                float sn, cs;
                rope_angle(pos, ra.omega_hi[i], ra.omega_lo[i], ra, sn, cs);
                const int a = ra.interleaved ? 2 * i : i;
                const int b = ra.interleaved ? 2 * i + 1 : i + half;
                const float xa = xs[a], xb = xs[b];
                xs[a] = fmaf(xa, cs, -__fmul_rn(xb, sn));
                xs[b] = fmaf(xa, sn, __fmul_rn(xb, cs));
            }
        __syncthreads();
    }
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int grp = threadIdx.x >> 3, seg = threadIdx.x & 7;  // 32 centroids at a time
    const float qn = qnorm[bh];
    const float* ch = cf + h * K * d;
    float emax = 0.f, best = -INFINITY;
    int32_t bj = 0;
    for (int pass = 0; pass < 2; pass++) {
        if (pass == 1 && cached) {
            // scores from the values pass 1 kept; each thread takes j = t,
            // t + 256, ... in ascending order
            for (int64_t j = threadIdx.x; j < K; j += blockDim.x) {
                const float e = ecache[j], dqv = ecache[K + j];
                const float cn = cnorm[h * K + j];
                const float cosv = (qn > 0.f && cn > 0.f) ? dqv / (qn * cn) : 0.f;
                const float err = emax > 0.f ? e / emax : 0.f;
                const float sc = fmaf(-beta, err, (1.f - beta) * cosv);
                if (sc > best || (sc == best && j < bj)) { best = sc; bj = (int32_t)j; }
            }
            break;
        }
        // uniform trip count: the shuffles below need every lane
        for (int64_t j0 = 0; j0 < K; j0 += 32) {
            const int64_t j = j0 + grp;
            const bool ok = j < K;
            const float* c = ch + (ok ? j : 0) * d;
            float e0 = 0.f, e1 = 0.f;
            Dot2 dq;
            for (int a = seg * 4; a < d; a += 32) {
                const float4 cv = *reinterpret_cast<const float4*>(c + a);
                const float4 xv = *reinterpret_cast<const float4*>(xs + a);
                const float t0 = xv.x - cv.x, t1 = xv.y - cv.y, t2 = xv.z - cv.z, t3 = xv.w - cv.w;
                e0 = fmaf(t0, t0, e0);
                e1 = fmaf(t1, t1, e1);
                e0 = fmaf(t2, t2, e0);
                e1 = fmaf(t3, t3, e1);
                if (pass == 1 || cached) {
                    const float4 qv = *reinterpret_cast<const float4*>(qs + a);
                    dq.add_prod(qv.x, cv.x);
                    dq.add_prod(qv.y, cv.y);
                    dq.add_prod(qv.z, cv.z);
                    dq.add_prod(qv.w, cv.w);
                }
            }
            float e = e0 + e1;
            for (int m = 4; m; m >>= 1) e += __shfl_xor_sync(0xffffffffu, e, m);
            if (pass == 0) {
                if (cached) {
                    for (int m = 4; m; m >>= 1) dq.merge(shfl_xor(dq, m));
                    if (ok && seg == 0) {
                        ecache[j] = e;
                        ecache[K + j] = dq.value();
                    }
                }
                if (ok) emax = fmaxf(emax, e);
                continue;
            }
            for (int m = 4; m; m >>= 1) dq.merge(shfl_xor(dq, m));
            if (ok) {
                const float cn = cnorm[h * K + j];
                const float cosv = (qn > 0.f && cn > 0.f) ? dq.value() / (qn * cn) : 0.f;
                const float err = emax > 0.f ? e / emax : 0.f;
                const float sc = fmaf(-beta, err, (1.f - beta) * cosv);
                if (sc > best || (sc == best && j < bj)) { best = sc; bj = (int32_t)j; }
            }
        }
        if (pass == 0) {
            // e_max over the block
            for (int m = 16; m; m >>= 1) emax = fmaxf(emax, __shfl_xor_sync(0xffffffffu, emax, m));
            if (lane == 0) wmax[w] = emax;
            __syncthreads();
            emax = wmax[0];
            for (int ww = 1; ww < 8; ww++) emax = fmaxf(emax, wmax[ww]);
        }
    }
    for (int m = 16; m; m >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, best, m);
        const int32_t oj = __shfl_xor_sync(0xffffffffu, bj, m);
        if (ov > best || (ov == best && oj < bj)) { best = ov; bj = oj; }
    }
    if (lane == 0) { wbest[w] = best; wj[w] = bj; }
    __syncthreads();
    if (threadIdx.x == 0) {
        for (int ww = 1; ww < 8; ww++)
            if (wbest[ww] > best || (wbest[ww] == best && wj[ww] < bj)) { best = wbest[ww]; bj = wj[ww]; }
        codes[bh * ncap + Ls - 1] = bj;
    }
}

size_t blend_smem(int d) { return sizeof(float) * (size_t)((kRB + kCT) * (d + 1) + d + kCT); }

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
    if (sel.mode == 3) {
        // one row per (b, h): the lanes go to the centroids
        const float* cf = reinterpret_cast<const float*>(c);
        const unsigned nbh = (unsigned)(s.B * s.H);
        const size_t smem = K <= kLastCache ? sizeof(float) * 2 * (size_t)K : 0;
        auto k = dt == kF32 ? assign_blend_last_kernel<kF32>
                            : (dt == kBF16 ? assign_blend_last_kernel<kBF16>
                                           : assign_blend_last_kernel<kF16>);
        cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)(sizeof(float) * 2 * kLastCache));
        if (e != cudaSuccess) return e;
        k<<<nbh, 256, smem, st>>>(x, cf, (int32_t)s.H, (int32_t)s.Ncap, (int32_t)s.d, len, ra, q,
                                  qnorm, beta, K, cnorm, codes);
        note_launches(1);
        return cudaGetLastError();
    }
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
