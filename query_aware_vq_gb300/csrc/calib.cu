// calib.cu -- query second moment, Cholesky factor, codebook transform.
//
// API page "veloxquant_mlx.quantizers.a2ats module":
//   a2ats_query_second_moment  H = E[q^T q] + ridge I        (paper Eq. 10)
//   a2ats_cholesky_factor      H = L L^T                     (paper Eq. 15)
//   a2ats_h_weighted_assignment, Eq. 16-18: centroids are mapped once into the
//   space z = kL (c' = cL, |c'|^2) so the assignment is a Euclidean argmin.
//
// GB300 executes fp64 at a small fraction of its fp32 rate, so the extra
// precision these small, latency-bound kernels need comes from compensated
// fp32 (TwoSum / TwoProduct) rather than from doubles.
#include "kernels.cuh"

namespace a2ats {
namespace {

// ----------------------------------------------------- second moment --
constexpr int kSmTile = 64;    // output tile edge
constexpr int kSmChunk = 32;   // query rows per plain-fp32 partial sum
constexpr int kSmThreads = 256;

// Partial second moment of one 64x64 tile of H over one slice of the M
// queries.  Each thread owns a 4x4 block of outputs fed by 16-byte shared
// memory reads; 32-row plain fp32 partials are folded into compensated
// accumulators, so the result is within a few units of fp32 rounding of the
// exact slice sum.
template <int DT>
__global__ void __launch_bounds__(kSmThreads)
second_moment_partial_kernel(const void* __restrict__ q, int64_t M, int32_t d, int64_t splits,
                             float* __restrict__ partial) {
    using T = typename Elem<DT>::T;
    constexpr int VE = 16 / (int)sizeof(T);                   // elements per 16-byte vector
    constexpr int VPR = kSmTile / VE;                         // vectors per 64-column row
    constexpr int NV = 2 * kSmChunk * VPR / kSmThreads;       // vectors per thread per chunk
    __shared__ __align__(16) float qa[kSmChunk][kSmTile];
    __shared__ __align__(16) float qb[kSmChunk][kSmTile];
    // decode the lower-triangular tile pair (ti >= tj) from blockIdx.x
    int ti = 0, rem = blockIdx.x;
    while (rem > ti) { rem -= ti + 1; ti++; }
    const int tj = rem;
    const int split = blockIdx.y;
    const int h = blockIdx.z;
    const int64_t m0 = M * split / splits, m1 = M * (split + 1) / splits;
    const int tid = threadIdx.x;
    const int ty = tid >> 4, tx = tid & 15;   // 4x4 block (rows ty*4.., cols tx*4..)
    float p[4][4];
    Dot2 acc[4][4];
    const T* qh = reinterpret_cast<const T*>(q) + (int64_t)h * M * d;
    uint4 buf[NV];
    // 16-byte loads of one chunk into registers (zeros past M or d)
    auto fetch = [&](int64_t mc) {
#pragma unroll
        for (int v = 0; v < NV; v++) {
            const int e = tid + v * kSmThreads;
            const int tile = e / (kSmChunk * VPR), r = (e / VPR) % kSmChunk, cv = e % VPR;
            const int col = (tile ? tj : ti) * kSmTile + cv * VE;
            buf[v] = make_uint4(0, 0, 0, 0);
            if (mc + r < m1 && col < d)
                buf[v] = __ldg(reinterpret_cast<const uint4*>(qh + (mc + r) * d + col));
        }
    };
    auto stage = [&]() {
#pragma unroll
        for (int v = 0; v < NV; v++) {
            const int e = tid + v * kSmThreads;
            const int tile = e / (kSmChunk * VPR), r = (e / VPR) % kSmChunk, cv = e % VPR;
            const T* el = reinterpret_cast<const T*>(&buf[v]);
            float* dst = tile ? &qb[r][cv * VE] : &qa[r][cv * VE];
#pragma unroll
            for (int u = 0; u < VE; u++) dst[u] = to_f32<DT>(el[u]);
        }
    };
    if (m0 < m1) fetch(m0);
    for (int64_t mc = m0; mc < m1; mc += kSmChunk) {
        const int rows = (int)(m1 - mc < kSmChunk ? m1 - mc : kSmChunk);
        stage();
        __syncthreads();
        if (mc + kSmChunk < m1) fetch(mc + kSmChunk);  // overlaps the arithmetic below
#pragma unroll
        for (int i = 0; i < 4; i++)
#pragma unroll
            for (int j = 0; j < 4; j++) p[i][j] = 0.f;
        for (int r = 0; r < rows; r++) {
            const float4 a4 = *reinterpret_cast<const float4*>(&qa[r][ty * 4]);
            const float4 b4 = *reinterpret_cast<const float4*>(&qb[r][tx * 4]);
            const float av[4] = {a4.x, a4.y, a4.z, a4.w};
            const float bv[4] = {b4.x, b4.y, b4.z, b4.w};
#pragma unroll
            for (int i = 0; i < 4; i++)
#pragma unroll
                for (int j = 0; j < 4; j++) p[i][j] = fmaf(av[i], bv[j], p[i][j]);
        }
#pragma unroll
        for (int i = 0; i < 4; i++)
#pragma unroll
            for (int j = 0; j < 4; j++) acc[i][j].add(p[i][j]);
        __syncthreads();
    }
    float* out = partial + ((int64_t)split * gridDim.z + h) * d * d;
    const int64_t plane = (int64_t)splits * gridDim.z * d * d;
#pragma unroll
    for (int i = 0; i < 4; i++)
#pragma unroll
        for (int j = 0; j < 4; j++) {
            const int a = ti * kSmTile + ty * 4 + i, b = tj * kSmTile + tx * 4 + j;
            if (a >= d || b >= d) continue;
            // hi and lo in two planes so the final sum stays compensated
            const int64_t idx = (int64_t)a * d + b;
            out[idx] = acc[i][j].s;
            out[idx + plane] = acc[i][j].c;
        }
}

// H[h][a][b] = H[h][b][a] = (sum over slices) / M + ridge [a == b], a >= b.
__global__ void second_moment_reduce_kernel(const float* __restrict__ partial, int64_t H,
                                            int64_t M, int32_t d, int64_t splits, float ridge,
                                            float* __restrict__ h_out) {
    const int64_t n = H * d * d;
    const int64_t plane = splits * H * d * d;
    for (int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; idx < n;
         idx += (int64_t)gridDim.x * blockDim.x) {
        const int64_t h = idx / ((int64_t)d * d);
        const int a = (int)((idx / d) % d), b = (int)(idx % d);
        if (a < b) continue;
        Dot2 acc;
        for (int64_t s = 0; s < splits; s++) {
            const int64_t p = (s * H + h) * d * d + (int64_t)a * d + b;
            acc.add(partial[p]);
            acc.add(partial[p + plane]);
        }
        float v = __fdiv_rn(acc.value(), (float)M);
        if (a == b) v = __fadd_rn(v, ridge);
        h_out[(h * d + a) * d + b] = v;
        h_out[(h * d + b) * d + a] = v;
    }
}

// ----------------------------------------------------------- Cholesky --
constexpr int kCholThreads = 512;
constexpr int kPanel = 32;

__device__ __forceinline__ int tri(int i, int k) { return i * (i + 1) / 2 + k; }

// double-float helpers on (hi, lo) pairs
struct DF {
    float hi, lo;
};
__device__ __forceinline__ DF df_from(float hi, float lo) {
    float s, e;
    two_sum(hi, lo, s, e);
    return DF{s, e};
}
// a - b * c with b, c plain floats
__device__ __forceinline__ DF df_sub_prod(DF a, float b, float c) {
    const float p = __fmul_rn(b, c);
    const float pe = fmaf(b, c, -p);
    float s, e;
    two_sum(a.hi, -p, s, e);
    e = __fadd_rn(e, __fsub_rn(a.lo, pe));
    return df_from(s, e);
}
// a / b (b a plain positive float): q = rn(a/b), then one correction step
__device__ __forceinline__ float df_div(DF a, float b) {
    const float q = __fdiv_rn(a.hi, b);
    const float r = fmaf(-q, b, a.hi);  // exact remainder of a.hi - q b
    return __fadd_rn(q, __fdiv_rn(__fadd_rn(r, a.lo), b));
}
// sqrt of a positive double-float, rounded to float
__device__ __forceinline__ float df_sqrt(DF a) {
    const float s = sqrtf(a.hi);
    const float r = fmaf(-s, s, a.hi);  // exact a.hi - s^2
    return __fadd_rn(s, __fdiv_rn(__fadd_rn(r, a.lo), __fmul_rn(2.f, s)));
}

// One block per head; the factor lives packed in shared memory.  Columns are
// taken 32 at a time (left-looking, Crout order):
//   1. every entry of the panel, H_ij - sum_{k<j0} L_ik L_jk, with a
//      compensated dot product (all entries in parallel), kept as a
//      double-float in shared memory;
//   2. the panel is factored column by column, left-looking: each row's
//      entry loses its compensated dot with the panel columns already done,
//      then every row is scaled by the pivot (two barriers per column).
// Each entry of L is within about one fp32 rounding of the factor of the
// values it depends on; a non-positive pivot stops the head and is reported.
constexpr int kPS = kPanel + 1;  // padded panel row stride (float2), conflict-free

__global__ void __launch_bounds__(kCholThreads)
cholesky_kernel(const float* __restrict__ hm, int32_t d, float* __restrict__ l_out,
                int32_t* __restrict__ info) {
    extern __shared__ float smem[];
    float* Lp = smem;                                     // d(d+1)/2 packed factor
    float2* panel = reinterpret_cast<float2*>(smem + ((d * (d + 1) / 2 + 1) & ~1));  // [d][kPS]
    const int h = blockIdx.x;
    const float* Hh = hm + (int64_t)h * d * d;
    const int tid = threadIdx.x;
    int failed = 0;
    for (int j0 = 0; j0 < d && !failed; j0 += kPanel) {
        const int pw = min(kPanel, d - j0);
        const int rows = d - j0;
        // 1. panel entries from the columns already factored
        for (int e = tid; e < rows * pw; e += blockDim.x) {
            const int ii = e / pw, jj = e % pw;
            if (jj > ii) continue;
            const int i = j0 + ii, j = j0 + jj;
            Dot2 acc;
            const float* Li = Lp + tri(i, 0);
            const float* Lj = Lp + tri(j, 0);
#pragma unroll 4
            for (int k = 0; k < j0; k++) acc.add_prod(Li[k], Lj[k]);
            acc.s = -acc.s;
            acc.c = -acc.c;
            acc.add(Hh[(int64_t)i * d + j]);
            const DF v = df_from(acc.s, acc.c);
            panel[ii * kPS + jj] = make_float2(v.hi, v.lo);
        }
        __syncthreads();
        // 2. factor the panel, left-looking: column jj of every row is its
        // panel entry minus the dot with the panel columns already done
        // (compensated), then scaled by the pivot every thread recomputes.
        for (int jj = 0; jj < pw; jj++) {
            const int ii = jj + tid;
            if (ii < rows) {
                const float2 pv = panel[ii * kPS + jj];
                Dot2 acc;
                acc.s = pv.x;
                acc.c = pv.y;
                const float* Li = Lp + tri(j0 + ii, j0);
                const float* Lj = Lp + tri(j0 + jj, j0);
                for (int kk = 0; kk < jj; kk++) acc.add_prod(-Li[kk], Lj[kk]);
                const DF v = df_from(acc.s, acc.c);
                panel[ii * kPS + jj] = make_float2(v.hi, v.lo);
            }
            __syncthreads();
            const float2 pvt = panel[jj * kPS + jj];
            if (!(pvt.x > 0.f)) {
                failed = j0 + jj + 1;
                break;
            }
            const float diag = df_sqrt(DF{pvt.x, pvt.y});
            if (ii < rows) {
                const float2 pv = panel[ii * kPS + jj];
                Lp[tri(j0 + ii, j0 + jj)] = (ii == jj) ? diag : df_div(DF{pv.x, pv.y}, diag);
            }
            __syncthreads();
        }
    }
    float* Lh = l_out + (int64_t)h * d * d;
    for (int e = tid; e < d * d; e += blockDim.x) {
        const int i = e / d, k = e % d;
        float v = 0.f;
        if (k <= i && (!failed || k < failed - 1)) v = Lp[tri(i, k)];
        Lh[e] = v;
    }
    if (tid == 0) info[h] = failed;
}

// ------------------------------------------------ codebook transform --
constexpr int kCtCent = 16;  // centroids per block (8 packed pairs)
constexpr int kCtVs = 20;    // row stride of the operand rows (float4-aligned, fewer conflicts)

__device__ __forceinline__ float2 neg2(float2 v) { return make_float2(-v.x, -v.y); }

// Dot2 on two independent sums at once (packed fp32 instructions).
struct Dot2x2 {
    float2 s = {0.f, 0.f}, c = {0.f, 0.f};
    __device__ __forceinline__ void add_prod(float2 a, float2 b) {
        const float2 p = __fmul2_rn(a, b);
        const float2 pe = __ffma2_rn(a, b, neg2(p));
        const float2 t = __fadd2_rn(s, p);
        const float2 bp = __fadd2_rn(t, neg2(s));
        const float2 te = __fadd2_rn(__fadd2_rn(s, neg2(__fadd2_rn(t, neg2(bp)))),
                                     __fadd2_rn(p, neg2(bp)));
        s = t;
        c = __fadd2_rn(c, __fadd2_rn(pe, te));
    }
    __device__ __forceinline__ float2 value() const { return __fadd2_rn(s, c); }
};

// cp[h][j] = c[h][j] Lc[h] and half_norm[h][j] = |cp[h][j]|^2 / 2, and when
// chat is given chat[h][j] = cp[h][j] Lc[h]^T, all compensated (Dot2).  Lc is
// lower triangular (zeros above the diagonal) and Lt its transpose, so output
// column b of c Lc sums rows a >= b only, and column a of cp Lc^T rows b <= a:
// each warp starts or stops at the first or last row its 32 columns need.
// Without Lc, cp is the decoded codebook.  A block holds 16 centroids and
// 2 x dr threads (dr = d rounded up to 32): thread (half, b) owns output
// column b of centroids 8 half .. 8 half + 7, as four packed pairs.  The
// factor is read straight from L1/L2 (no barriers in the loops); the
// centroid rows sit in shared memory.
template <int DT>
__global__ void __launch_bounds__(2 * kMaxD)
codebook_transform_kernel(const void* __restrict__ c, int64_t K, int32_t d,
                          const float* __restrict__ Lc, const float* __restrict__ Lt,
                          float* __restrict__ cp, float* __restrict__ half_norm,
                          float* __restrict__ chat) {
    __shared__ __align__(16) float vs[kMaxD][kCtVs];  // operand rows (c, then cp)
    __shared__ Dot2 red[kCtCent][2 * kMaxD / 32];
    const int h = blockIdx.y;
    const int64_t j0 = (int64_t)blockIdx.x * kCtCent;
    const int dr = (d + 31) / 32 * 32;
    const int t = threadIdx.x, half = t >= dr ? 1 : 0, b = t - half * dr;
    const int lane = t & 31, w = t >> 5;
    const int wcol = b & ~31;      // first column of this warp
    const int kb = half * (kCtCent / 2);
    const int nc = (int)(K - j0 < (int64_t)(kCtCent) ? K - j0 : (int64_t)(kCtCent));
    const bool col = b < d;
    for (int i = t; i < d * kCtCent; i += blockDim.x) {
        const int k = i / d, a = i - k * d;
        vs[a][k] = k < nc ? load1<DT>(c, ((int64_t)h * K + j0 + k) * d + a) : 0.f;
    }
    __syncthreads();
    float out[kCtCent / 2];
    if (Lc) {
        Dot2x2 acc[kCtCent / 4];
        if (col) {
            const float* Lb = Lc + (int64_t)h * d * d + b;
            for (int a0 = wcol; a0 < d; a0 += 8) {  // d % 8 == 0
                float l[8];
#pragma unroll
                for (int u = 0; u < 8; u++) l[u] = __ldg(Lb + (int64_t)(a0 + u) * d);
#pragma unroll
                for (int u = 0; u < 8; u++) {
                    const float2 l2 = make_float2(l[u], l[u]);
                    const float4* v4 = reinterpret_cast<const float4*>(&vs[a0 + u][kb]);
                    const float4 v0 = v4[0], v1 = v4[1];
                    acc[0].add_prod(make_float2(v0.x, v0.y), l2);
                    acc[1].add_prod(make_float2(v0.z, v0.w), l2);
                    acc[2].add_prod(make_float2(v1.x, v1.y), l2);
                    acc[3].add_prod(make_float2(v1.z, v1.w), l2);
                }
            }
        }
#pragma unroll
        for (int k = 0; k < kCtCent / 4; k++) {
            const float2 v = acc[k].value();
            out[2 * k] = col ? v.x : 0.f;
            out[2 * k + 1] = col ? v.y : 0.f;
        }
    } else {
#pragma unroll
        for (int k = 0; k < kCtCent / 2; k++) out[k] = col ? vs[b][kb + k] : 0.f;
    }
#pragma unroll
    for (int k = 0; k < kCtCent / 2; k++) {
        if (kb + k < nc && col) cp[((int64_t)h * K + j0 + kb + k) * d + b] = out[k];
        Dot2 n;
        n.add_prod(out[k], out[k]);
        for (int m = 16; m; m >>= 1) n.merge(shfl_xor(n, m));
        if (lane == 0) red[kb + k][w - half * (dr >> 5)] = n;
    }
    __syncthreads();
    if (t < nc) {
        Dot2 s2 = red[t][0];
        for (int ww = 1; ww < (dr >> 5); ww++) s2.merge(red[t][ww]);
        half_norm[(int64_t)h * K + j0 + t] = 0.5f * s2.value();
    }
    if (!Lc || !chat) return;
    // second factor: the operand rows become cp (every read of c is done)
    if (col)
#pragma unroll
        for (int k = 0; k < kCtCent / 2; k++) vs[b][kb + k] = out[k];
    __syncthreads();
    Dot2x2 acc[kCtCent / 4];
    if (col) {
        const float* Tb = Lt + (int64_t)h * d * d + b;
        const int aend = wcol + 32 < d ? wcol + 32 : d;
        for (int a0 = 0; a0 < aend; a0 += 8) {
            float l[8];
#pragma unroll
            for (int u = 0; u < 8; u++) l[u] = __ldg(Tb + (int64_t)(a0 + u) * d);
#pragma unroll
            for (int u = 0; u < 8; u++) {
                const float2 l2 = make_float2(l[u], l[u]);
                const float4* v4 = reinterpret_cast<const float4*>(&vs[a0 + u][kb]);
                const float4 v0 = v4[0], v1 = v4[1];
                acc[0].add_prod(make_float2(v0.x, v0.y), l2);
                acc[1].add_prod(make_float2(v0.z, v0.w), l2);
                acc[2].add_prod(make_float2(v1.x, v1.y), l2);
                acc[3].add_prod(make_float2(v1.z, v1.w), l2);
            }
        }
#pragma unroll
        for (int k = 0; k < kCtCent / 4; k++) {
            const float2 v = acc[k].value();
            if (kb + 2 * k < nc) chat[((int64_t)h * K + j0 + kb + 2 * k) * d + b] = v.x;
            if (kb + 2 * k + 1 < nc) chat[((int64_t)h * K + j0 + kb + 2 * k + 1) * d + b] = v.y;
        }
    }
}

// Lc = the lower triangle of L with zeros above the diagonal, Lt = Lc^T.
__global__ void factor_prep_kernel(const float* __restrict__ L, int64_t H, int32_t d,
                                   float* __restrict__ Lc, float* __restrict__ Lt) {
    const int64_t n = H * d * d;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t h = i / ((int64_t)d * d);
        const int a = (int)((i / d) % d), b = (int)(i % d);
        const float v = b <= a ? L[i] : 0.f;
        Lc[i] = v;
        Lt[(h * d + b) * d + a] = v;
    }
}

// cnorm[h][j] = |c[h][j]| (compensated sum of squares); one warp per centroid.
template <int DT>
__global__ void centroid_norm_kernel(const void* __restrict__ c, int64_t HK, int32_t d,
                                     float* __restrict__ cnorm) {
    const int lane = threadIdx.x & 31;
    for (int64_t j = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; j < HK;
         j += ((int64_t)gridDim.x * blockDim.x) >> 5) {
        Dot2 n;
        for (int a = lane; a < d; a += 32) {
            const float v = load1<DT>(c, j * d + a);
            n.add_prod(v, v);
        }
        for (int m = 16; m; m >>= 1) n.merge(shfl_xor(n, m));
        if (lane == 0) cnorm[j] = sqrtf(n.value());
    }
}

}  // namespace

// Slices of the M queries per head: about 256 queries each, at most 64;
// halved while the grid would need more than one wave of three CTAs per SM
// (about 448) and a slice stays within 2048 queries (the tensor-core
// kernel's four accumulators of 512).
int64_t second_moment_splits(int64_t M, int64_t H) {
    int64_t s = M / 256;
    s = s < 1 ? 1 : (s > 64 ? 64 : s);
    while (s > 1 && s * H > 448 && (M + s / 2 - 1) / (s / 2) <= 2048) s /= 2;
    return s;
}

cudaError_t launch_second_moment(const void* q, int dt, int64_t H, int64_t M, int64_t d,
                                 double ridge, float* partial, int32_t* status, float* h_out,
                                 cudaStream_t st) {
    const int64_t splits = second_moment_splits(M, H);
    cudaError_t e = cudaSuccess;
    if (second_moment_tc_supported(dt, H, M, d)) {
        e = cudaMemsetAsync(status, 0, sizeof(int32_t), st);
        if (e != cudaSuccess) return e;
        e = launch_second_moment_tc(q, dt, H, M, partial, status, st);
    } else {
        // tiles past the edge of H (d not a multiple of 32) read zeros and write nothing
        const int Tt = (int)((d + kSmTile - 1) / kSmTile);
        dim3 grid(Tt * (Tt + 1) / 2, (unsigned)splits, (unsigned)H);
        switch (dt) {
            case kF32:
                second_moment_partial_kernel<kF32><<<grid, kSmThreads, 0, st>>>(
                    q, M, (int32_t)d, splits, partial);
                break;
            case kBF16:
                second_moment_partial_kernel<kBF16><<<grid, kSmThreads, 0, st>>>(
                    q, M, (int32_t)d, splits, partial);
                break;
            default:
                second_moment_partial_kernel<kF16><<<grid, kSmThreads, 0, st>>>(
                    q, M, (int32_t)d, splits, partial);
        }
        note_launches(1);
        e = cudaGetLastError();
    }
    if (e != cudaSuccess) return e;
    const int64_t n = H * d * d;
    second_moment_reduce_kernel<<<(unsigned)((n + 255) / 256 < 4096 ? (n + 255) / 256 : 4096),
                                  256, 0, st>>>(partial, H, M, (int32_t)d, splits, (float)ridge,
                                                h_out);
    note_launches(1);
    return cudaGetLastError();
}

cudaError_t launch_cholesky(const float* h, int64_t H, int64_t d, float* l_out, int32_t* info,
                            cudaStream_t st) {
    if (H == 0) return cudaSuccess;
    const size_t packed = (size_t)((d * (d + 1) / 2 + 1) & ~1);
    const size_t smem = sizeof(float) * packed + sizeof(float2) * (size_t)(d * kPS) +
                        sizeof(float) * (size_t)d;
    cudaError_t e = cudaFuncSetAttribute(cholesky_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    cholesky_kernel<<<(unsigned)H, kCholThreads, smem, st>>>(h, (int32_t)d, l_out, info);
    note_launches(1);
    return cudaGetLastError();
}

cudaError_t launch_factor_prep(const float* L, int64_t H, int64_t d, float* Lc, float* Lt,
                               cudaStream_t st) {
    const int64_t n = H * d * d;
    if (n == 0) return cudaSuccess;
    const int64_t blocks = (n + 255) / 256;
    factor_prep_kernel<<<(unsigned)(blocks < 4096 ? blocks : 4096), 256, 0, st>>>(
        L, H, (int32_t)d, Lc, Lt);
    note_launches(1);
    return cudaGetLastError();
}

cudaError_t launch_codebook_transform(const void* c, int dt, int64_t H, int64_t K, int64_t d,
                                      const float* Lc, const float* Lt, float* cp,
                                      float* half_norm, float* chat, cudaStream_t st) {
    if (H * K == 0) return cudaSuccess;
    dim3 grid((unsigned)((K + kCtCent - 1) / kCtCent), (unsigned)H);
    const unsigned threads = (unsigned)(2 * ((d + 31) / 32 * 32));
    switch (dt) {
        case kF32:
            codebook_transform_kernel<kF32><<<grid, threads, 0, st>>>(c, K, (int32_t)d, Lc, Lt, cp,
                                                                       half_norm, chat);
            break;
        case kBF16:
            codebook_transform_kernel<kBF16><<<grid, threads, 0, st>>>(c, K, (int32_t)d, Lc, Lt,
                                                                        cp, half_norm, chat);
            break;
        default:
            codebook_transform_kernel<kF16><<<grid, threads, 0, st>>>(c, K, (int32_t)d, Lc, Lt, cp,
                                                                       half_norm, chat);
    }
    note_launches(1);
    return cudaGetLastError();
}

cudaError_t launch_centroid_norms(const void* c, int dt, int64_t H, int64_t K, int64_t d,
                                  float* cnorm, cudaStream_t st) {
    const int64_t HK = H * K;
    const unsigned blocks = (unsigned)((HK * 32 + 255) / 256 < 2048 ? (HK * 32 + 255) / 256 : 2048);
    switch (dt) {
        case kF32:
            centroid_norm_kernel<kF32><<<blocks, 256, 0, st>>>(c, HK, (int32_t)d, cnorm);
            note_launches(1);
            break;
        case kBF16:
            centroid_norm_kernel<kBF16><<<blocks, 256, 0, st>>>(c, HK, (int32_t)d, cnorm);
            note_launches(1);
            break;
        default:
            centroid_norm_kernel<kF16><<<blocks, 256, 0, st>>>(c, HK, (int32_t)d, cnorm);
            note_launches(1);
    }
    return cudaGetLastError();
}

}  // namespace a2ats
