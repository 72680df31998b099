// kmeans.cu -- codebook calibration in Cholesky space (sm_103a).
//
// API page "veloxquant_mlx.quantizers.a2ats module", a2ats_cholesky_factor:
// with H = L L^T the H-weighted distance (k - c) H (k - c)^T is the plain
// squared distance between z = k L and c L, so ordinary k-means++ on the
// rows z trains the codebook, and c = c_z L^-1 takes it back to key space.
//
//   kmeans_seed_kernel     k-means++ seeding with caller-given uniform draws:
//                          one CTA per head, persistent over the K picks.
//   kmeans_update_kernel   one Lloyd mean step (and the objective of the
//                          assignment it is given): a warp per centroid.
//   kmeans_objective_kernel  the per-head sum of the per-centroid objectives.
//   cholesky_solve_kernel  c with c L = z_c (back substitution), a warp per row.
//
// The nearest-centroid step of every Lloyd round is the library's exact
// assignment (L = identity on the fp32 rows z), launched from api.cu.
//
// Precision.  Which point a seeding round picks is a floating-point decision
// (the first running sum of D^2 above u * sum D^2), so D^2 is carried in
// fp64 with the same operation order as a plain sequential sum over the
// columns.  GB300's fp64 rate is a small fraction of its fp32 rate, so each
// round first screens the new centre in fp32 and computes the fp64 distance
// only for rows that the new centre may bring closer (the screen's bound is
// the a-priori error bound of an fp32 sum of d squares, doubled).  The Lloyd
// means are fp64 sums over each centroid's rows in ascending row order,
// divided by the count, then rounded to fp32.
#include <math.h>

#include "kernels.cuh"

namespace a2ats {
namespace {

constexpr int kSeedThreads = 512;
constexpr int kSeedWarps = kSeedThreads / 32;
constexpr int kUpdWarps = 8;
constexpr int kUpdChunk = 1024;
constexpr int kSolveWarps = 8;

// Row index of a uniform draw u in [0, 1) over n rows, clamped to [0, n).
__device__ __forceinline__ int64_t draw_index(double u, int64_t n) {
    const double f = floor(__dmul_rn(u, (double)n));
    int64_t p = (f >= 0.0) ? (int64_t)f : 0;  // also 0 for NaN
    return p < n ? p : n - 1;
}

// |z_i - c|^2 in fp64, columns summed in ascending order without contraction.
__device__ __forceinline__ double sq_dist_f64(const float* __restrict__ zi, const float* c, int d) {
    double s = 0.0;
    for (int a = 0; a < d; a++) {
        const double t = __dsub_rn((double)zi[a], (double)c[a]);
        s = __dadd_rn(s, __dmul_rn(t, t));
    }
    return s;
}

// One CTA per head.  Thread t owns the contiguous rows [lo, hi) of its head,
// so the running sums the pick needs are its own sequential sum plus an
// exclusive block scan of the threads' sums.  d2 [H, n] fp64 is workspace.
__global__ void __launch_bounds__(kSeedThreads, 1)
kmeans_seed_kernel(const float* __restrict__ z, int64_t n, int32_t d, int64_t K,
                   const double* __restrict__ u, float* __restrict__ cent,
                   double* __restrict__ d2g) {
    __shared__ __align__(16) float s_c[kMaxD];
    __shared__ double s_wsum[kSeedWarps];
    __shared__ double s_woff[kSeedWarps];
    __shared__ double s_total;
    __shared__ int s_first;
    __shared__ long long s_pick;
    const int h = blockIdx.x, t = threadIdx.x, lane = t & 31, warp = t >> 5;
    const float* zh = z + (int64_t)h * n * d;
    float* ch = cent + (int64_t)h * K * d;
    double* d2 = d2g + (int64_t)h * n;
    const double* uh = u + (int64_t)h * K;
    const int64_t chunk = (n + kSeedThreads - 1) / kSeedThreads;
    const int64_t lo = (int64_t)t * chunk < n ? (int64_t)t * chunk : n;
    const int64_t hi = lo + chunk < n ? lo + chunk : n;
    // a row is skipped when fp32 D^2 times this factor still exceeds its D^2
    const double keep = 1.0 - (double)(d + 8) * 0x1p-23;

    int64_t pick = draw_index(uh[0], n);
    if (t < d) {
        const float v = zh[pick * d + t];
        s_c[t] = v;
        ch[t] = v;
    }
    if (t == 0) s_first = kSeedThreads;
    __syncthreads();

    for (int64_t k = 1; k < K; k++) {
        // D^2 of the own rows against the newest centre (s_c), and their sum
        double csum = 0.0;
        for (int64_t i = lo; i < hi; i++) {
            const float* zi = zh + i * d;
            double cur = k == 1 ? (double)INFINITY : d2[i];
            bool write = k == 1;  // the first round sets every row's D^2
            float acc = 0.f;
            for (int a = 0; a < d; a += 4) {
                const float4 v = *reinterpret_cast<const float4*>(zi + a);
                const float4 c = *reinterpret_cast<const float4*>(s_c + a);
                const float e0 = v.x - c.x, e1 = v.y - c.y, e2 = v.z - c.z, e3 = v.w - c.w;
                acc = fmaf(e0, e0, acc);
                acc = fmaf(e1, e1, acc);
                acc = fmaf(e2, e2, acc);
                acc = fmaf(e3, e3, acc);
            }
            if (!(isfinite(acc) && (double)acc * keep > cur)) {
                const double s = sq_dist_f64(zi, s_c, d);
                if (s < cur) {
                    cur = s;
                    write = true;
                }
            }
            if (write) d2[i] = cur;
            csum = __dadd_rn(csum, cur);
        }
        // exclusive scan of the threads' sums (block order = row order)
        double x = csum;
        for (int o = 1; o < 32; o <<= 1) {
            const double y = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o) x = __dadd_rn(x, y);
        }
        double ex = __shfl_up_sync(0xffffffffu, x, 1);
        if (lane == 0) ex = 0.0;
        if (lane == 31) s_wsum[warp] = x;
        __syncthreads();
        if (warp == 0) {
            if (t == 0) s_first = kSeedThreads;
            const double w = lane < kSeedWarps ? s_wsum[lane] : 0.0;
            double xi = w;
            for (int o = 1; o < 32; o <<= 1) {
                const double y = __shfl_up_sync(0xffffffffu, xi, o);
                if (lane >= o) xi = __dadd_rn(xi, y);
            }
            double wex = __shfl_up_sync(0xffffffffu, xi, 1);
            if (lane == 0) wex = 0.0;
            if (lane < kSeedWarps) s_woff[lane] = wex;
        }
        __syncthreads();
        const double E = __dadd_rn(s_woff[warp], ex);  // sum of the rows before lo
        const double P = __dadd_rn(E, csum);           // ... through hi - 1
        if (t == kSeedThreads - 1) s_total = P;
        __syncthreads();
        const double total = s_total;
        const double target = __dmul_rn(uh[k], total);
        if (total > 0.0 && hi > lo && P > target) atomicMin(&s_first, t);
        __syncthreads();
        if (total > 0.0 && t == s_first) {
            // E + (the same running sum as csum) reaches P at hi - 1, so the
            // first crossing lies in [lo, hi)
            double run = 0.0;
            long long p = hi - 1;
            for (int64_t i = lo; i < hi; i++) {
                run = __dadd_rn(run, d2[i]);
                if (__dadd_rn(E, run) > target) {
                    p = i;
                    break;
                }
            }
            s_pick = p;
        }
        __syncthreads();
        if (total > 0.0)
            pick = s_first < kSeedThreads ? (int64_t)s_pick : n - 1;
        else
            pick = draw_index(uh[k], n);
        if (t < d) {
            const float v = zh[pick * d + t];
            s_c[t] = v;
            ch[k * d + t] = v;
        }
        __syncthreads();
    }
}

// Warp (blockIdx.x * kUpdWarps + warp) of head blockIdx.y owns centroid j:
// it walks the codes of its head in ascending row order (a chunk of codes at
// a time, shared by the block's warps), and for every row coded j adds the
// row to its fp64 column sums and the row's squared distance to the current
// centroid to its objective.  update != 0: centroid j <- sum / count (kept
// when no row has code j).  obj_part [H, K] receives the objectives.
__global__ void __launch_bounds__(kUpdWarps * 32, 1)
kmeans_update_kernel(const float* __restrict__ z, int64_t n, int32_t d, int64_t K,
                     const int32_t* __restrict__ codes, float* __restrict__ cent,
                     double* __restrict__ obj_part, int32_t update) {
    constexpr int kCols = kMaxD / 32;
    __shared__ int32_t s_codes[kUpdChunk];
    const int h = blockIdx.y;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t j = (int64_t)blockIdx.x * kUpdWarps + warp;
    const bool active = j < K;
    const float* zh = z + (int64_t)h * n * d;
    const int32_t* code_h = codes + (int64_t)h * n;
    float* cj = cent + ((int64_t)h * K + (active ? j : 0)) * d;
    float c_old[kCols];
    double sum[kCols];
#pragma unroll
    for (int m = 0; m < kCols; m++) {
        const int a = lane + 32 * m;
        c_old[m] = (active && a < d) ? cj[a] : 0.f;
        sum[m] = 0.0;
    }
    double obj = 0.0;
    int64_t cnt = 0;
    for (int64_t base = 0; base < n; base += kUpdChunk) {
        const int m_rows = (int)(n - base < kUpdChunk ? n - base : kUpdChunk);
        __syncthreads();  // every warp is done with the previous chunk
        for (int i = threadIdx.x; i < m_rows; i += blockDim.x) s_codes[i] = code_h[base + i];
        __syncthreads();
        if (!active) continue;
        for (int i0 = 0; i0 < m_rows; i0 += 32) {
            const int i = i0 + lane;
            unsigned mask = __ballot_sync(0xffffffffu, i < m_rows && s_codes[i] == (int32_t)j);
            while (mask) {
                const int b = __ffs(mask) - 1;
                mask &= mask - 1;
                const float* zr = zh + (base + i0 + b) * d;
                cnt++;
#pragma unroll
                for (int m = 0; m < kCols; m++) {
                    const int a = lane + 32 * m;
                    if (a < d) {
                        const double v = (double)zr[a];
                        sum[m] = __dadd_rn(sum[m], v);
                        const double e = __dsub_rn(v, (double)c_old[m]);
                        obj = __dadd_rn(obj, __dmul_rn(e, e));
                    }
                }
            }
        }
    }
    if (!active) return;
    for (int o = 16; o; o >>= 1) obj = __dadd_rn(obj, __shfl_xor_sync(0xffffffffu, obj, o));
    if (lane == 0) obj_part[(int64_t)h * K + j] = obj;
    if (update && cnt > 0) {
        const double members = (double)cnt;
#pragma unroll
        for (int m = 0; m < kCols; m++) {
            const int a = lane + 32 * m;
            if (a < d) cj[a] = (float)(sum[m] / members);
        }
    }
}

// objective[h * stride] = sum_j obj_part[h][j]: one warp per head, lanes
// strided over j, then a fixed xor tree.
__global__ void kmeans_objective_kernel(const double* __restrict__ obj_part, int64_t H, int64_t K,
                                        double* __restrict__ objective, int64_t stride) {
    const int64_t h = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (h >= H) return;  // whole warps leave together
    double s = 0.0;
    for (int64_t j = lane; j < K; j += 32) s = __dadd_rn(s, obj_part[h * K + j]);
    for (int o = 16; o; o >>= 1) s = __dadd_rn(s, __shfl_xor_sync(0xffffffffu, s, o));
    if (lane == 0) objective[h * stride] = s;
}

// c [H, rows, d] with c L = zc (L [H, d, d] lower triangular, only a >= b
// read): column b of c L is sum_{a >= b} c_a L_ab, so c is solved from the
// last column down.  One warp per row, fp64 throughout, rounded to fp32.
__global__ void __launch_bounds__(kSolveWarps * 32)
cholesky_solve_kernel(const float* __restrict__ zc, int64_t H, int64_t rows, int32_t d,
                      const float* __restrict__ L, float* __restrict__ c) {
    __shared__ double s_row[kSolveWarps][kMaxD];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t r = (int64_t)blockIdx.x * kSolveWarps + warp;
    if (r >= H * rows) return;  // whole warps leave together
    const int64_t h = r / rows;
    const float* Lh = L + h * d * d;
    const float* zr = zc + r * d;
    double* cr = s_row[warp];
    for (int b = d - 1; b >= 0; b--) {
        double s = 0.0;
        for (int a = b + 1 + lane; a < d; a += 32)
            s = __dadd_rn(s, __dmul_rn(cr[a], (double)Lh[(int64_t)a * d + b]));
        for (int o = 16; o; o >>= 1) s = __dadd_rn(s, __shfl_xor_sync(0xffffffffu, s, o));
        const double v = __ddiv_rn(__dsub_rn((double)zr[b], s), (double)Lh[(int64_t)b * d + b]);
        if (lane == 0) cr[b] = v;
        __syncwarp();
    }
    for (int a = lane; a < d; a += 32) c[r * d + a] = (float)cr[a];
}

}  // namespace

cudaError_t launch_kmeans_seed(const float* z, int64_t H, int64_t n, int64_t d, int64_t K,
                               const double* u, float* cent, double* d2, cudaStream_t st) {
    if (H == 0) return cudaSuccess;
    kmeans_seed_kernel<<<(unsigned)H, kSeedThreads, 0, st>>>(z, n, (int32_t)d, K, u, cent, d2);
    note_launches(1);
    return cudaGetLastError();
}

cudaError_t launch_kmeans_update(const float* z, int64_t H, int64_t n, int64_t d, int64_t K,
                                 const int32_t* codes, float* cent, double* obj_part,
                                 bool update, double* objective, int64_t obj_stride,
                                 cudaStream_t st) {
    if (H == 0) return cudaSuccess;
    dim3 grid((unsigned)((K + kUpdWarps - 1) / kUpdWarps), (unsigned)H);
    kmeans_update_kernel<<<grid, kUpdWarps * 32, 0, st>>>(z, n, (int32_t)d, K, codes, cent,
                                                          obj_part, update ? 1 : 0);
    note_launches(1);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const int64_t threads = H * 32;
    kmeans_objective_kernel<<<(unsigned)((threads + 255) / 256), 256, 0, st>>>(
        obj_part, H, K, objective, obj_stride);
    note_launches(1);
    return cudaGetLastError();
}

cudaError_t launch_cholesky_solve(const float* zc, int64_t H, int64_t rows, int64_t d,
                                  const float* L, float* c, cudaStream_t st) {
    const int64_t total = H * rows;
    if (total == 0) return cudaSuccess;
    cholesky_solve_kernel<<<(unsigned)((total + kSolveWarps - 1) / kSolveWarps),
                            kSolveWarps * 32, 0, st>>>(zc, H, rows, (int32_t)d, L, c);
    note_launches(1);
    return cudaGetLastError();
}

}  // namespace a2ats
