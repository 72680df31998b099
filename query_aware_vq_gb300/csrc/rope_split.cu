// rope_split.cu -- windowed RoPE and the retrieval-set split.
//
// Windowed RoPE: deploy-preview "A2ATS-adapted" page, paper-fidelity section,
// "Windowed RoPE (Eq. 11-12)" and "Per-step re-rotation"; v0.39.0 page, "How it
// works" step 4.  Retrieval split: API page, a2ats_select_retrieval_set (top
// ceil(fraction * N) tokens by key-query cosine; the two sets are disjoint and
// cover every position).
//
// Both passes stream the key cache once and are bound by HBM bandwidth: each
// thread moves 16-byte vectors, a row of d elements is handled by d/16
// (half-split) or d/8 (interleaved) consecutive threads so every warp touches
// whole 128-byte lines, and the grid is a multiple of the SM count.
#include <cooperative_groups.h>

#include "kernels.cuh"

namespace a2ats {
namespace {

constexpr int kRopeThreads = 256;

// 8 consecutive elements as floats (one or two 16-byte accesses).
template <int DT>
__device__ __forceinline__ void load8(const void* base, int64_t off, float* v) {
    if constexpr (DT == kF32) {
        load_vec<kF32>(base, off, v);
        load_vec<kF32>(base, off + 4, v + 4);
    } else {
        load_vec<DT>(base, off, v);
    }
}

template <int DT>
__device__ __forceinline__ void store8(void* base, int64_t off, const float* v) {
    if constexpr (DT == kF32) {
        store_vec<kF32>(base, off, v);
        store_vec<kF32>(base, off + 4, v + 4);
    } else {
        store_vec<DT>(base, off, v);
    }
}

// Rotate the 8 elements a thread holds.  Half-split: v0[k] pairs with v1[k]
// (pair index pair0 + k).  Interleaved: v0[2k] pairs with v0[2k+1] (pair
// index pair0 + k).
template <bool INTERLEAVED>
__device__ __forceinline__ void rotate8(float* v0, float* v1, const float* c, const float* s) {
    if constexpr (!INTERLEAVED) {
#pragma unroll
        for (int k = 0; k < 8; k++) {
            const float xa = v0[k], xb = v1[k];
            v0[k] = fmaf(xa, c[k], -__fmul_rn(xb, s[k]));
            v1[k] = fmaf(xa, s[k], __fmul_rn(xb, c[k]));
        }
    } else {
#pragma unroll
        for (int k = 0; k < 4; k++) {
            const float xa = v0[2 * k], xb = v0[2 * k + 1];
            v0[2 * k] = fmaf(xa, c[k], -__fmul_rn(xb, s[k]));
            v0[2 * k + 1] = fmaf(xa, s[k], __fmul_rn(xb, c[k]));
        }
    }
}

template <bool INTERLEAVED>
__device__ __forceinline__ void angles8(int32_t pos, int pair0, const RopeArgs& ra, float* c,
                                        float* s) {
    constexpr int NP = INTERLEAVED ? 4 : 8;
#pragma unroll
    for (int k = 0; k < NP; k++)
        rope_angle(pos, ra.omega_hi[pair0 + k], ra.omega_lo[pair0 + k], ra, s[k], c[k]);
}

// One pass over every valid row: k_out = windowed RoPE of k_in.
template <int IN, int OUT, bool INTERLEAVED>
__global__ void __launch_bounds__(kRopeThreads)
windowed_rope_kernel(const void* __restrict__ kin, void* __restrict__ kout, int64_t rows,
                     int32_t H, int32_t ncap, int32_t d, const int32_t* __restrict__ len,
                     const RopeArgs ra) {
    const int lpr = INTERLEAVED ? d / 8 : d / 16;  // threads per row
    const int rpb = kRopeThreads / lpr;            // rows per block iteration
    const int lane = threadIdx.x % lpr;
    const int e0 = lane * 8;
    const int e1 = e0 + d / 2;
    const int pair0 = INTERLEAVED ? e0 / 2 : e0;
    const bool far_rot = ra.enabled && ra.far_offset != 0;
    float fc[8], fs[8];
    if (far_rot) angles8<INTERLEAVED>(ra.far_offset, pair0, ra, fc, fs);
    if ((int)threadIdx.x >= rpb * lpr) return;  // lpr need not divide the block

    for (int64_t row = (int64_t)blockIdx.x * rpb + threadIdx.x / lpr; row < rows;
         row += (int64_t)gridDim.x * rpb) {
        const int32_t j = (int32_t)(row % ncap);
        const int32_t b = (int32_t)(row / ncap / H);
        const int32_t L = seq_len(len, b, ncap);
        if (j >= L) continue;
        const int64_t base = row * d;
        float v0[8], v1[8];
        load8<IN>(kin, base + e0, v0);
        if (!INTERLEAVED) load8<IN>(kin, base + e1, v1);
        if (ra.enabled) {
            const bool near = ra.window > 0 && (L - 1 - j) < ra.window;
            if (near) {
                float c[8], s[8];
                angles8<INTERLEAVED>(j, pair0, ra, c, s);
                rotate8<INTERLEAVED>(v0, v1, c, s);
            } else if (far_rot) {
                rotate8<INTERLEAVED>(v0, v1, fc, fs);
            }
        }
        store8<OUT>(kout, base + e0, v0);
        if (!INTERLEAVED) store8<OUT>(kout, base + e1, v1);
    }
}

// Fallback for widths that are a multiple of 8 but not of 16 (half-split):
// one thread per pair, scalar accesses.
template <int IN, int OUT>
__global__ void __launch_bounds__(kRopeThreads)
windowed_rope_scalar_kernel(const void* __restrict__ kin, void* __restrict__ kout, int64_t rows,
                            int32_t H, int32_t ncap, int32_t d, const int32_t* __restrict__ len,
                            const RopeArgs ra) {
    const int half = d / 2;
    const int64_t pairs = rows * half;
    for (int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; idx < pairs;
         idx += (int64_t)gridDim.x * blockDim.x) {
        const int64_t row = idx / half;
        const int i = (int)(idx % half);
        const int32_t j = (int32_t)(row % ncap);
        const int32_t b = (int32_t)(row / ncap / H);
        const int32_t L = seq_len(len, b, ncap);
        if (j >= L) continue;
        const int a = ra.interleaved ? 2 * i : i;
        const int bb = ra.interleaved ? 2 * i + 1 : i + half;
        float xa = load1<IN>(kin, row * d + a), xb = load1<IN>(kin, row * d + bb);
        if (ra.enabled) {
            const int32_t pos = rope_position(j, L - 1, ra);
            if (pos != 0) {
                float s, c;
                rope_angle(pos, ra.omega_hi[i], ra.omega_lo[i], ra, s, c);
                const float ya = fmaf(xa, c, -__fmul_rn(xb, s));
                const float yb = fmaf(xa, s, __fmul_rn(xb, c));
                xa = ya;
                xb = yb;
            }
        }
        using TO = typename Elem<OUT>::T;
        reinterpret_cast<TO*>(kout)[row * d + a] = from_f32<OUT>(xa);
        reinterpret_cast<TO*>(kout)[row * d + bb] = from_f32<OUT>(xb);
    }
}

int grid_for(int64_t work_items, int per_block) {
    int dev = 0, sms = 152;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int64_t need = (work_items + per_block - 1) / per_block;
    const int64_t cap = (int64_t)sms * 8;
    return (int)(need < cap ? (need > 0 ? need : 1) : cap);
}

template <int IN, int OUT>
cudaError_t rope_dispatch_out(const void* kin, void* kout, const Shape& s, const int32_t* len,
                              const RopeArgs& ra, cudaStream_t st) {
    const int64_t rows = s.B * s.H * s.Ncap;
    const int d = (int)s.d;
    if (ra.interleaved) {
        const int lpr = d / 8;
        windowed_rope_kernel<IN, OUT, true><<<grid_for(rows, kRopeThreads / lpr), kRopeThreads, 0,
                                              st>>>(kin, kout, rows, (int32_t)s.H,
                                                    (int32_t)s.Ncap, d, len, ra);
                                                    note_launches(1);
    } else if (d % 16 == 0) {
        const int lpr = d / 16;
        windowed_rope_kernel<IN, OUT, false><<<grid_for(rows, kRopeThreads / lpr), kRopeThreads,
                                               0, st>>>(kin, kout, rows, (int32_t)s.H,
                                                        (int32_t)s.Ncap, d, len, ra);
                                                        note_launches(1);
    } else {
        windowed_rope_scalar_kernel<IN, OUT><<<grid_for(rows * (d / 2), kRopeThreads),
                                               kRopeThreads, 0, st>>>(
            kin, kout, rows, (int32_t)s.H, (int32_t)s.Ncap, d, len, ra);
            note_launches(1);
    }
    return cudaGetLastError();
}

template <int IN>
cudaError_t rope_dispatch(const void* kin, void* kout, int out_dt, const Shape& s,
                          const int32_t* len, const RopeArgs& ra, cudaStream_t st) {
    switch (out_dt) {
        case kF32: return rope_dispatch_out<IN, kF32>(kin, kout, s, len, ra, st);
        case kBF16: return rope_dispatch_out<IN, kBF16>(kin, kout, s, len, ra, st);
        default: return rope_dispatch_out<IN, kF16>(kin, kout, s, len, ra, st);
    }
}

// ------------------------------------------------------------ split --
// Query of each (b, h), decoded to fp32, and its norm (compensated sum).
// query == nullptr: the proxy query, the key at t = len-1 after windowed RoPE.
template <int DT>
__global__ void __launch_bounds__(128)
prepare_query_kernel(const void* __restrict__ keys, const void* __restrict__ query, int32_t H,
                     int32_t ncap, int32_t d, const int32_t* __restrict__ len, const RopeArgs ra,
                     float* __restrict__ q_out, float* __restrict__ qnorm) {
    __shared__ float v[kMaxD];
    __shared__ Dot2 red[4];
    const int bh = blockIdx.x;
    const int b = bh / H;
    const int32_t L = seq_len(len, b, ncap);
    const int tid = threadIdx.x;
    if (query) {
        for (int i = tid; i < d; i += blockDim.x) v[i] = load1<DT>(query, (int64_t)bh * d + i);
    } else if (L == 0) {
        for (int i = tid; i < d; i += blockDim.x) v[i] = 0.f;
    } else {
        const int64_t row = ((int64_t)bh * ncap + (L - 1)) * d;
        for (int i = tid; i < d; i += blockDim.x) v[i] = load1<DT>(keys, row + i);
    }
    __syncthreads();
    if (!query && L > 0 && ra.enabled) {
        const int32_t pos = rope_position(L - 1, L - 1, ra);
        const int half = d / 2;
        float a = 0.f, bv = 0.f;
        int ia = 0, ib = 0;
        if (tid < half) {
            ia = ra.interleaved ? 2 * tid : tid;
            ib = ra.interleaved ? 2 * tid + 1 : tid + half;
            a = v[ia];
            bv = v[ib];
        }
        __syncthreads();
        if (tid < half && pos != 0) {
            float s, c;
            rope_angle(pos, ra.omega_hi[tid], ra.omega_lo[tid], ra, s, c);
            v[ia] = fmaf(a, c, -__fmul_rn(bv, s));
            v[ib] = fmaf(a, s, __fmul_rn(bv, c));
        }
        __syncthreads();
    }
    Dot2 acc;
    for (int i = tid; i < d; i += blockDim.x) {
        q_out[(int64_t)bh * d + i] = v[i];
        acc.add_prod(v[i], v[i]);
    }
    for (int m = 16; m; m >>= 1) acc.merge(shfl_xor(acc, m));
    if ((tid & 31) == 0) red[tid >> 5] = acc;
    __syncthreads();
    if (tid == 0) {
        Dot2 t = red[0];
        for (int w = 1; w < (int)(blockDim.x >> 5); w++) t.merge(red[w]);
        qnorm[bh] = sqrtf(t.value());
    }
}

// Cosine of every valid row with its query (fp32; fused windowed RoPE).
template <int DT, bool INTERLEAVED>
__global__ void __launch_bounds__(kRopeThreads)
cosine_score_kernel(const void* __restrict__ keys, int64_t rows, int32_t H, int32_t ncap,
                    int32_t d, const int32_t* __restrict__ len, const RopeArgs ra,
                    const float* __restrict__ q, const float* __restrict__ qnorm,
                    float* __restrict__ scores) {
    const int lpr = INTERLEAVED ? d / 8 : d / 16;
    const int rpb = kRopeThreads / lpr;
    const int lane = threadIdx.x % lpr;
    const int e0 = lane * 8;
    const int e1 = e0 + d / 2;
    const int pair0 = INTERLEAVED ? e0 / 2 : e0;
    const bool far_rot = ra.enabled && ra.far_offset != 0;
    float fc[8], fs[8];
    if (far_rot) angles8<INTERLEAVED>(ra.far_offset, pair0, ra, fc, fs);
    for (int64_t row0 = (int64_t)blockIdx.x * rpb; row0 < rows; row0 += (int64_t)gridDim.x * rpb) {
        const int64_t row = row0 + threadIdx.x / lpr;
        bool valid = row < rows;
        int32_t j = 0, L = 0;
        int64_t bh = 0;
        if (valid) {
            j = (int32_t)(row % ncap);
            bh = row / ncap;
            L = seq_len(len, (int32_t)(bh / H), ncap);
            valid = j < L;
        }
        float dot = 0.f, nn = 0.f;
        if (valid) {
            const int64_t base = row * d;
            float v0[8], v1[8];
            load8<DT>(keys, base + e0, v0);
            if (!INTERLEAVED) load8<DT>(keys, base + e1, v1);
            if (ra.enabled) {
                const bool near = ra.window > 0 && (L - 1 - j) < ra.window;
                if (near) {
                    float c[8], s[8];
                    angles8<INTERLEAVED>(j, pair0, ra, c, s);
                    rotate8<INTERLEAVED>(v0, v1, c, s);
                } else if (far_rot) {
                    rotate8<INTERLEAVED>(v0, v1, fc, fs);
                }
            }
            const float* qq = q + bh * d;
#pragma unroll
            for (int k = 0; k < 8; k++) {
                dot = fmaf(v0[k], qq[e0 + k], dot);
                nn = fmaf(v0[k], v0[k], nn);
            }
            if (!INTERLEAVED) {
#pragma unroll
                for (int k = 0; k < 8; k++) {
                    dot = fmaf(v1[k], qq[e1 + k], dot);
                    nn = fmaf(v1[k], v1[k], nn);
                }
            }
        }
        // reduce over the lpr lanes of the row (lpr is a power of two <= 32)
        for (int m = lpr >> 1; m; m >>= 1) {
            dot += __shfl_xor_sync(0xffffffffu, dot, m);
            nn += __shfl_xor_sync(0xffffffffu, nn, m);
        }
        if (valid && lane == 0) {
            const float qn = qnorm[bh];
            const float kn = sqrtf(nn);
            scores[row] = (kn > 0.f && qn > 0.f) ? dot / (kn * qn) : 0.f;
        }
    }
}

// Generic-width score kernel: one warp per row.
template <int DT>
__global__ void __launch_bounds__(kRopeThreads)
cosine_score_warp_kernel(const void* __restrict__ keys, int64_t rows, int32_t H, int32_t ncap,
                         int32_t d, const int32_t* __restrict__ len, const RopeArgs ra,
                         const float* __restrict__ q, const float* __restrict__ qnorm,
                         float* __restrict__ scores) {
    __shared__ float buf[kRopeThreads / 32][kMaxD];
    const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int64_t row = (int64_t)blockIdx.x * (kRopeThreads / 32) + w; row < rows;
         row += (int64_t)gridDim.x * (kRopeThreads / 32)) {
        const int32_t j = (int32_t)(row % ncap);
        const int64_t bh = row / ncap;
        const int32_t L = seq_len(len, (int32_t)(bh / H), ncap);
        if (j >= L) continue;
        float* v = buf[w];
        for (int i = lane; i < d; i += 32) v[i] = load1<DT>(keys, row * d + i);
        __syncwarp();
        if (ra.enabled) {
            const int32_t pos = rope_position(j, L - 1, ra);
            if (pos != 0) {
                const int half = d / 2;
                for (int i = lane; i < half; i += 32) {
                    const int a = ra.interleaved ? 2 * i : i;
                    const int bb = ra.interleaved ? 2 * i + 1 : i + half;
                    float s, c;
                    rope_angle(pos, ra.omega_hi[i], ra.omega_lo[i], ra, s, c);
                    const float xa = v[a], xb = v[bb];
                    v[a] = fmaf(xa, c, -__fmul_rn(xb, s));
                    v[bb] = fmaf(xa, s, __fmul_rn(xb, c));
                }
            }
        }
        __syncwarp();
        float dot = 0.f, nn = 0.f;
        for (int i = lane; i < d; i += 32) {
            dot = fmaf(v[i], q[bh * d + i], dot);
            nn = fmaf(v[i], v[i], nn);
        }
        for (int m = 16; m; m >>= 1) {
            dot += __shfl_xor_sync(0xffffffffu, dot, m);
            nn += __shfl_xor_sync(0xffffffffu, nn, m);
        }
        if (lane == 0) {
            const float qn = qnorm[bh];
            const float kn = sqrtf(nn);
            scores[row] = (kn > 0.f && qn > 0.f) ? dot / (kn * qn) : 0.f;
        }
        __syncwarp();
    }
}

constexpr int kSelThreads = 512;
constexpr int kSelCluster = 8;

// Exclusive block-wide scan of one flag per thread; returns the block total.
__device__ __forceinline__ int block_scan_flag(bool f, int& excl, int* warp_tot) {
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const unsigned bal = __ballot_sync(0xffffffffu, f);
    const int in_warp = __popc(bal & ((1u << lane) - 1u));
    if (lane == 0) warp_tot[w] = __popc(bal);
    __syncthreads();
    if (w == 0) {
        const int nw = blockDim.x >> 5;
        int v = lane < nw ? warp_tot[lane] : 0;
        int inc = v;
        for (int m = 1; m < 32; m <<= 1) {
            const int t = __shfl_up_sync(0xffffffffu, inc, m);
            if (lane >= m) inc += t;
        }
        warp_tot[32 + lane] = inc - v;  // exclusive prefix of warp totals
        if (lane == 31) warp_tot[64] = inc;
    }
    __syncthreads();
    excl = warp_tot[32 + w] + in_warp;
    const int total = warp_tot[64];
    __syncthreads();
    return total;
}

// Exact top-n_r per (b, h) by radix select on order-preserving keys of the
// scores, ties on the threshold broken by lower index, then a stable
// two-sided compaction: retrieval rows ascending, then bulk rows ascending.
// One cluster of kSelCluster CTAs per (b, h): each CTA owns a contiguous
// segment of the row; the per-pass histograms and the compaction offsets are
// combined through distributed shared memory.
__global__ void __cluster_dims__(kSelCluster, 1, 1) __launch_bounds__(kSelThreads)
select_kernel(const float* __restrict__ scores, int32_t H, int32_t ncap,
              const int32_t* __restrict__ len, double fraction, int32_t* __restrict__ perm,
              int32_t* __restrict__ count) {
    namespace cg = cooperative_groups;
    cg::cluster_group cluster = cg::this_cluster();
    __shared__ uint32_t hist[256];
    __shared__ int seg_counts[2];   // this CTA's rows above the threshold, equal to it
    __shared__ int warp_tot[65];
    const int rank = (int)cluster.block_rank();
    const int bh = blockIdx.x / kSelCluster;
    const int32_t n = seq_len(len, bh / H, ncap);
    const float* s = scores + (int64_t)bh * ncap;
    int32_t* out = perm + (int64_t)bh * ncap;
    const double kd = ceil(fraction * (double)n);
    const int32_t k = kd < 0.0 ? 0 : (kd > (double)n ? n : (int32_t)kd);
    if (rank == 0 && threadIdx.x == 0) count[bh] = k;
    const int32_t seg = (n + kSelCluster - 1) / kSelCluster;
    const int32_t lo = min(n, rank * seg), hi = min(n, lo + seg);

    uint32_t prefix = 0, mask = 0, need = (uint32_t)k;
    const bool partial = k > 0 && k < n;
    if (partial) {
        for (int shift = 24; shift >= 0; shift -= 8) {
            for (int i = threadIdx.x; i < 256; i += blockDim.x) hist[i] = 0;
            __syncthreads();
            for (int i = lo + threadIdx.x; i < hi; i += blockDim.x) {
                const uint32_t u = ordered_key(s[i]);
                if ((u & mask) == prefix) atomicAdd(&hist[(u >> shift) & 255u], 1u);
            }
            cluster.sync();
            // every CTA sums the cluster's histograms and takes the same digit
            __shared__ uint32_t tot[256];
            for (int i = threadIdx.x; i < 256; i += blockDim.x) {
                uint32_t t = 0;
                for (int r = 0; r < kSelCluster; r++) t += cluster.map_shared_rank(hist, r)[i];
                tot[i] = t;
            }
            cluster.sync();  // no CTA resets its histogram while another reads it
            __shared__ uint32_t sel_prefix, sel_need;
            if (threadIdx.x == 0) {
                uint32_t cum = 0;
                for (int dg = 255; dg >= 0; --dg) {
                    const uint32_t hcount = tot[dg];
                    if (cum + hcount >= need) {
                        sel_prefix = prefix | ((uint32_t)dg << shift);
                        sel_need = need - cum;
                        break;
                    }
                    cum += hcount;
                }
            }
            __syncthreads();
            prefix = sel_prefix;
            need = sel_need;
            mask |= 255u << shift;
            __syncthreads();
        }
    }
    // per-CTA counts of rows above and equal to the threshold, then prefixes
    // over the CTAs of lower rank
    int gt_local = 0, eq_local = 0;
    if (partial) {
        for (int i = lo + threadIdx.x; i < hi; i += blockDim.x) {
            const uint32_t u = ordered_key(s[i]);
            gt_local += u > prefix;
            eq_local += u == prefix;
        }
    }
    gt_local = __reduce_add_sync(0xffffffffu, gt_local);
    eq_local = __reduce_add_sync(0xffffffffu, eq_local);
    if (threadIdx.x == 0) { seg_counts[0] = 0; seg_counts[1] = 0; }
    __syncthreads();
    if ((threadIdx.x & 31) == 0) {
        atomicAdd(&seg_counts[0], gt_local);
        atomicAdd(&seg_counts[1], eq_local);
    }
    cluster.sync();
    int gt_before = 0, eq_before = 0;
    for (int r = 0; r < rank; r++) {
        const int* other = cluster.map_shared_rank(seg_counts, r);
        gt_before += other[0];
        eq_before += other[1];
    }
    cluster.sync();  // the counts stay readable until every CTA has them
    // rows taken before this segment: those above the threshold plus the
    // equal ones that fit in `need`, in index order
    const int eq_taken_before = min(eq_before, (int)need);
    int carry_take = partial ? gt_before + eq_taken_before : (k == n ? lo : 0);
    int carry_eq = eq_before;
    for (int base = lo; base < hi; base += blockDim.x) {
        const int i = base + threadIdx.x;
        const bool valid = i < hi;
        uint32_t u = 0;
        if (valid && partial) u = ordered_key(s[i]);
        const bool eq = valid && partial && u == prefix;
        int eq_excl;
        const int eq_tot = block_scan_flag(eq, eq_excl, warp_tot);
        const bool take = valid && (k == n || (partial && (u > prefix ||
                                                           (eq && carry_eq + eq_excl < (int)need))));
        int t_excl;
        const int t_tot = block_scan_flag(take, t_excl, warp_tot);
        if (valid) {
            const int pos_r = carry_take + t_excl;
            if (take) out[pos_r] = i;
            else out[k + (i - pos_r)] = i;
        }
        carry_eq += eq_tot;
        carry_take += t_tot;
    }
}

// One block per sequence: every head's new row is copied into slot len[b]
// (16-byte vectors), then one thread advances len[b].
__global__ void append_rows_kernel(uint4* __restrict__ cache, int32_t H, int32_t ncap,
                                   int32_t vec, int32_t* __restrict__ len,
                                   const uint4* __restrict__ rows) {
    const int b = blockIdx.x;
    const int32_t L = len[b];
    if (L >= 0 && L < ncap) {
        for (int e = threadIdx.x; e < H * vec; e += blockDim.x) {
            const int h = e / vec, v = e % vec;
            cache[(((int64_t)b * H + h) * ncap + L) * vec + v] = rows[((int64_t)b * H + h) * vec + v];
        }
    }
    __syncthreads();
    if (threadIdx.x == 0 && L >= 0 && L < ncap) len[b] = L + 1;
}

template <int DT>
cudaError_t score_dispatch(const void* keys, const Shape& s, const int32_t* len,
                           const RopeArgs& ra, const float* q, const float* qnorm,
                           float* scores, cudaStream_t st) {
    const int64_t rows = s.B * s.H * s.Ncap;
    const int d = (int)s.d;
    // the score kernel reduces a row over lpr lanes with xor shuffles, so lpr
    // must be a power of two no larger than a warp
    const int lpr = ra.interleaved ? d / 8 : d / 16;
    const bool vec_ok = (ra.interleaved || d % 16 == 0) && lpr <= 32 && (lpr & (lpr - 1)) == 0;
    if (vec_ok && ra.interleaved) {
        cosine_score_kernel<DT, true><<<grid_for(rows, kRopeThreads / (d / 8)), kRopeThreads, 0,
                                        st>>>(keys, rows, (int32_t)s.H, (int32_t)s.Ncap, d, len,
                                              ra, q, qnorm, scores);
                                              note_launches(1);
    } else if (vec_ok) {
        cosine_score_kernel<DT, false><<<grid_for(rows, kRopeThreads / (d / 16)), kRopeThreads,
                                         0, st>>>(keys, rows, (int32_t)s.H, (int32_t)s.Ncap, d,
                                                  len, ra, q, qnorm, scores);
                                                  note_launches(1);
    } else {
        cosine_score_warp_kernel<DT><<<grid_for(rows, kRopeThreads / 32), kRopeThreads, 0, st>>>(
            keys, rows, (int32_t)s.H, (int32_t)s.Ncap, d, len, ra, q, qnorm, scores);
            note_launches(1);
    }
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_windowed_rope(const void* k_in, int in_dt, void* k_out, int out_dt,
                                 const Shape& s, const int32_t* len, const RopeArgs& ra,
                                 cudaStream_t st) {
    switch (in_dt) {
        case kF32: return rope_dispatch<kF32>(k_in, k_out, out_dt, s, len, ra, st);
        case kBF16: return rope_dispatch<kBF16>(k_in, k_out, out_dt, s, len, ra, st);
        default: return rope_dispatch<kF16>(k_in, k_out, out_dt, s, len, ra, st);
    }
}

cudaError_t launch_prepare_query(const void* keys, const void* query, int dt, const Shape& s,
                                 const int32_t* len, const RopeArgs& ra, float* q_out,
                                 float* qnorm, cudaStream_t st) {
    const int nbh = (int)(s.B * s.H);
    if (nbh == 0) return cudaSuccess;
    switch (dt) {
        case kF32:
            prepare_query_kernel<kF32><<<nbh, 128, 0, st>>>(keys, query, (int32_t)s.H,
                                                            (int32_t)s.Ncap, (int32_t)s.d, len,
                                                            ra, q_out, qnorm);
                                                            note_launches(1);
            break;
        case kBF16:
            prepare_query_kernel<kBF16><<<nbh, 128, 0, st>>>(keys, query, (int32_t)s.H,
                                                             (int32_t)s.Ncap, (int32_t)s.d, len,
                                                             ra, q_out, qnorm);
                                                             note_launches(1);
            break;
        default:
            prepare_query_kernel<kF16><<<nbh, 128, 0, st>>>(keys, query, (int32_t)s.H,
                                                            (int32_t)s.Ncap, (int32_t)s.d, len,
                                                            ra, q_out, qnorm);
                                                            note_launches(1);
    }
    return cudaGetLastError();
}

cudaError_t launch_cosine_scores(const void* keys, int dt, const Shape& s, const int32_t* len,
                                 const RopeArgs& ra, const float* q, const float* qnorm,
                                 float* scores, cudaStream_t st) {
    if (s.B * s.H * s.Ncap == 0) return cudaSuccess;
    switch (dt) {
        case kF32: return score_dispatch<kF32>(keys, s, len, ra, q, qnorm, scores, st);
        case kBF16: return score_dispatch<kBF16>(keys, s, len, ra, q, qnorm, scores, st);
        default: return score_dispatch<kF16>(keys, s, len, ra, q, qnorm, scores, st);
    }
}

cudaError_t launch_append_rows(void* cache, int dt, const Shape& s, int32_t* len, const void* rows,
                               cudaStream_t st) {
    const int32_t vec = (int32_t)(s.d * (dt == kF32 ? 4 : 2) / 16);
    append_rows_kernel<<<(unsigned)s.B, 256, 0, st>>>(reinterpret_cast<uint4*>(cache),
                                                      (int32_t)s.H, (int32_t)s.Ncap, vec, len,
                                                      reinterpret_cast<const uint4*>(rows));
    note_launches(1);
    return cudaGetLastError();
}

cudaError_t launch_select(const float* scores, const Shape& s, const int32_t* len,
                          double fraction, int32_t* perm, int32_t* count, cudaStream_t st) {
    const int nbh = (int)(s.B * s.H);
    if (nbh == 0) return cudaSuccess;
    select_kernel<<<nbh * kSelCluster, kSelThreads, 0, st>>>(scores, (int32_t)s.H,
                                                             (int32_t)s.Ncap, len, fraction, perm,
                                                             count);
                                               note_launches(1);
    return cudaGetLastError();
}

}  // namespace a2ats
