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

// One pass over every valid row: k_out = windowed RoPE of k_in (launched for
// the interleaved pairing; the half-split one takes windowed_rope_bh_kernel).
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

    // grid-stride over rows; (bh, j) of the thread's row advance by the
    // stride (qs whole sequences plus rs rows) without 64-bit divisions
    const int64_t stride = (int64_t)gridDim.x * rpb;
    const int64_t qs = stride / ncap;
    const int32_t rs = (int32_t)(stride - qs * ncap);
    int64_t row = (int64_t)blockIdx.x * rpb + threadIdx.x / lpr;
    int64_t bh = row / ncap;
    int32_t j = (int32_t)(row - bh * ncap);
    for (; row < rows; row += stride) {
        const int32_t L = seq_len(len, (int32_t)bh / H, ncap);
        const int32_t jr = j;
        j += rs;
        bh += qs;
        if (j >= ncap) {
            j -= ncap;
            bh++;
        }
        if (jr >= L) continue;
        const int64_t base = row * d;
        float v0[8], v1[8];
        load8<IN>(kin, base + e0, v0);
        if (!INTERLEAVED) load8<IN>(kin, base + e1, v1);
        if (ra.enabled) {
            const bool near = ra.window > 0 && (L - 1 - jr) < ra.window;
            if (near) {
                float c[8], s[8];
                angles8<INTERLEAVED>(jr, pair0, ra, c, s);
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

// The same scores (and stored rows) as cosine_score_kernel for the
// half-split pairing with d % 16 == 0, launched over (chunk of kBhRows rows,
// (b, h)) so that no thread walks the rows past a sequence's length; the
// (b, h) query is held in registers, and each lane group takes two rows at
// a time (four 16-byte loads in flight per lane).  The arithmetic of a row
// is that of cosine_score_kernel, so both give the same bits.
constexpr int kBhRows = 1024;

template <int DT, int OUT>
__global__ void __launch_bounds__(kRopeThreads, 3)
cosine_score_bh_kernel(const void* __restrict__ keys, int32_t H, int32_t ncap, int32_t d,
                       const int32_t* __restrict__ len, const RopeArgs ra,
                       const float* __restrict__ q, const float* __restrict__ qnorm,
                       float* __restrict__ scores, void* __restrict__ kout) {
    const int lpr = d / 16;
    const int rpb = kRopeThreads / lpr;
    const int lane = threadIdx.x & (lpr - 1);
    const int rl = threadIdx.x / lpr;
    const int e0 = lane * 8;
    const int e1 = e0 + d / 2;
    const int64_t bh = blockIdx.y;
    const int32_t L = seq_len(len, (int32_t)(bh / H), ncap);
    const int32_t jbeg = blockIdx.x * kBhRows;
    if (jbeg >= L) return;  // uniform over the block
    const int32_t jend = min(jbeg + kBhRows, L);
    const bool far_rot = ra.enabled && ra.far_offset != 0;
    float qv0[8], qv1[8];
    {
        const float4* qa = reinterpret_cast<const float4*>(q + bh * d + e0);
        const float4* qb = reinterpret_cast<const float4*>(q + bh * d + e1);
        const float4 a0 = __ldg(qa), a1 = __ldg(qa + 1), b0 = __ldg(qb), b1 = __ldg(qb + 1);
        qv0[0] = a0.x; qv0[1] = a0.y; qv0[2] = a0.z; qv0[3] = a0.w;
        qv0[4] = a1.x; qv0[5] = a1.y; qv0[6] = a1.z; qv0[7] = a1.w;
        qv1[0] = b0.x; qv1[1] = b0.y; qv1[2] = b0.z; qv1[3] = b0.w;
        qv1[4] = b1.x; qv1[5] = b1.y; qv1[6] = b1.z; qv1[7] = b1.w;
    }
    const float qn = qnorm[bh];
    // Blocks whose rows are all far, with no far rotation (the keys as they
    // are): four rows per thread per step, every row's loads issued before
    // the first is used and 16-bit keys kept packed until then, so that
    // enough bytes are in flight to cover the memory latency.
    const bool plain = DT != kF32 && !far_rot &&
                       !(ra.enabled && ra.window > 0 && (L - 1 - (jend - 1)) < ra.window);
    if constexpr (DT != kF32) {
        if (plain) {
            constexpr int RPT = 4;
            for (int32_t jb = jbeg; jb < jend; jb += RPT * rpb) {
                int32_t jr[RPT];
                bool valid[RPT];
                uint4 raw0[RPT], raw1[RPT];
#pragma unroll
                for (int u = 0; u < RPT; u++) {
                    jr[u] = jb + rl + u * rpb;
                    valid[u] = jr[u] < jend;
                    if (valid[u]) {
                        const typename Elem<DT>::T* kr =
                            reinterpret_cast<const typename Elem<DT>::T*>(keys) + (bh * ncap + jr[u]) * d;
                        raw0[u] = *reinterpret_cast<const uint4*>(kr + e0);
                        raw1[u] = *reinterpret_cast<const uint4*>(kr + e1);
                    }
                }
                float dot[RPT], nn[RPT];
#pragma unroll
                for (int u = 0; u < RPT; u++) {
                    dot[u] = 0.f;
                    nn[u] = 0.f;
                    if (!valid[u]) continue;
                    if constexpr (OUT >= 0) {
                        // the copy is the key itself (converted when OUT differs)
                        const int64_t row = bh * ncap + jr[u];
                        if constexpr (OUT == DT) {
                            typename Elem<DT>::T* ko = reinterpret_cast<typename Elem<DT>::T*>(kout) + row * d;
                            *reinterpret_cast<uint4*>(ko + e0) = raw0[u];
                            *reinterpret_cast<uint4*>(ko + e1) = raw1[u];
                        } else {
                            float v[8];
                            const typename Elem<DT>::T* a = reinterpret_cast<const typename Elem<DT>::T*>(&raw0[u]);
#pragma unroll
                            for (int k = 0; k < 8; k++) v[k] = to_f32<DT>(a[k]);
                            store8<OUT>(kout, row * d + e0, v);
                            const typename Elem<DT>::T* b = reinterpret_cast<const typename Elem<DT>::T*>(&raw1[u]);
#pragma unroll
                            for (int k = 0; k < 8; k++) v[k] = to_f32<DT>(b[k]);
                            store8<OUT>(kout, row * d + e1, v);
                        }
                    }
                    const typename Elem<DT>::T* a = reinterpret_cast<const typename Elem<DT>::T*>(&raw0[u]);
                    const typename Elem<DT>::T* b = reinterpret_cast<const typename Elem<DT>::T*>(&raw1[u]);
#pragma unroll
                    for (int k = 0; k < 8; k++) {
                        const float x = to_f32<DT>(a[k]);
                        dot[u] = fmaf(x, qv0[k], dot[u]);
                        nn[u] = fmaf(x, x, nn[u]);
                    }
#pragma unroll
                    for (int k = 0; k < 8; k++) {
                        const float x = to_f32<DT>(b[k]);
                        dot[u] = fmaf(x, qv1[k], dot[u]);
                        nn[u] = fmaf(x, x, nn[u]);
                    }
                }
                for (int m = lpr >> 1; m; m >>= 1) {
#pragma unroll
                    for (int u = 0; u < RPT; u++) {
                        dot[u] += __shfl_xor_sync(0xffffffffu, dot[u], m);
                        nn[u] += __shfl_xor_sync(0xffffffffu, nn[u], m);
                    }
                }
#pragma unroll
                for (int u = 0; u < RPT; u++)
                    if (valid[u] && lane == 0) {
                        const float kn = sqrtf(nn[u]);
                        scores[bh * ncap + jr[u]] = (kn > 0.f && qn > 0.f) ? dot[u] / (kn * qn) : 0.f;
                    }
            }
            return;
        }
    }
    // the loop bounds are uniform over the warp (the shuffles take it whole)
    for (int32_t jb = jbeg; jb < jend; jb += 2 * rpb) {
        int32_t jr[2] = {jb + rl, jb + rl + rpb};
        bool valid[2] = {jr[0] < jend, jr[1] < jend};
        float v0[2][8], v1[2][8];
#pragma unroll
        for (int u = 0; u < 2; u++)
            if (valid[u]) {
                const int64_t row = bh * ncap + jr[u];
                load8<DT>(keys, row * d + e0, v0[u]);
                load8<DT>(keys, row * d + e1, v1[u]);
            }
        float dot[2] = {0.f, 0.f}, nn[2] = {0.f, 0.f};
#pragma unroll
        for (int u = 0; u < 2; u++) {
            if (!valid[u]) continue;
            const int64_t row = bh * ncap + jr[u];
            if (ra.enabled) {
                const bool near = ra.window > 0 && (L - 1 - jr[u]) < ra.window;
                if (near || far_rot) {
                    float c[8], sn[8];
                    angles8<false>(near ? jr[u] : ra.far_offset, e0, ra, c, sn);
                    rotate8<false>(v0[u], v1[u], c, sn);
                }
            }
            if constexpr (OUT >= 0) {
                store8<OUT>(kout, row * d + e0, v0[u]);
                store8<OUT>(kout, row * d + e1, v1[u]);
            }
#pragma unroll
            for (int k = 0; k < 8; k++) {
                dot[u] = fmaf(v0[u][k], qv0[k], dot[u]);
                nn[u] = fmaf(v0[u][k], v0[u][k], nn[u]);
            }
#pragma unroll
            for (int k = 0; k < 8; k++) {
                dot[u] = fmaf(v1[u][k], qv1[k], dot[u]);
                nn[u] = fmaf(v1[u][k], v1[u][k], nn[u]);
            }
        }
        for (int m = lpr >> 1; m; m >>= 1) {
#pragma unroll
            for (int u = 0; u < 2; u++) {
                dot[u] += __shfl_xor_sync(0xffffffffu, dot[u], m);
                nn[u] += __shfl_xor_sync(0xffffffffu, nn[u], m);
            }
        }
#pragma unroll
        for (int u = 0; u < 2; u++)
            if (valid[u] && lane == 0) {
                const float kn = sqrtf(nn[u]);
                scores[bh * ncap + jr[u]] = (kn > 0.f && qn > 0.f) ? dot[u] / (kn * qn) : 0.f;
            }
    }
}

// Windowed RoPE alone over (chunk of kBhRows rows, (b, h)) blocks for the
// half-split pairing with d % 16 == 0: no thread walks the rows past a
// sequence's length.  A block whose rows are all far with no far rotation
// copies its rows (converted when the dtypes differ) four rows per thread
// per step, every row's loads issued before the first store, so that enough
// bytes are in flight to cover the memory latency; other blocks rotate row
// by row as windowed_rope_kernel does, with the same arithmetic.
template <int IN, int OUT>
__global__ void __launch_bounds__(kRopeThreads, 3)
windowed_rope_bh_kernel(const void* __restrict__ kin, void* __restrict__ kout, int32_t H,
                        int32_t ncap, int32_t d, const int32_t* __restrict__ len,
                        const RopeArgs ra) {
    const int lpr = d / 16;
    const int rpb = kRopeThreads / lpr;
    const int lane = threadIdx.x % lpr;
    const int rl = threadIdx.x / lpr;
    const int e0 = lane * 8;
    const int e1 = e0 + d / 2;
    const int64_t bh = blockIdx.y;
    const int32_t L = seq_len(len, (int32_t)(bh / H), ncap);
    const int32_t jbeg = blockIdx.x * kBhRows;
    if (jbeg >= L) return;  // uniform over the block
    const int32_t jend = min(jbeg + kBhRows, L);
    const bool far_rot = ra.enabled && ra.far_offset != 0;
    const bool plain = !far_rot && !(ra.enabled && ra.window > 0 && (L - 1 - (jend - 1)) < ra.window);
    if constexpr (IN != kF32) {
        if (plain) {
            constexpr int RPT = 4;
            using TI = typename Elem<IN>::T;
            for (int32_t jb = jbeg; jb < jend; jb += RPT * rpb) {
                int32_t jr[RPT];
                bool valid[RPT];
                uint4 raw0[RPT], raw1[RPT];
#pragma unroll
                for (int u = 0; u < RPT; u++) {
                    jr[u] = jb + rl + u * rpb;
                    valid[u] = jr[u] < jend;
                    if (valid[u]) {
                        const TI* kr = reinterpret_cast<const TI*>(kin) + (bh * ncap + jr[u]) * d;
                        raw0[u] = *reinterpret_cast<const uint4*>(kr + e0);
                        raw1[u] = *reinterpret_cast<const uint4*>(kr + e1);
                    }
                }
#pragma unroll
                for (int u = 0; u < RPT; u++) {
                    if (!valid[u]) continue;
                    const int64_t row = bh * ncap + jr[u];
                    if constexpr (OUT == IN) {
                        TI* ko = reinterpret_cast<TI*>(kout) + row * d;
                        *reinterpret_cast<uint4*>(ko + e0) = raw0[u];
                        *reinterpret_cast<uint4*>(ko + e1) = raw1[u];
                    } else {
                        float v[8];
                        const TI* a = reinterpret_cast<const TI*>(&raw0[u]);
#pragma unroll
                        for (int k = 0; k < 8; k++) v[k] = to_f32<IN>(a[k]);
                        store8<OUT>(kout, row * d + e0, v);
                        const TI* b = reinterpret_cast<const TI*>(&raw1[u]);
#pragma unroll
                        for (int k = 0; k < 8; k++) v[k] = to_f32<IN>(b[k]);
                        store8<OUT>(kout, row * d + e1, v);
                    }
                }
            }
            return;
        }
    }
    float fc[8], fs[8];
    if (far_rot) angles8<false>(ra.far_offset, e0, ra, fc, fs);
    for (int32_t jb = jbeg; jb < jend; jb += 2 * rpb) {
        int32_t jr[2] = {jb + rl, jb + rl + rpb};
        bool valid[2] = {jr[0] < jend, jr[1] < jend};
        float v0[2][8], v1[2][8];
#pragma unroll
        for (int u = 0; u < 2; u++)
            if (valid[u]) {
                const int64_t row = bh * ncap + jr[u];
                load8<IN>(kin, row * d + e0, v0[u]);
                load8<IN>(kin, row * d + e1, v1[u]);
            }
#pragma unroll
        for (int u = 0; u < 2; u++) {
            if (!valid[u]) continue;
            const int64_t row = bh * ncap + jr[u];
            if (ra.enabled) {
                const bool near = ra.window > 0 && (L - 1 - jr[u]) < ra.window;
                if (near) {
                    float c[8], sn[8];
                    angles8<false>(jr[u], e0, ra, c, sn);
                    rotate8<false>(v0[u], v1[u], c, sn);
                } else if (far_rot) {
                    rotate8<false>(v0[u], v1[u], fc, fs);
                }
            }
            store8<OUT>(kout, row * d + e0, v0[u]);
            store8<OUT>(kout, row * d + e1, v1[u]);
        }
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
    } else if (d % 16 == 0) {  // d <= kMaxD: d / 16 lanes per row fit a warp
        dim3 grid((unsigned)((s.Ncap + kBhRows - 1) / kBhRows), (unsigned)(s.B * s.H));
        windowed_rope_bh_kernel<IN, OUT><<<grid, kRopeThreads, 0, st>>>(
            kin, kout, (int32_t)s.H, (int32_t)s.Ncap, d, len, ra);
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
// The lpr lanes of a row (an aligned group of a warp: lpr is a power of two
// no larger than 32) each take 16 (or 8) of its elements; xor shuffles sum
// their partial dot and squared norm, and the group's first lane divides, so
// the square root and the division run once per row.  There are no block
// barriers: every warp streams on its own (with partials met in shared
// memory behind two block barriers per row the split of the decode workload
// took 1.37 ms against 1.22 ms; two rows in flight per lane group, at 79
// registers, took 1.53 ms).  Grid-stride over rows, with (bh, j) advanced by
// the stride without 64-bit divisions.
// OUT >= 0: the rotated rows are also stored in that dtype (the same values
// windowed_rope_kernel writes), so one pass over the keys serves both.
template <int DT, bool INTERLEAVED, int OUT>
__global__ void __launch_bounds__(kRopeThreads)
cosine_score_kernel(const void* __restrict__ keys, int64_t rows, int32_t H, int32_t ncap,
                    int32_t d, const int32_t* __restrict__ len, const RopeArgs ra,
                    const float* __restrict__ q, const float* __restrict__ qnorm,
                    float* __restrict__ scores, void* __restrict__ kout) {
    const int lpr = INTERLEAVED ? d / 8 : d / 16;
    const int rpb = kRopeThreads / lpr;
    const int lane = threadIdx.x & (lpr - 1);
    const int rl = threadIdx.x / lpr;
    const int e0 = lane * 8;
    const int e1 = e0 + d / 2;
    const int pair0 = INTERLEAVED ? e0 / 2 : e0;
    const bool far_rot = ra.enabled && ra.far_offset != 0;
    const int64_t stride = (int64_t)gridDim.x * rpb;
    const int64_t qs = stride / ncap;
    const int32_t rs = (int32_t)(stride - qs * ncap);
    int64_t bh = ((int64_t)blockIdx.x * rpb + rl) / ncap;
    int32_t j = (int32_t)(((int64_t)blockIdx.x * rpb + rl) - bh * ncap);
    // the loop bounds are uniform over the warp (the shuffles take it whole)
    for (int64_t base = (int64_t)blockIdx.x * rpb; base < rows; base += stride) {
        const int64_t row = base + rl;
        bool valid = row < rows;
        int32_t L = 0;
        if (valid) {
            L = seq_len(len, (int32_t)bh / H, ncap);
            valid = j < L;
        }
        float dot = 0.f, nn = 0.f;
        if (valid) {
            float v0[8], v1[8];
            load8<DT>(keys, row * d + e0, v0);
            if (!INTERLEAVED) load8<DT>(keys, row * d + e1, v1);
            if (ra.enabled) {
                const bool near = ra.window > 0 && (L - 1 - j) < ra.window;
                if (near || far_rot) {
                    float c[8], sn[8];
                    angles8<INTERLEAVED>(near ? j : ra.far_offset, pair0, ra, c, sn);
                    rotate8<INTERLEAVED>(v0, v1, c, sn);
                }
            }
            if constexpr (OUT >= 0) {
                store8<OUT>(kout, row * d + e0, v0);
                if (!INTERLEAVED) store8<OUT>(kout, row * d + e1, v1);
            }
            const float4* qa = reinterpret_cast<const float4*>(q + bh * d + e0);
            const float4 a0 = __ldg(qa), a1 = __ldg(qa + 1);
            const float qv0[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
#pragma unroll
            for (int k = 0; k < 8; k++) {
                dot = fmaf(v0[k], qv0[k], dot);
                nn = fmaf(v0[k], v0[k], nn);
            }
            if (!INTERLEAVED) {
                const float4* qb = reinterpret_cast<const float4*>(q + bh * d + e1);
                const float4 b0 = __ldg(qb), b1 = __ldg(qb + 1);
                const float qv1[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
                for (int k = 0; k < 8; k++) {
                    dot = fmaf(v1[k], qv1[k], dot);
                    nn = fmaf(v1[k], v1[k], nn);
                }
            }
        }
        for (int m = lpr >> 1; m; m >>= 1) {
            dot += __shfl_xor_sync(0xffffffffu, dot, m);
            nn += __shfl_xor_sync(0xffffffffu, nn, m);
        }
        if (valid && lane == 0) {
            const float qn = qnorm[bh];
            const float kn = sqrtf(nn);
            scores[row] = (kn > 0.f && qn > 0.f) ? dot / (kn * qn) : 0.f;
        }
        j += rs;
        bh += qs;
        if (j >= ncap) {
            j -= ncap;
            bh++;
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

constexpr int kSelCluster = 8;
constexpr int kSelCache = 16384;  // keys of a CTA's segment kept in shared memory (66 KB)

// Exclusive block-wide scan of one count per thread; returns the block total.
__device__ __forceinline__ int block_scan(int v, int& excl, int* warp_tot) {
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    int inc = v;
    for (int m = 1; m < 32; m <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, inc, m);
        if (lane >= m) inc += t;
    }
    if (lane == 31) warp_tot[w] = inc;
    __syncthreads();
    if (w == 0) {
        const int nw = blockDim.x >> 5;
        const int x = lane < nw ? warp_tot[lane] : 0;
        int wi = x;
        for (int m = 1; m < 32; m <<= 1) {
            const int t = __shfl_up_sync(0xffffffffu, wi, m);
            if (lane >= m) wi += t;
        }
        warp_tot[32 + lane] = wi - x;  // exclusive prefix of warp totals
        if (lane == 31) warp_tot[64] = wi;
    }
    __syncthreads();
    excl = warp_tot[32 + w] + inc - v;
    const int total = warp_tot[64];
    __syncthreads();
    return total;
}

// Exact top-n_r per (b, h) by radix select on order-preserving keys of the
// scores, ties on the threshold broken by lower index, then a stable
// two-sided compaction: retrieval rows ascending, then bulk rows ascending.
// One cluster of kCl CTAs per (b, h) (kSelCluster, or half of it when many
// (b, h) fill the GPU): each CTA owns a contiguous
// segment of the row (its keys cached in shared memory when they fit); the
// per-pass histograms and the compaction offsets are combined through
// distributed shared memory.  In the compaction each thread owns a contiguous
// run of the segment, so two block scans place every row.
template <int kSelThreads, int kCl>
__global__ void __cluster_dims__(kCl, 1, 1) __launch_bounds__(kSelThreads)
select_kernel(const float* __restrict__ scores, int32_t H, int32_t ncap,
              const int32_t* __restrict__ len, double fraction, int32_t* __restrict__ perm,
              int32_t* __restrict__ count) {
    namespace cg = cooperative_groups;
    cg::cluster_group cluster = cg::this_cluster();
    extern __shared__ uint32_t ks[];  // [kSelCache] ordered keys of the segment
    // per-pass histogram the cluster reads, alternating between two buffers:
    // the one a pass fills was last read by the other CTAs two passes
    // earlier, before the cluster barrier of the previous pass
    __shared__ uint32_t hist[2][256];
    // per-warp histograms: a pass's keys crowd into few digits, so each warp
    // counts on its own copy
    __shared__ uint32_t hist_w[kSelThreads / 32][256];
    __shared__ uint32_t tot[256];
    __shared__ int seg_counts[2];     // this CTA's rows above the threshold, equal to it
    __shared__ int warp_tot[65];
    __shared__ uint32_t sel_prefix, sel_need, sel_all;
    const int rank = (int)cluster.block_rank();
    const int bh = blockIdx.x / kCl;
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    const int32_t n = seq_len(len, bh / H, ncap);
    const float* s = scores + (int64_t)bh * ncap;
    int32_t* out = perm + (int64_t)bh * ncap;
    const double kd = ceil(fraction * (double)n);
    const int32_t k = kd < 0.0 ? 0 : (kd > (double)n ? n : (int32_t)kd);
    if (rank == 0 && tid == 0) count[bh] = k;
    const int32_t seg = (n + kCl - 1) / kCl;
    const int32_t lo = min(n, rank * seg), hi = min(n, lo + seg);
    const int32_t m = hi - lo;
    // the launch gives ks room for a segment of the capacity when that fits
    const bool cached = (ncap + kCl - 1) / kCl <= kSelCache;
    const bool partial = k > 0 && k < n;
    // key i of the segment sits at ks[i + i / 32], so the contiguous runs of
    // the compaction (thread t reads t * per + e) fall on distinct banks
    if (cached && partial)
        for (int i = tid; i < m; i += blockDim.x) ks[i + (i >> 5)] = ordered_key(s[lo + i]);
    auto key = [&](int32_t i) -> uint32_t {  // i relative to lo
        return cached ? ks[i + (i >> 5)] : ordered_key(s[lo + i]);
    };

    uint32_t prefix = 0, mask = 0, need = (uint32_t)k;
    if (partial) {
        int pass = 0;
        for (int shift = 24; shift >= 0; shift -= 8, pass++) {
            uint32_t* hb = hist[pass & 1];
            uint32_t* hw = &hist_w[0][0];
            for (int i = tid; i < (kSelThreads / 32) * 256; i += blockDim.x) hw[i] = 0;
            __syncthreads();
            for (int i = tid; i < m; i += blockDim.x) {
                const uint32_t u = key(i);
                if ((u & mask) == prefix) atomicAdd(&hist_w[w][(u >> shift) & 255u], 1u);
            }
            __syncthreads();
            if (tid < 256) {
                uint32_t t = 0;
#pragma unroll
                for (int ww = 0; ww < kSelThreads / 32; ww++) t += hist_w[ww][tid];
                hb[tid] = t;
            }
            cluster.sync();
            // every CTA sums the cluster's histograms and takes the same digit
            if (tid < 256) {
                uint32_t part[kCl];
#pragma unroll
                for (int r = 0; r < kCl; r++) part[r] = cluster.map_shared_rank(hb, r)[tid];
                uint32_t t = 0;
#pragma unroll
                for (int r = 0; r < kCl; r++) t += part[r];
                tot[tid] = t;
            }
            __syncthreads();
            if (w == 0) {
                // lane l holds digits 255 - 8l ... 248 - 8l (descending);
                // suffix sums from the top digit find the one holding the
                // need-th largest key
                uint32_t c[8], local = 0;
#pragma unroll
                for (int e = 0; e < 8; e++) {
                    c[e] = tot[255 - 8 * lane - e];
                    local += c[e];
                }
                uint32_t incl = local;
                for (int o = 1; o < 32; o <<= 1) {
                    const uint32_t t = __shfl_up_sync(0xffffffffu, incl, o);
                    if (lane >= o) incl += t;
                }
                const uint32_t before = incl - local;
                const bool here = before < need && incl >= need;
                if (here) {
                    uint32_t cum = before;
#pragma unroll
                    for (int e = 0; e < 8; e++) {
                        if (cum + c[e] >= need) {
                            sel_prefix = prefix | ((uint32_t)(255 - 8 * lane - e) << shift);
                            sel_need = need - cum;
                            // every key of the digit is taken: the later
                            // digits cannot change the set
                            sel_all = c[e] == need - cum;
                            break;
                        }
                        cum += c[e];
                    }
                }
            }
            __syncthreads();
            prefix = sel_prefix;
            need = sel_need;
            mask |= 255u << shift;
            // the same on every CTA of the cluster (the same totals), so they
            // leave after the same number of cluster barriers
            if (sel_all) break;
        }
    }
    // each thread owns the contiguous run [r0, r1) of the segment
    const int per = (m + (int)blockDim.x - 1) / (int)blockDim.x;
    const int r0 = min(m, tid * per), r1 = min(m, r0 + per);
    int gt_local = 0, eq_local = 0;
    // keys compare on the digits chosen so far (all of them unless the
    // selection ended early, when every key equal on them is taken)
    if (partial)
        for (int i = r0; i < r1; i++) {
            const uint32_t u = key(i) & mask;
            gt_local += u > prefix;
            eq_local += u == prefix;
        }
    int eq_excl, gt_excl;
    const int eq_cta = block_scan(eq_local, eq_excl, warp_tot);
    const int gt_cta = block_scan(gt_local, gt_excl, warp_tot);
    if (tid == 0) {
        seg_counts[0] = gt_cta;
        seg_counts[1] = eq_cta;
    }
    cluster.sync();
    int gt_before = 0, eq_before = 0;
    {
        int g[kCl], q[kCl];
#pragma unroll
        for (int r = 0; r < kCl; r++) {
            const int* other = cluster.map_shared_rank(seg_counts, r);
            g[r] = r < rank ? other[0] : 0;
            q[r] = r < rank ? other[1] : 0;
        }
#pragma unroll
        for (int r = 0; r < kCl; r++) {
            gt_before += g[r];
            eq_before += q[r];
        }
    }
    cluster.sync();  // the counts stay readable until every CTA has them
    // rows of this thread's run that are taken: all above the threshold, and
    // the equal ones among the first `need` equal rows in index order
    int eq_seen = eq_before + eq_excl;
    int take_local = 0;
    if (k == n) take_local = r1 - r0;
    else if (partial) {
        const int eq_take = max(0, min((int)need - eq_seen, eq_local));
        take_local = gt_local + eq_take;
    }
    int take_excl;
    block_scan(take_local, take_excl, warp_tot);
    const int take_before_seg = partial ? gt_before + min(eq_before, (int)need) : (k == n ? lo : 0);
    int pos_r = take_before_seg + take_excl;      // next retrieval slot
    int pos_b = k + (lo + r0 - pos_r);            // next bulk slot: rows before minus taken
    for (int i = r0; i < r1; i++) {
        bool take = k == n;
        if (partial) {
            const uint32_t u = key(i) & mask;
            const bool eq = u == prefix;
            take = u > prefix || (eq && eq_seen < (int)need);
            eq_seen += eq;
        }
        if (take) out[pos_r++] = lo + i;
        else out[pos_b++] = lo + i;
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

// dst[b, h, j] = src[b, h, j] for the retrieval rows j = perm[b, h, i],
// i < count[b, h], j < len[b].
__global__ void copy_retrieval_rows_kernel(const int32_t* __restrict__ src,
                                           int32_t* __restrict__ dst, int32_t H, int32_t ncap,
                                           const int32_t* __restrict__ len,
                                           const int32_t* __restrict__ perm,
                                           const int32_t* __restrict__ count) {
    const int bh = blockIdx.y;
    const int32_t L = seq_len(len, bh / H, ncap);
    const int32_t n = min(max(count[bh], 0), L);
    const int64_t base = (int64_t)bh * ncap;
    for (int32_t i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) {
        const int32_t j = perm[base + i];
        if (j >= 0 && j < L) dst[base + j] = src[base + j];
    }
}

template <int DT, int OUT>
cudaError_t score_dispatch(const void* keys, const Shape& s, const int32_t* len,
                           const RopeArgs& ra, const float* q, const float* qnorm,
                           float* scores, void* kout, cudaStream_t st) {
    const int64_t rows = s.B * s.H * s.Ncap;
    const int d = (int)s.d;
    // the score kernel reduces a row over lpr lanes with xor shuffles, so lpr
    // must be a power of two no larger than a warp
    const int lpr = ra.interleaved ? d / 8 : d / 16;
    const bool vec_ok = (ra.interleaved || d % 16 == 0) && lpr <= 32 && (lpr & (lpr - 1)) == 0;
    if (vec_ok && ra.interleaved) {
        cosine_score_kernel<DT, true, OUT><<<grid_for(rows, kRopeThreads / (d / 8)), kRopeThreads,
                                             0, st>>>(keys, rows, (int32_t)s.H, (int32_t)s.Ncap,
                                                      d, len, ra, q, qnorm, scores, kout);
        note_launches(1);
    } else if (vec_ok) {
        dim3 grid((unsigned)((s.Ncap + kBhRows - 1) / kBhRows), (unsigned)(s.B * s.H));
        cosine_score_bh_kernel<DT, OUT><<<grid, kRopeThreads, 0, st>>>(
            keys, (int32_t)s.H, (int32_t)s.Ncap, d, len, ra, q, qnorm, scores, kout);
        note_launches(1);
    } else {
        if (OUT >= 0) return cudaErrorNotSupported;  // the caller rotates in a pass of its own
        cosine_score_warp_kernel<DT><<<grid_for(rows, kRopeThreads / 32), kRopeThreads, 0, st>>>(
            keys, rows, (int32_t)s.H, (int32_t)s.Ncap, d, len, ra, q, qnorm, scores);
        note_launches(1);
    }
    return cudaGetLastError();
}

template <int DT>
cudaError_t score_dispatch_out(const void* keys, const Shape& s, const int32_t* len,
                               const RopeArgs& ra, const float* q, const float* qnorm,
                               float* scores, void* kout, int out_dt, cudaStream_t st) {
    switch (out_dt) {
        case -1: return score_dispatch<DT, -1>(keys, s, len, ra, q, qnorm, scores, nullptr, st);
        case kF32: return score_dispatch<DT, kF32>(keys, s, len, ra, q, qnorm, scores, kout, st);
        case kBF16: return score_dispatch<DT, kBF16>(keys, s, len, ra, q, qnorm, scores, kout, st);
        default: return score_dispatch<DT, kF16>(keys, s, len, ra, q, qnorm, scores, kout, st);
    }
}

// The RoPE window only, with the query: blocks (x, bh) of a (b, h) first
// form its query as prepare_query_kernel does (the first 128 threads, the
// same order of operations, so the values are the same) and block x = 0
// stores it; then each block takes window rows j in [len - W, len), lpr
// lanes per row as in cosine_score_kernel: the row rotated at its own
// position is stored in the keys' dtype (the values windowed_rope_kernel
// writes) and its cosine with the query goes to scores.  The rows outside
// the window are left to the pass over the stored keys, which copies them
// and scores them.
template <int DT, bool INTERLEAVED>
__global__ void __launch_bounds__(kRopeThreads)
window_score_kernel(const void* __restrict__ keys, const void* __restrict__ query, int32_t H,
                    int32_t ncap, int32_t d, int32_t win, const int32_t* __restrict__ len,
                    const RopeArgs ra, float* __restrict__ q_out, float* __restrict__ qnorm_out,
                    float* __restrict__ scores, void* __restrict__ kout) {
    __shared__ __align__(16) float qv[kMaxD];
    __shared__ Dot2 red[4];
    __shared__ float qn_s;
    __shared__ float2 part[kRopeThreads];
    const int bh = blockIdx.y;
    const int32_t L = seq_len(len, bh / H, ncap);
    const int tid = threadIdx.x;
    // ---- the query (threads 0..127)
    if (tid < 128) {
        if (query) {
            for (int i = tid; i < d; i += 128) qv[i] = load1<DT>(query, (int64_t)bh * d + i);
        } else if (L == 0) {
            for (int i = tid; i < d; i += 128) qv[i] = 0.f;
        } else {
            const int64_t row = ((int64_t)bh * ncap + (L - 1)) * d;
            for (int i = tid; i < d; i += 128) qv[i] = load1<DT>(keys, row + i);
        }
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
            a = qv[ia];
            bv = qv[ib];
        }
        __syncthreads();
        if (tid < half && pos != 0) {
            float sn, cs;
            rope_angle(pos, ra.omega_hi[tid], ra.omega_lo[tid], ra, sn, cs);
            qv[ia] = fmaf(a, cs, -__fmul_rn(bv, sn));
            qv[ib] = fmaf(a, sn, __fmul_rn(bv, cs));
        }
        __syncthreads();
    }
    if (tid < 128) {
        Dot2 acc;
        for (int i = tid; i < d; i += 128) {
            if (blockIdx.x == 0) q_out[(int64_t)bh * d + i] = qv[i];
            acc.add_prod(qv[i], qv[i]);
        }
        for (int m = 16; m; m >>= 1) acc.merge(shfl_xor(acc, m));
        if ((tid & 31) == 0) red[tid >> 5] = acc;
    }
    __syncthreads();
    if (tid == 0) {
        Dot2 t = red[0];
        for (int w = 1; w < 4; w++) t.merge(red[w]);
        qn_s = sqrtf(t.value());
        if (blockIdx.x == 0) qnorm_out[bh] = qn_s;
    }
    __syncthreads();
    const float qn = qn_s;

    // ---- the window rows of this block
    const int lpr = INTERLEAVED ? d / 8 : d / 16;
    const int rpb = kRopeThreads / lpr;
    const int lane = tid % lpr, rl = tid / lpr;
    const bool active = tid < rpb * lpr;
    const int e0 = lane * 8, e1 = e0 + d / 2;
    const int pair0 = INTERLEAVED ? e0 / 2 : e0;
    const int32_t j0 = L - win;  // window rows are j0 + i, i in [0, win), kept if j >= 0
    for (int base = blockIdx.x * rpb; base < win; base += gridDim.x * rpb) {
        const int32_t j = j0 + base + rl;
        const bool valid = active && base + rl < win && j >= 0 && j < L;
        const int64_t row = (int64_t)bh * ncap + j;
        float dot = 0.f, nn = 0.f;
        if (valid) {
            float v0[8], v1[8];
            load8<DT>(keys, row * d + e0, v0);
            if (!INTERLEAVED) load8<DT>(keys, row * d + e1, v1);
            const int32_t pos = rope_position(j, L - 1, ra);
            if (ra.enabled && pos != 0) {
                float c[8], sn[8];
                angles8<INTERLEAVED>(pos, pair0, ra, c, sn);
                rotate8<INTERLEAVED>(v0, v1, c, sn);
            }
            store8<DT>(kout, row * d + e0, v0);
            if (!INTERLEAVED) store8<DT>(kout, row * d + e1, v1);
#pragma unroll
            for (int k = 0; k < 8; k++) {
                dot = fmaf(v0[k], qv[e0 + k], dot);
                nn = fmaf(v0[k], v0[k], nn);
            }
            if (!INTERLEAVED) {
#pragma unroll
                for (int k = 0; k < 8; k++) {
                    dot = fmaf(v1[k], qv[e1 + k], dot);
                    nn = fmaf(v1[k], v1[k], nn);
                }
            }
        }
        part[tid] = make_float2(dot, nn);
        __syncthreads();
        if (tid < rpb) {
            const int32_t jj = j0 + base + tid;
            if (base + tid < win && jj >= 0 && jj < L) {
                float dd = 0.f, n2 = 0.f;
                for (int i = 0; i < lpr; i++) {
                    const float2 pp = part[tid * lpr + i];
                    dd += pp.x;
                    n2 += pp.y;
                }
                const float kn = sqrtf(n2);
                scores[(int64_t)bh * ncap + jj] = (kn > 0.f && qn > 0.f) ? dd / (kn * qn) : 0.f;
            }
        }
        __syncthreads();
    }
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

cudaError_t launch_window_scores(const void* keys, const void* query, int dt, const Shape& s,
                                 const int32_t* len, const RopeArgs& ra, float* q, float* qnorm,
                                 float* scores, void* kout, cudaStream_t st) {
    const int64_t nbh = s.B * s.H;
    const int64_t win = ra.enabled ? (ra.window < s.Ncap ? ra.window : s.Ncap) : 0;
    const int d = (int)s.d;
    if (nbh == 0) return cudaSuccess;
    if (d % 16 != 0 || d > kMaxD) return cudaErrorNotSupported;
    const bool il = ra.enabled && ra.interleaved;
    const int rpb = kRopeThreads / (il ? d / 8 : d / 16);
    int dev = 0, sms = 152;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    int64_t per = (win + rpb - 1) / rpb;
    const int64_t cap = (4 * (int64_t)sms + nbh - 1) / nbh;
    if (per > cap) per = cap;
    if (per < 1) per = 1;
    const dim3 g((unsigned)per, (unsigned)nbh);
#define A2ATS_WIN(DT, IL)                                                                      \
    window_score_kernel<DT, IL><<<g, kRopeThreads, 0, st>>>(keys, query, (int32_t)s.H,         \
                                                            (int32_t)s.Ncap, d, (int32_t)win,  \
                                                            len, ra, q, qnorm, scores, kout)
    if (dt == kBF16) {
        if (il) A2ATS_WIN(kBF16, true); else A2ATS_WIN(kBF16, false);
    } else if (dt == kF16) {
        if (il) A2ATS_WIN(kF16, true); else A2ATS_WIN(kF16, false);
    } else {
        if (il) A2ATS_WIN(kF32, true); else A2ATS_WIN(kF32, false);
    }
#undef A2ATS_WIN
    note_launches(1);
    return cudaGetLastError();
}

cudaError_t launch_cosine_scores(const void* keys, int dt, const Shape& s, const int32_t* len,
                                 const RopeArgs& ra, const float* q, const float* qnorm,
                                 float* scores, cudaStream_t st, void* kout, int out_dt) {
    if (s.B * s.H * s.Ncap == 0) return cudaSuccess;
    if (!kout) out_dt = -1;
    switch (dt) {
        case kF32: return score_dispatch_out<kF32>(keys, s, len, ra, q, qnorm, scores, kout, out_dt, st);
        case kBF16: return score_dispatch_out<kBF16>(keys, s, len, ra, q, qnorm, scores, kout, out_dt, st);
        default: return score_dispatch_out<kF16>(keys, s, len, ra, q, qnorm, scores, kout, out_dt, st);
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

cudaError_t launch_copy_retrieval_rows(const int32_t* src, int32_t* dst, const Shape& s,
                                       const int32_t* len, const int32_t* perm,
                                       const int32_t* count, cudaStream_t st) {
    const int64_t nbh = s.B * s.H;
    if (nbh == 0 || s.Ncap == 0) return cudaSuccess;
    const int64_t blocks = (s.Ncap + 255) / 256;
    dim3 g((unsigned)(blocks < 32 ? blocks : 32), (unsigned)nbh);
    copy_retrieval_rows_kernel<<<g, 256, 0, st>>>(src, dst, (int32_t)s.H, (int32_t)s.Ncap, len,
                                                  perm, count);
    note_launches(1);
    return cudaGetLastError();
}

cudaError_t launch_select(const float* scores, const Shape& s, const int32_t* len,
                          double fraction, int32_t* perm, int32_t* count, cudaStream_t st) {
    const int nbh = (int)(s.B * s.H);
    if (nbh == 0) return cudaSuccess;
    // 512 threads and clusters of kSelCluster CTAs for a few (b, h); with
    // many (a decode batch, more clusters than about four CTAs per SM), 256
    // threads and half the cluster, so fewer CTAs run the same chain of
    // barriers
    int dev = 0, sms = 152;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const bool few = (int64_t)nbh * kSelCluster <= 4 * (int64_t)sms;
    const int cl = few ? kSelCluster : kSelCluster / 2;
    const int64_t seg = (s.Ncap + cl - 1) / cl;
    const size_t smem = seg <= kSelCache ? sizeof(uint32_t) * (size_t)(seg + seg / 32 + 1) : 0;
    const int cache_bytes = (int)(sizeof(uint32_t) * (kSelCache + kSelCache / 32 + 1));
    cudaError_t e = cudaFuncSetAttribute(select_kernel<512, kSelCluster>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, cache_bytes);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(select_kernel<256, kSelCluster / 2>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, cache_bytes);
    if (e != cudaSuccess) return e;
    if (few)
        select_kernel<512, kSelCluster><<<nbh * kSelCluster, 512, smem, st>>>(
            scores, (int32_t)s.H, (int32_t)s.Ncap, len, fraction, perm, count);
    else
        select_kernel<256, kSelCluster / 2><<<nbh * (kSelCluster / 2), 256, smem, st>>>(
            scores, (int32_t)s.H, (int32_t)s.Ncap, len, fraction, perm, count);
    note_launches(1);
    return cudaGetLastError();
}

}  // namespace a2ats
