// common.cuh -- device helpers shared by the A2ATS kernels (sm_103a).
//
// Element access for the three storage dtypes, the windowed-RoPE rotation
// (deploy-preview "A2ATS-adapted" page, paper-fidelity section, Eq. 11-12),
// compensated fp32 arithmetic, and the launch-parameter structs the host side
// fills in.  GB300 runs fp64 at a small fraction of its fp32 rate, so every
// place that needs more than fp32 precision uses error-free transformations
// on fp32 pairs instead of doubles.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace a2ats {

constexpr int kF32 = 0, kBF16 = 1, kF16 = 2;
constexpr int kMaxD = 256;

// ---------------------------------------------------------------- dtypes --
template <int DT> struct Elem;
template <> struct Elem<kF32> { using T = float; static constexpr int kVec = 4; };
template <> struct Elem<kBF16> { using T = __nv_bfloat16; static constexpr int kVec = 8; };
template <> struct Elem<kF16> { using T = __half; static constexpr int kVec = 8; };

template <int DT>
__device__ __forceinline__ float to_f32(typename Elem<DT>::T v);
template <> __device__ __forceinline__ float to_f32<kF32>(float v) { return v; }
template <> __device__ __forceinline__ float to_f32<kBF16>(__nv_bfloat16 v) {
    return __bfloat162float(v);
}
template <> __device__ __forceinline__ float to_f32<kF16>(__half v) { return __half2float(v); }

template <int DT>
__device__ __forceinline__ typename Elem<DT>::T from_f32(float v);
template <> __device__ __forceinline__ float from_f32<kF32>(float v) { return v; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<kBF16>(float v) {
    return __float2bfloat16_rn(v);
}
template <> __device__ __forceinline__ __half from_f32<kF16>(float v) { return __float2half_rn(v); }

// Load n = Elem<DT>::kVec consecutive elements (16 bytes) as floats.
template <int DT>
__device__ __forceinline__ void load_vec(const void* base, int64_t elem_off, float* out) {
    constexpr int V = Elem<DT>::kVec;
    const uint4 raw = *reinterpret_cast<const uint4*>(
        reinterpret_cast<const typename Elem<DT>::T*>(base) + elem_off);
    const typename Elem<DT>::T* e = reinterpret_cast<const typename Elem<DT>::T*>(&raw);
#pragma unroll
    for (int i = 0; i < V; i++) out[i] = to_f32<DT>(e[i]);
}

template <int DT>
__device__ __forceinline__ void store_vec(void* base, int64_t elem_off, const float* in) {
    constexpr int V = Elem<DT>::kVec;
    uint4 raw;
    typename Elem<DT>::T* e = reinterpret_cast<typename Elem<DT>::T*>(&raw);
#pragma unroll
    for (int i = 0; i < V; i++) e[i] = from_f32<DT>(in[i]);
    *reinterpret_cast<uint4*>(reinterpret_cast<typename Elem<DT>::T*>(base) + elem_off) = raw;
}

template <int DT>
__device__ __forceinline__ float load1(const void* base, int64_t off) {
    return to_f32<DT>(reinterpret_cast<const typename Elem<DT>::T*>(base)[off]);
}

// ------------------------------------------------------- windowed RoPE --
// Per-call constants.  omega_i = rope_base^(-2i/d) is evaluated on the host in
// double and carried as an unevaluated pair hi + lo of floats.  2*pi is split
// into three floats (a exact to 24 bits, b the next 24, c the rest) so the
// angle p * omega_i can be reduced to [-pi, pi] without fp64: p * omega_hi is
// split exactly with an FMA, and n * a is subtracted exactly because both
// operands are multiples of 2^-22 (a lies in [4, 8), p * omega_hi is at least
// pi whenever n != 0).
struct RopeArgs {
    int32_t window;
    int32_t far_offset;
    int32_t interleaved;
    int32_t enabled;  // 0: keys are already rotated, apply nothing
    float inv_2pi, two_pi_a, two_pi_b, two_pi_c;
    float omega_hi[kMaxD / 2];
    float omega_lo[kMaxD / 2];
};

__device__ __forceinline__ void rope_angle(int32_t pos, float om_hi, float om_lo,
                                           const RopeArgs& ra, float& s, float& c) {
    const float pf = (float)pos;  // exact: positions are below 2^24
    const float ph = __fmul_rn(pf, om_hi);
    float pl = fmaf(pf, om_hi, -ph);      // exact low part of pf * om_hi
    pl = fmaf(pf, om_lo, pl);
    const float n = rintf(ph * ra.inv_2pi);
    float r = fmaf(-n, ra.two_pi_a, ph);  // exact (see above)
    r = fmaf(-n, ra.two_pi_b, r);
    r = __fadd_rn(r, fmaf(-n, ra.two_pi_c, pl));
    sincosf(r, &s, &c);
}

// Is row p near the decode position t (exact RoPE at p) or far (far_offset)?
__device__ __forceinline__ int32_t rope_position(int32_t p, int32_t t, const RopeArgs& ra) {
    const int32_t dist = t - p;
    const bool near = ra.window > 0 && dist >= 0 && dist < ra.window;
    return near ? p : ra.far_offset;
}

// Rotate a full row held in `v` (fp32, length d, in place) at position pos.
__device__ __forceinline__ void rope_row_inplace(float* v, int d, int32_t pos, const RopeArgs& ra) {
    const int half = d >> 1;
    for (int i = 0; i < half; i++) {
        float s, c;
        rope_angle(pos, ra.omega_hi[i], ra.omega_lo[i], ra, s, c);
        const int a = ra.interleaved ? 2 * i : i;
        const int b = ra.interleaved ? 2 * i + 1 : i + half;
        const float xa = v[a], xb = v[b];
        v[a] = fmaf(xa, c, -__fmul_rn(xb, s));
        v[b] = fmaf(xa, s, __fmul_rn(xb, c));
    }
}

// ------------------------------------------- compensated fp32 arithmetic --
// Error-free transformations (Knuth's TwoSum, FMA-based TwoProduct) and the
// Ogita-Rump-Oishi Dot2 accumulator.  The _rn intrinsics keep the compiler
// from contracting or reassociating them.
__device__ __forceinline__ void two_sum(float a, float b, float& s, float& e) {
    s = __fadd_rn(a, b);
    const float bp = __fsub_rn(s, a);
    e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bp)), __fsub_rn(b, bp));
}

struct Dot2 {
    float s = 0.f, c = 0.f;
    __device__ __forceinline__ void add_prod(float a, float b) {
        const float p = __fmul_rn(a, b);
        const float pe = fmaf(a, b, -p);
        float t, te;
        two_sum(s, p, t, te);
        s = t;
        c = __fadd_rn(c, __fadd_rn(pe, te));
    }
    __device__ __forceinline__ void add(float a) {
        float t, te;
        two_sum(s, a, t, te);
        s = t;
        c = __fadd_rn(c, te);
    }
    __device__ __forceinline__ void merge(const Dot2& o) {
        float t, te;
        two_sum(s, o.s, t, te);
        s = t;
        c = __fadd_rn(c, __fadd_rn(o.c, te));
    }
    __device__ __forceinline__ float value() const { return __fadd_rn(s, c); }
};

__device__ __forceinline__ Dot2 shfl_xor(const Dot2& v, int m) {
    Dot2 r;
    r.s = __shfl_xor_sync(0xffffffffu, v.s, m);
    r.c = __shfl_xor_sync(0xffffffffu, v.c, m);
    return r;
}

// Order-preserving map of a float to uint32 (larger float -> larger key),
// with -0 folded onto +0.
__device__ __forceinline__ uint32_t ordered_key(float f) {
    if (f == 0.f) f = 0.f;
    const uint32_t u = __float_as_uint(f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ int32_t seq_len(const int32_t* len, int b, int32_t ncap) {
    return len ? min(max(len[b], 0), ncap) : ncap;
}

}  // namespace a2ats
