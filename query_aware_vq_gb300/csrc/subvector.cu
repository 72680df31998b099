// subvector.cu -- sub-vector (product) VQ of keys and values (sm_103a).
//
// v0.39.0 page "A2ATS-adapted -- Windowed RoPE + Query-Aware Retrieval VQ",
// configuration (a2ats_sub_dim = 8, a2ats_codebook_bits = 8) and "How it
// works" steps 2 and 5: a token of width d is d / sub_dim sub-vectors, each
// coded by its nearest entry of a per-head table of K sub_dim-wide
// centroids.  The retrieval tokens' sub-vectors take the H-weighted rule
// (API page, a2ats_h_weighted_assignment, through the Cholesky identity
// |x L - c L|^2), the others and the values plain nearest-centroid VQ.
//
//   mark_retrieval_kernel    one byte per token: 1 on the retrieval side of
//                            the split (perm[:count]), 0 on the bulk side
//   subvector_assign_kernel  one thread per sub-vector: both tables (c and
//                            c L) and L sit in shared memory; a retrieval
//                            sub-vector is moved to z = x L (compensated
//                            dot products), then the direct fp32 distance
//                            sum_a (z_a - t_a)^2 to every table entry,
//                            ties to the lower index.
//
//   subvector_blend_kernel   the same walk for the cosine blend (API page,
//                            a2ats_query_aware_assignment), the rule the
//                            page's wrapper takes when no calibrated H is
//                            given: on a retrieval token, sub-vector g with
//                            the query's slice g, e_k = |x_g - c_k|^2,
//                            m = max_k e_k, score_k = -beta e_k / m +
//                            (1 - beta) cos(q_g, c_k), argmax (lowest k on
//                            ties); elsewhere (and for beta = 1) plain VQ.
//
// The direct distance of a sub_dim-wide difference has a relative error
// below (sub_dim + 2) 2^-24, so a code can differ from the exact argmin only
// where the two best distances are that close.
#include "kernels.cuh"

namespace a2ats {
namespace {

constexpr int kSvThreads = 256;

__global__ void mark_retrieval_kernel(const int32_t* __restrict__ perm,
                                      const int32_t* __restrict__ count,
                                      const int32_t* __restrict__ len, int32_t H, int64_t BH,
                                      int64_t ncap, uint8_t* __restrict__ mark) {
    const int64_t total = BH * ncap;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t bh = i / ncap, pos = i - bh * ncap;
        const int32_t n = seq_len(len, (int)(bh / H), (int32_t)ncap);
        if (pos >= n) continue;
        const int32_t j = perm[i];
        if (j < 0 || j >= n) continue;  // not a split of this length: nothing to mark
        mark[bh * ncap + j] = pos < count[bh] ? 1 : 0;
    }
}

// Block (x, bh) walks the sub-vectors r = token * G + g of (b, h) with a
// grid stride.  Shared memory: the plain table [K][S], then (with L) the
// table c L [K][S] and L [S][S].
template <int DT, int S>
__global__ void __launch_bounds__(kSvThreads, 2)
subvector_assign_kernel(const void* __restrict__ x, int32_t H, int64_t ncap, int32_t d,
                        const int32_t* __restrict__ len, const float* __restrict__ tab_plain,
                        const float* __restrict__ tab_weighted, const float* __restrict__ Lc,
                        const uint8_t* __restrict__ mark, int32_t K,
                        int32_t* __restrict__ codes) {
    extern __shared__ __align__(16) float sv_smem[];
    constexpr int V = Elem<DT>::kVec;
    const int64_t bh = blockIdx.y;
    const int b = (int)(bh / H), h = (int)(bh % H);
    const int KS = K * S;
    float* plain = sv_smem;
    float* weighted = sv_smem + KS;
    float* Ls = sv_smem + 2 * KS;
    for (int i = threadIdx.x; i < KS; i += blockDim.x) plain[i] = tab_plain[(int64_t)h * KS + i];
    if (Lc) {
        for (int i = threadIdx.x; i < KS; i += blockDim.x)
            weighted[i] = tab_weighted[(int64_t)h * KS + i];
        for (int i = threadIdx.x; i < S * S; i += blockDim.x)
            Ls[i] = Lc[(int64_t)h * S * S + i];
    }
    __syncthreads();
    const int G = d / S;
    const int64_t rows = (int64_t)seq_len(len, b, (int32_t)ncap) * G;
    for (int64_t r = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; r < rows;
         r += (int64_t)gridDim.x * blockDim.x) {
        const int64_t j = r / G;
        const int g = (int)(r - j * G);
        float v[S];
        const int64_t off = (bh * ncap + j) * d + (int64_t)g * S;
#pragma unroll
        for (int a = 0; a < S; a += V) load_vec<DT>(x, off + a, v + a);
        const bool use_l = Lc != nullptr && (mark == nullptr || mark[bh * ncap + j] != 0);
        const float* tab = use_l ? weighted : plain;
        if (use_l) {
            float z[S];
#pragma unroll
            for (int c = 0; c < S; c++) {
                Dot2 acc;
#pragma unroll
                for (int a = c; a < S; a++) acc.add_prod(v[a], Ls[a * S + c]);
                z[c] = acc.value();
            }
#pragma unroll
            for (int a = 0; a < S; a++) v[a] = z[a];
        }
        float best = __int_as_float(0x7f800000);
        int32_t bj = 0;
        for (int k = 0; k < K; k++) {
            const float4* t4 = reinterpret_cast<const float4*>(tab + k * S);
            float dist = 0.f;
#pragma unroll
            for (int q = 0; q < S / 4; q++) {
                const float4 t = t4[q];
                const float e0 = v[4 * q] - t.x, e1 = v[4 * q + 1] - t.y;
                const float e2 = v[4 * q + 2] - t.z, e3 = v[4 * q + 3] - t.w;
                dist = fmaf(e0, e0, dist);
                dist = fmaf(e1, e1, dist);
                dist = fmaf(e2, e2, dist);
                dist = fmaf(e3, e3, dist);
            }
            if (dist < best) {
                best = dist;
                bj = k;
            }
        }
        codes[(bh * ncap + j) * G + g] = bj;
    }
}

template <int DT, int S>
cudaError_t launch_sv(const void* x, const Shape& s, const int32_t* len, const float* tab_plain,
                      const float* tab_weighted, const float* Lc, const uint8_t* mark, int64_t K,
                      int32_t* codes, cudaStream_t st) {
    const size_t smem = sizeof(float) * (size_t)((Lc ? 2 : 1) * K * S + (Lc ? S * S : 0));
    cudaError_t e = cudaFuncSetAttribute(subvector_assign_kernel<DT, S>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    int dev = 0, sms = 148;
    if (cudaGetDevice(&dev) == cudaSuccess)
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int64_t BH = s.B * s.H;
    const int64_t rows = s.Ncap * (s.d / S);
    int64_t per = (rows + kSvThreads - 1) / kSvThreads;
    const int64_t cap = (8 * (int64_t)sms + BH - 1) / BH;  // about 8 blocks per SM in all
    if (per > cap) per = cap;
    if (per < 1) per = 1;
    dim3 grid((unsigned)per, (unsigned)BH);
    subvector_assign_kernel<DT, S><<<grid, kSvThreads, smem, st>>>(
        x, (int32_t)s.H, s.Ncap, (int32_t)s.d, len, tab_plain, tab_weighted, Lc, mark,
        (int32_t)K, codes);
    note_launches(1);
    return cudaGetLastError();
}

template <int DT, int S>
__global__ void __launch_bounds__(kSvThreads, 2)
subvector_blend_kernel(const void* __restrict__ x, int32_t H, int64_t ncap, int32_t d,
                       const int32_t* __restrict__ len, const float* __restrict__ tab,
                       const float* __restrict__ cnorm, const void* __restrict__ query,
                       float beta, const uint8_t* __restrict__ mark, int32_t K,
                       int32_t* __restrict__ codes) {
    extern __shared__ __align__(16) float sv_smem[];
    constexpr int V = Elem<DT>::kVec;
    const int64_t bh = blockIdx.y;
    const int b = (int)(bh / H), h = (int)(bh % H);
    const int KS = K * S;
    float* table = sv_smem;    // [K][S]
    float* cn = sv_smem + KS;  // [K] |c_k|
    for (int i = threadIdx.x; i < KS; i += blockDim.x) table[i] = tab[(int64_t)h * KS + i];
    for (int i = threadIdx.x; i < K; i += blockDim.x) cn[i] = cnorm[(int64_t)h * K + i];
    __syncthreads();
    const int G = d / S;
    const int32_t n = seq_len(len, b, (int32_t)ncap);
    const int64_t rows = (int64_t)n * G;
    for (int64_t r = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; r < rows;
         r += (int64_t)gridDim.x * blockDim.x) {
        const int64_t j = r / G;
        const int g = (int)(r - j * G);
        float v[S];
#pragma unroll
        for (int a = 0; a < S; a += V) load_vec<DT>(x, (bh * ncap + j) * d + (int64_t)g * S + a, v + a);
        const bool blend = beta < 1.f && (mark == nullptr || mark[bh * ncap + j] != 0);
        float emax = 0.f;
        float best = blend ? -__int_as_float(0x7f800000) : __int_as_float(0x7f800000);
        int32_t bj = 0;
        // pass 0: the largest distance (blend only); pass 1: the decision
        for (int pass = blend ? 0 : 1; pass < 2; pass++) {
            float qv[S];
            float qn = 0.f;
            if (blend && pass == 1) {
                // the query's slice g: the given query, or the row at t = n - 1
                const void* src = query ? query : x;
                const int64_t qoff = query ? bh * d + (int64_t)g * S
                                           : (bh * ncap + (n - 1)) * d + (int64_t)g * S;
#pragma unroll
                for (int a = 0; a < S; a += V) load_vec<DT>(src, qoff + a, qv + a);
                Dot2 qq;
#pragma unroll
                for (int a = 0; a < S; a++) qq.add_prod(qv[a], qv[a]);
                qn = sqrtf(qq.value());
            }
            for (int k = 0; k < K; k++) {
                const float4* t4 = reinterpret_cast<const float4*>(table + k * S);
                float dist = 0.f;
#pragma unroll
                for (int q = 0; q < S / 4; q++) {
                    const float4 t = t4[q];
                    const float e0 = v[4 * q] - t.x, e1 = v[4 * q + 1] - t.y;
                    const float e2 = v[4 * q + 2] - t.z, e3 = v[4 * q + 3] - t.w;
                    dist = fmaf(e0, e0, dist);
                    dist = fmaf(e1, e1, dist);
                    dist = fmaf(e2, e2, dist);
                    dist = fmaf(e3, e3, dist);
                }
                if (!blend) {
                    if (dist < best) {
                        best = dist;
                        bj = k;
                    }
                    continue;
                }
                if (pass == 0) {
                    emax = fmaxf(emax, dist);
                    continue;
                }
                Dot2 dq;
#pragma unroll
                for (int a = 0; a < S; a++) dq.add_prod(qv[a], table[k * S + a]);
                const float ck = cn[k];
                const float cosv = (qn > 0.f && ck > 0.f) ? dq.value() / (qn * ck) : 0.f;
                const float err = emax > 0.f ? dist / emax : 0.f;
                const float sc = fmaf(-beta, err, (1.f - beta) * cosv);
                if (sc > best) {
                    best = sc;
                    bj = k;
                }
            }
        }
        codes[(bh * ncap + j) * G + g] = bj;
    }
}

template <int DT, int S>
cudaError_t launch_sv_blend(const void* x, const Shape& s, const int32_t* len, const float* tab,
                            const float* cnorm, const void* query, float beta,
                            const uint8_t* mark, int64_t K, int32_t* codes, cudaStream_t st) {
    const size_t smem = sizeof(float) * (size_t)(K * S + K);
    cudaError_t e = cudaFuncSetAttribute(subvector_blend_kernel<DT, S>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    int dev = 0, sms = 148;
    if (cudaGetDevice(&dev) == cudaSuccess)
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int64_t BH = s.B * s.H;
    const int64_t rows = s.Ncap * (s.d / S);
    int64_t per = (rows + kSvThreads - 1) / kSvThreads;
    const int64_t cap = (8 * (int64_t)sms + BH - 1) / BH;
    if (per > cap) per = cap;
    if (per < 1) per = 1;
    dim3 grid((unsigned)per, (unsigned)BH);
    subvector_blend_kernel<DT, S><<<grid, kSvThreads, smem, st>>>(
        x, (int32_t)s.H, s.Ncap, (int32_t)s.d, len, tab, cnorm, query, beta, mark, (int32_t)K,
        codes);
    note_launches(1);
    return cudaGetLastError();
}

}  // namespace

int64_t subvector_table_limit() { return 8192; }

cudaError_t launch_subvector_blend(const void* x, int dt, const Shape& s, const int32_t* len,
                                   int64_t sub_dim, const float* tab, const float* cnorm,
                                   const void* query, float beta, const uint8_t* mark, int64_t K,
                                   int32_t* codes, cudaStream_t st) {
    if (s.B * s.H * s.Ncap == 0) return cudaSuccess;
#define A2ATS_SVB(DTV, SV) \
    return launch_sv_blend<DTV, SV>(x, s, len, tab, cnorm, query, beta, mark, K, codes, st)
    if (sub_dim == 8) {
        if (dt == kF32) A2ATS_SVB(kF32, 8);
        if (dt == kBF16) A2ATS_SVB(kBF16, 8);
        A2ATS_SVB(kF16, 8);
    }
    if (dt == kF32) A2ATS_SVB(kF32, 16);
    if (dt == kBF16) A2ATS_SVB(kBF16, 16);
    A2ATS_SVB(kF16, 16);
#undef A2ATS_SVB
}

cudaError_t launch_mark_retrieval(const int32_t* perm, const int32_t* count, const int32_t* len,
                                  const Shape& s, uint8_t* mark, cudaStream_t st) {
    const int64_t total = s.B * s.H * s.Ncap;
    if (total == 0) return cudaSuccess;
    const int64_t blocks = (total + 255) / 256;
    mark_retrieval_kernel<<<(unsigned)(blocks < 4096 ? blocks : 4096), 256, 0, st>>>(
        perm, count, len, (int32_t)s.H, s.B * s.H, s.Ncap, mark);
    note_launches(1);
    return cudaGetLastError();
}

cudaError_t launch_subvector_assign(const void* x, int dt, const Shape& s, const int32_t* len,
                                    int64_t sub_dim, const float* tab_plain,
                                    const float* tab_weighted, const float* Lc,
                                    const uint8_t* mark, int64_t K, int32_t* codes,
                                    cudaStream_t st) {
    if (s.B * s.H * s.Ncap == 0) return cudaSuccess;
#define A2ATS_SV(DTV, SV) \
    return launch_sv<DTV, SV>(x, s, len, tab_plain, tab_weighted, Lc, mark, K, codes, st)
    if (sub_dim == 8) {
        if (dt == kF32) A2ATS_SV(kF32, 8);
        if (dt == kBF16) A2ATS_SV(kBF16, 8);
        A2ATS_SV(kF16, 8);
    }
    if (dt == kF32) A2ATS_SV(kF32, 16);
    if (dt == kBF16) A2ATS_SV(kBF16, 16);
    A2ATS_SV(kF16, 16);
#undef A2ATS_SV
}

}  // namespace a2ats
