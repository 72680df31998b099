// split_static.cu -- the retrieval split with library-owned scratch.
//
// a2ats_select_retrieval_set needs scratch for the per-(b, h) query, its norm
// and one cosine per key, and normally takes it from a caller-supplied
// workspace.  Some callers cannot allocate device memory at all: code whose
// device memory is entirely reserved by another allocator (a caching
// allocator that has claimed the pool), or latency-critical paths that must
// never risk an allocation failure or its cost.  For them this file keeps the
// scratch in one fixed array that lives in the library's device image: every
// GPU that loads the library holds it (a few MB) until the process exits.
// Shapes beyond the array are refused; nothing is ever allocated.
#include <math.h>
#include <string.h>

#include <mutex>

#include "../../include/a2ats.h"
#include "kernels.cuh"

namespace a2ats {
namespace {

constexpr int64_t kStaticKeys = int64_t(1) << 20;  // B*H*Ncap cosines
constexpr int64_t kStaticHeads = 1024;             // B*H queries of up to kMaxD floats
constexpr int64_t kQOff = 0;
constexpr int64_t kQNormOff = kStaticHeads * kMaxD;
constexpr int64_t kScoreOff = kQNormOff + kStaticHeads + 64;  // 256-byte aligned start
constexpr int64_t kStaticFloats = kScoreOff + kStaticKeys;

static __device__ __align__(256) float g_split_scratch[kStaticFloats];

// Device address of g_split_scratch on each device, looked up once per device
// with that device current (the host-side symbol is not a device address).
std::mutex g_mu;
float* g_addr[256] = {nullptr};

cudaError_t static_scratch(float** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 256) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_addr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_split_scratch);
        if (e != cudaSuccess) return e;
        g_addr[dev] = static_cast<float*>(p);
    }
    *out = g_addr[dev];
    return cudaSuccess;
}

}  // namespace
}  // namespace a2ats

using namespace a2ats;

extern "C" int a2ats_select_retrieval_set_static(const void* keys, int32_t dtype, int64_t B,
                                                 int64_t H, int64_t Ncap, int64_t d,
                                                 const int32_t* len, const void* query,
                                                 double fraction,
                                                 const a2ats_rope_params* fused_rope,
                                                 int32_t* perm, int32_t* count, void* stream) {
    if (dtype != A2ATS_F32 && dtype != A2ATS_BF16 && dtype != A2ATS_F16) return A2ATS_ERR_DTYPE;
    if (B < 0 || H < 0 || Ncap < 0 || d < 8 || d > kMaxD || d % 8 != 0 ||
        Ncap >= (int64_t(1) << 24) || B * H > 65535)
        return A2ATS_ERR_SHAPE;
    if (!(fraction >= 0.0 && fraction <= 1.0)) return A2ATS_ERR_INVALID_ARG;
    if (B * H > kStaticHeads || B * H * Ncap > kStaticKeys) return A2ATS_ERR_CAPACITY;
    RopeArgs ra;
    memset(&ra, 0, sizeof(ra));
    if (fused_rope) {
        if (!(fused_rope->rope_base > 0.0) || !isfinite(fused_rope->rope_base))
            return A2ATS_ERR_INVALID_ARG;
        if (fused_rope->far_offset <= -(1 << 24) || fused_rope->far_offset >= (1 << 24))
            return A2ATS_ERR_INVALID_ARG;
        ra.enabled = 1;
        ra.window = fused_rope->window;
        ra.far_offset = fused_rope->far_offset;
        ra.interleaved = fused_rope->interleaved ? 1 : 0;
        const double two_pi = 6.283185307179586476925286766559;
        ra.two_pi_a = (float)two_pi;
        ra.two_pi_b = (float)(two_pi - (double)ra.two_pi_a);
        ra.two_pi_c = (float)(two_pi - (double)ra.two_pi_a - (double)ra.two_pi_b);
        ra.inv_2pi = (float)(1.0 / two_pi);
        for (int64_t i = 0; i < d / 2; i++) {
            const double om = pow(fused_rope->rope_base, -2.0 * (double)i / (double)d);
            ra.omega_hi[i] = (float)om;
            ra.omega_lo[i] = (float)(om - (double)ra.omega_hi[i]);
        }
    }
    if (B * H == 0) return A2ATS_OK;
    if (!count || (Ncap > 0 && (!keys || !perm))) return A2ATS_ERR_INVALID_ARG;
    if (((uintptr_t)keys & 15u) || ((uintptr_t)query & 15u) || ((uintptr_t)perm & 15u))
        return A2ATS_ERR_ALIGN;
    float* base = nullptr;
    cudaError_t e = static_scratch(&base);
    if (e != cudaSuccess) return A2ATS_ERR_CUDA;
    cudaStream_t s = (cudaStream_t)stream;
    const Shape sh{B, H, Ncap, d};
    // every scratch word the kernels read is written first in the same call,
    // so nothing has to be cleared between calls
    if (Ncap > 0) {
        e = launch_prepare_query(keys, query, dtype, sh, len, ra, base + kQOff, base + kQNormOff, s);
        if (e != cudaSuccess) return A2ATS_ERR_CUDA;
        e = launch_cosine_scores(keys, dtype, sh, len, ra, base + kQOff, base + kQNormOff,
                                 base + kScoreOff, s);
        if (e != cudaSuccess) return A2ATS_ERR_CUDA;
    }
    e = launch_select(base + kScoreOff, sh, len, fraction, perm, count, s);
    return e == cudaSuccess ? A2ATS_OK : A2ATS_ERR_CUDA;
}
