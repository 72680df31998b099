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
#include <cuda.h>
#include <string.h>

#include <mutex>

#include "../../include/a2ats.h"
#include "entry.cuh"
#include "kernels.cuh"

namespace a2ats {
namespace {

constexpr int64_t kStaticKeys = int64_t(1) << 20;  // B*H*Ncap cosines
constexpr int64_t kStaticHeads = 1024;             // B*H queries of up to kMaxD floats
constexpr int64_t kQOff = 0;
constexpr int64_t kQNormOff = kStaticHeads * kMaxD;
constexpr int64_t kScoreOff = kQNormOff + kStaticHeads + 64;  // 256-byte aligned start
constexpr int64_t kStaticFloats = kScoreOff + kStaticKeys;
static_assert(kQNormOff >= kQOff + kStaticHeads * kMaxD, "queries overlap their norms");
static_assert(kScoreOff >= kQNormOff + kStaticHeads, "norms overlap the scores");
static_assert((kQNormOff * sizeof(float)) % 256 == 0, "norms start 256-byte aligned");
static_assert((kScoreOff * sizeof(float)) % 256 == 0, "scores start 256-byte aligned");

static __device__ __align__(256) float g_split_scratch[kStaticFloats];

// Device address of g_split_scratch on each device, looked up with that
// device current (the host-side symbol is not a device address).  It is
// cached with the id of the context it was taken in and looked up again
// when the device's current context differs (after cudaDeviceReset the
// module is loaded anew, possibly at another address).
typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);

std::mutex g_mu;
float* g_addr[256] = {nullptr};
unsigned long long g_ctx[256] = {0};

// The current context's unique id, or 0 when it cannot be read.
unsigned long long current_context_id() {
    static CtxGetCurrentFn get_current = nullptr;
    static CtxGetIdFn get_id = nullptr;
    static bool looked = false;
    if (!looked) {
        looked = true;
        cudaDriverEntryPointQueryResult qr;
        void* f = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault,
                                             &qr) == cudaSuccess &&
            qr == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<CtxGetCurrentFn>(f);
        f = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &qr) ==
                cudaSuccess &&
            qr == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<CtxGetIdFn>(f);
    }
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || !ctx) return 0;
    if (get_id(ctx, &id) != CUDA_SUCCESS) return 0;
    return id;
}

cudaError_t static_scratch(float** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 256) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_mu);
    unsigned long long id = current_context_id();
    if (!g_addr[dev] || id == 0 || id != g_ctx[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_split_scratch);
        if (e != cudaSuccess) return e;
        g_addr[dev] = static_cast<float*>(p);
        // the lookup made the device's primary context current if it was not
        g_ctx[dev] = id ? id : current_context_id();
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
    // the checks of a2ats_select_retrieval_set, then the array's limits
    if (!dtype_ok(dtype)) return A2ATS_ERR_DTYPE;
    int st = check_shape(B, H, Ncap, d);
    if (st) return st;
    if (!unit_interval(fraction)) return A2ATS_ERR_INVALID_ARG;
    RopeArgs ra;
    if ((st = make_rope(fused_rope, d, ra))) return st;
    if (B * H > kStaticHeads || B * H * Ncap > kStaticKeys) return A2ATS_ERR_CAPACITY;
    if (B * H == 0) return A2ATS_OK;
    if (!count || (Ncap > 0 && (!keys || !perm))) return A2ATS_ERR_INVALID_ARG;
    if (((uintptr_t)keys & 15u) || ((uintptr_t)query & 15u) || ((uintptr_t)perm & 15u))
        return A2ATS_ERR_ALIGN;
    float* base = nullptr;
    cudaError_t e = static_scratch(&base);
    if (e != cudaSuccess) return cuda_fail(e);
    cudaStream_t s = (cudaStream_t)stream;
    const Shape sh{B, H, Ncap, d};
    // every scratch word the kernels read is written first in the same call,
    // so nothing has to be cleared between calls
    if (Ncap > 0) {
        e = launch_prepare_query(keys, query, dtype, sh, len, ra, base + kQOff, base + kQNormOff, s);
        if (e != cudaSuccess) return cuda_fail(e);
        e = launch_cosine_scores(keys, dtype, sh, len, ra, base + kQOff, base + kQNormOff,
                                 base + kScoreOff, s);
        if (e != cudaSuccess) return cuda_fail(e);
    }
    e = launch_select(base + kScoreOff, sh, len, fraction, perm, count, s);
    return e == cudaSuccess ? A2ATS_OK : cuda_fail(e);
}
