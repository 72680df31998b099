// assign_tc.cu -- nearest-centroid assignment as a tensor-core contraction.
//
// API page, a2ats_h_weighted_assignment: argmin_j (k - c_j) H (k - c_j)^T with
// H = L L^T (paper Eq. 14-18).  Expanding the square,
//     argmin_j |kL - c_jL|^2 = argmax_j  k . chat_j - |c_j L|^2 / 2,
//     chat_j = c_j L L^T,
// so the per-row transform z = kL is folded into a per-head transform of the
// codebook, and the row side of the contraction is the stored key itself (for
// every key outside the RoPE window, whose rotation is the one shared far
// rotation, folded into chat as well).  The keys are 16-bit floats, so the
// products are exact when chat is split into 16-bit planes
// chat = P0 + P1 + P2 (bf16: 3 planes hold an fp32 exactly; fp16: 2 planes
// give 22 bits, with a per-head power-of-two scale); plain VQ on a 16-bit
// codebook needs one plane.  Each plane is one more pass of tcgen05.mma into
// the same TMEM accumulator.
//
// Kernel layout (one persistent CTA per SM, 10 warps):
//   warp 0     TMA producer: the 128-row key tile once per tile (kept for all
//              centroids), then the codebook in 256 x 64-element stages;
//   warp 1     TMEM allocation and tcgen05.mma issue (128 x 256 x 16,
//              bf16/fp16 -> fp32), two accumulators of 256 columns so the
//              epilogue of one centroid chunk overlaps the MMAs of the next;
//   warps 2-9  epilogue: tcgen05.ld of the accumulator, v = acc - |c'|^2/2,
//              branch-free top-2 per row with the column index carried in the
//              5 low mantissa bits, and a rigorous error bound: rows whose top
//              two are closer than the bound, and rows inside the RoPE window,
//              go to the exact SIMT kernel through a list.
// Every mbarrier wait is bounded; on time-out the kernel records an error
// code and leaves.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <float.h>

#include "kernels.cuh"

namespace a2ats {
namespace tc {

constexpr int BM = 128;   // rows per tile (UMMA M)
constexpr int BN = 256;   // centroids per accumulator (UMMA N)
constexpr int BK = 64;    // 16-bit elements per 128-byte swizzle atom
constexpr int kEpiWarps = 8;
constexpr int kThreads = 64 + 32 * kEpiWarps;
constexpr uint64_t kWaitNs = 2000000000ull;  // every mbarrier wait gives up after 2 s

struct Params {
    int32_t H, ncap, d, K, P;
    int32_t num_bh, tiles_per_bh, nchunks;
    const int32_t* len;        // [B] or null
    const int32_t* count;      // compact mode: rows per (b, h); null = natural mode
    const int32_t* row_map;    // compact mode: original row of each compact row
    const uint8_t* skip;       // rows to leave untouched (bulk mode), or null
    int32_t window;            // rows with t - j < window go to the exact list
    const float* half_norm;    // [H, K]
    const float* head;         // [H, 4]: max |chat_j|, max h_j, 1/scale, abs error
    float err_coef;            // relative error of the contraction (see host)
    int32_t* codes;            // [num_bh * ncap]
    int64_t* exact_list;       // rows for the exact kernel
    int32_t* exact_count;
    int32_t* status;           // 0, or the code of a timed-out wait
};

// ------------------------------------------------------------ PTX helpers --
__device__ __forceinline__ uint32_t su32(const void* p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void mbar_init(uint64_t* b, uint32_t n) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(su32(b)), "r"(n) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* b, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(su32(b)),
                 "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* b) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(su32(b)) : "memory");
}
__device__ __forceinline__ bool mbar_try(uint64_t* b, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(su32(b)), "r"(parity)
        : "memory");
    return ok != 0;
}
__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
    return t;
}
// Bounded wait: false (and an error code in *status) after kWaitNs.
__device__ __forceinline__ bool mbar_wait(uint64_t* b, uint32_t parity, int32_t* status,
                                          int code) {
    if (mbar_try(b, parity)) return true;
    const uint64_t t0 = global_ns();
    for (uint32_t i = 1;; i++) {
        if (mbar_try(b, parity)) return true;
        if ((i & 255u) == 0 && global_ns() - t0 > kWaitNs) break;
    }
    atomicCAS(status, 0, code);
    return false;
}
__device__ __forceinline__ void tma_2d(void* dst, const CUtensorMap* m, uint64_t* bar, int x,
                                       int y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4}], [%2];" ::"r"(su32(dst)),
        "l"(reinterpret_cast<uint64_t>(m)), "r"(su32(bar)), "r"(x), "r"(y)
        : "memory");
}
__device__ __forceinline__ void tma_3d(void* dst, const CUtensorMap* m, uint64_t* bar, int x,
                                       int y, int z) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(su32(dst)),
        "l"(reinterpret_cast<uint64_t>(m)), "r"(su32(bar)), "r"(x), "r"(y), "r"(z)
        : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
            su32(bar))
        : "memory");
}
__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                       uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// Shared-memory matrix descriptor: K-major operand in the 128-byte swizzled
// layout TMA writes (8-row groups 1024 bytes apart), descriptor version 1.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
    d |= (uint64_t)1u << 16;            // leading offset: unused by this layout
    d |= (uint64_t)(1024u >> 4) << 32;  // stride offset between 8-row groups
    d |= (uint64_t)1u << 46;            // descriptor version
    d |= (uint64_t)2u << 61;            // 128-byte swizzle
    return d;
}
#define A2ATS_TMEM_LD32(taddr, r)                                                               \
    asm volatile(                                                                               \
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, " \
        "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, " \
        "%28, %29, %30, %31}, [%32];"                                                           \
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),  \
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),           \
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),        \
          "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),        \
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),        \
          "=r"(r[31])                                                                           \
        : "r"(taddr))

__device__ __forceinline__ void tmem_wait_ld() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Top two of a 32-value chunk by a merge tree of (max, second) pairs.
__device__ __forceinline__ void top2_32(const float* k, float& t1, float& t2) {
    float hi[16], lo[16];
#pragma unroll
    for (int i = 0; i < 16; i++) {
        hi[i] = fmaxf(k[2 * i], k[2 * i + 1]);
        lo[i] = fminf(k[2 * i], k[2 * i + 1]);
    }
#pragma unroll
    for (int w = 8; w >= 1; w >>= 1) {
#pragma unroll
        for (int i = 0; i < w; i++) {
            const float h = fmaxf(hi[i], hi[i + w]);
            const float l = fmaxf(fminf(hi[i], hi[i + w]), fmaxf(lo[i], lo[i + w]));
            hi[i] = h;
            lo[i] = l;
        }
    }
    t1 = hi[0];
    t2 = lo[0];
}

struct TileInfo {
    int32_t bh, r0, nvalid;
    bool skip;
};

__device__ __forceinline__ TileInfo tile_info(const Params& p, int t) {
    TileInfo ti;
    ti.bh = t / p.tiles_per_bh;
    ti.r0 = (t % p.tiles_per_bh) * BM;
    ti.nvalid = seq_len(p.len, ti.bh / p.H, p.ncap);
    if (p.count) ti.nvalid = min(max(p.count[ti.bh], 0), ti.nvalid);
    ti.skip = ti.r0 >= ti.nvalid;
    return ti;
}

template <int DK, int AST, int BST>
struct Smem {
    static constexpr int kA = BM * 128;        // bytes of one 64-element k-block of A
    static constexpr int kB = BN * 128;        // bytes of one B stage
    static constexpr int kABytes = AST * DK * kA;
    static constexpr int kBBytes = BST * kB;
    static constexpr int kBarOff = kABytes + kBBytes;
    static constexpr int kBars = 2 * AST + 2 * BST + 6;
    static constexpr int kMergeOff = kBarOff + kBars * 8 + 16;
    static constexpr int kTotal = kMergeOff + 4 * 32 * 16 + 1024;  // + alignment slack
};

template <bool BF16, int DK, int AST, int BST>
__global__ void __launch_bounds__(kThreads, 1)
assign_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                 const Params p) {
    using S = Smem<DK, AST, BST>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
    uint8_t* smA = sm;
    uint8_t* smB = sm + S::kABytes;
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + S::kBarOff);
    uint64_t* a_full = bars;
    uint64_t* a_empty = bars + AST;
    uint64_t* b_full = bars + 2 * AST;
    uint64_t* b_empty = bars + 2 * AST + BST;
    uint64_t* acc_full = bars + 2 * AST + 2 * BST;
    uint64_t* acc_empty = acc_full + 2;
    uint64_t* merge_full = acc_full + 4;   // column-half 1 -> half 0 handoff per tile
    uint64_t* merge_empty = acc_full + 5;
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + S::kBars);
    float4* merge = reinterpret_cast<float4*>(sm + S::kMergeOff);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int total_tiles = p.num_bh * p.tiles_per_bh;

    if (threadIdx.x == 0) {
        for (int i = 0; i < AST; i++) {
            mbar_init(&a_full[i], 1);
            mbar_init(&a_empty[i], 1 + kEpiWarps);
        }
        for (int i = 0; i < BST; i++) {
            mbar_init(&b_full[i], 1);
            mbar_init(&b_empty[i], 1);
        }
        for (int i = 0; i < 2; i++) {
            mbar_init(&acc_full[i], 1);
            mbar_init(&acc_empty[i], kEpiWarps);
        }
        mbar_init(merge_full, kEpiWarps / 2);
        mbar_init(merge_empty, kEpiWarps / 2);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         su32(tmem_holder)),
                     "r"(2 * BN)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;

    if (warp == 0) {
        // ------------------------------------------------------ producer --
        if (lane == 0) {
            uint32_t a_it = 0, b_it = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < total_tiles && ok; t += gridDim.x) {
                const TileInfo ti = tile_info(p, t);
                if (ti.skip) continue;
                const int sa = a_it % AST;
                ok = mbar_wait(&a_empty[sa], ((a_it / AST) & 1) ^ 1, p.status, 1);
                if (!ok) break;
                mbar_expect_tx(&a_full[sa], DK * S::kA);
                const int row0 = ti.bh * p.ncap + ti.r0;
#pragma unroll
                for (int kb = 0; kb < DK; kb++)
                    tma_2d(smA + (sa * DK + kb) * S::kA, &tmA, &a_full[sa], kb * BK, row0);
                a_it++;
                const int h = ti.bh % p.H;
                for (int c = 0; c < p.nchunks && ok; c++)
                    for (int pl = 0; pl < p.P && ok; pl++)
                        for (int kb = 0; kb < DK; kb++) {
                            const int sb = b_it % BST;
                            ok = mbar_wait(&b_empty[sb], ((b_it / BST) & 1) ^ 1, p.status, 2);
                            if (!ok) break;
                            mbar_expect_tx(&b_full[sb], S::kB);
                            tma_3d(smB + sb * S::kB, &tmB, &b_full[sb], kb * BK, c * BN,
                                   h * p.P + pl);
                            b_it++;
                        }
            }
            // every issued copy has landed before the CTA may leave
            for (int s = 0; s < BST; s++)
                if (b_it > (uint32_t)s) {
                    const uint32_t last = b_it - 1 - ((b_it - 1 - s) % BST);
                    mbar_wait(&b_full[last % BST], (last / BST) & 1, p.status, 3);
                }
            for (int s = 0; s < AST; s++)
                if (a_it > (uint32_t)s) {
                    const uint32_t last = a_it - 1 - ((a_it - 1 - s) % AST);
                    mbar_wait(&a_full[last % AST], (last / AST) & 1, p.status, 3);
                }
        }
    } else if (warp == 1) {
        // ----------------------------------------------------------- MMA --
        if (lane == 0) {
            const uint32_t idesc = (1u << 4) | ((BF16 ? 1u : 0u) << 7) | ((BF16 ? 1u : 0u) << 10) |
                                   ((uint32_t)(BN >> 3) << 17) | ((uint32_t)(BM >> 4) << 24);
            uint32_t a_it = 0, b_it = 0, acc_it = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < total_tiles && ok; t += gridDim.x) {
                const TileInfo ti = tile_info(p, t);
                if (ti.skip) continue;
                const int sa = a_it % AST;
                ok = mbar_wait(&a_full[sa], (a_it / AST) & 1, p.status, 4);
                if (!ok) break;
                tc_fence_after();
                for (int c = 0; c < p.nchunks && ok; c++) {
                    const int acc = acc_it & 1;
                    ok = mbar_wait(&acc_empty[acc], ((acc_it >> 1) & 1) ^ 1, p.status, 5);
                    if (!ok) break;
                    tc_fence_after();
                    const uint32_t d_tmem = tmem + (uint32_t)(acc * BN);
                    uint32_t accumulate = 0;
                    for (int pl = 0; pl < p.P && ok; pl++)
                        for (int kb = 0; kb < DK; kb++) {
                            const int sb = b_it % BST;
                            ok = mbar_wait(&b_full[sb], (b_it / BST) & 1, p.status, 6);
                            if (!ok) break;
                            tc_fence_after();
                            const uint32_t a_base = su32(smA + (sa * DK + kb) * S::kA);
                            const uint32_t b_base = su32(smB + sb * S::kB);
#pragma unroll
                            for (int ks = 0; ks < BK / 16; ks++) {
                                tc_mma(d_tmem, sw128_desc(a_base + ks * 32),
                                       sw128_desc(b_base + ks * 32), idesc, accumulate);
                                accumulate = 1;
                            }
                            tc_commit(&b_empty[sb]);
                            b_it++;
                        }
                    tc_commit(&acc_full[acc]);
                    acc_it++;
                }
                tc_commit(&a_empty[sa]);
                a_it++;
            }
        }
    } else {
        // ------------------------------------------------------ epilogue --
        const int ew = warp - 2;
        const int q = warp & 3;          // TMEM lane quarter this warp may access
        const int half = ew >> 2;        // which 128 of the 256 accumulator columns
        const int row_in_tile = 32 * q + lane;
        uint32_t a_it = 0, acc_it = 0, m_it = 0;
        bool ok = true;
        for (int t = blockIdx.x; t < total_tiles && ok; t += gridDim.x) {
            const TileInfo ti = tile_info(p, t);
            if (ti.skip) continue;
            const int h = ti.bh % p.H;
            const int sa = a_it % AST;
            ok = mbar_wait(&a_full[sa], (a_it / AST) & 1, p.status, 7);
            if (!ok) break;
            // |x|^2 of this row from the swizzled tile (order does not matter)
            float nrm = 0.f;
            if (half == 0) {
#pragma unroll
                for (int kb = 0; kb < DK; kb++) {
                    const uint8_t* rowp = smA + (sa * DK + kb) * S::kA + row_in_tile * 128;
#pragma unroll
                    for (int c = 0; c < 8; c++) {
                        const uint4 raw = *reinterpret_cast<const uint4*>(
                            rowp + 16 * (c ^ (row_in_tile & 7)));
                        const uint32_t w4[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
                        for (int u = 0; u < 4; u++) {
                            float lo, hi;
                            if (BF16) {
                                lo = __uint_as_float(w4[u] << 16);
                                hi = __uint_as_float(w4[u] & 0xFFFF0000u);
                            } else {
                                const __half2 hv = *reinterpret_cast<const __half2*>(&w4[u]);
                                const float2 f = __half22float2(hv);
                                lo = f.x;
                                hi = f.y;
                            }
                            nrm = fmaf(lo, lo, nrm);
                            nrm = fmaf(hi, hi, nrm);
                        }
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&a_empty[sa]);
            a_it++;

            float m1 = -FLT_MAX, m2 = -FLT_MAX;
            int32_t c1 = 0;
            const float* hn = p.half_norm + (int64_t)h * p.K;
            const float inv_scale = p.head[h * 4 + 2];
            for (int c = 0; c < p.nchunks && ok; c++) {
                const int acc = acc_it & 1;
                ok = mbar_wait(&acc_full[acc], (acc_it >> 1) & 1, p.status, 8);
                if (!ok) break;
                tc_fence_after();
#pragma unroll 1
                for (int sub = 0; sub < 4; sub++) {
                    const int col = half * 128 + sub * 32;
                    uint32_t r[32];
                    A2ATS_TMEM_LD32(tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(acc * BN + col),
                                    r);
                    tmem_wait_ld();
                    const int j0 = c * BN + col;
                    float key[32];
                    if (j0 + 32 <= p.K && (p.K & 3) == 0) {
                        const float4* h4 = reinterpret_cast<const float4*>(hn + j0);
#pragma unroll
                        for (int u = 0; u < 8; u++) {
                            const float4 hv = __ldg(h4 + u);
                            key[4 * u + 0] = fmaf(__uint_as_float(r[4 * u + 0]), inv_scale, -hv.x);
                            key[4 * u + 1] = fmaf(__uint_as_float(r[4 * u + 1]), inv_scale, -hv.y);
                            key[4 * u + 2] = fmaf(__uint_as_float(r[4 * u + 2]), inv_scale, -hv.z);
                            key[4 * u + 3] = fmaf(__uint_as_float(r[4 * u + 3]), inv_scale, -hv.w);
                        }
                    } else {
#pragma unroll
                        for (int u = 0; u < 32; u++)
                            key[u] = (j0 + u < p.K)
                                         ? fmaf(__uint_as_float(r[u]), inv_scale, -hn[j0 + u])
                                         : -FLT_MAX;
                    }
#pragma unroll
                    for (int u = 0; u < 32; u++)
                        key[u] = __uint_as_float((__float_as_uint(key[u]) & ~31u) | (31u - u));
                    float t1, t2;
                    top2_32(key, t1, t2);
                    if (t1 > m1) c1 = j0 >> 5;
                    const float n1 = fmaxf(m1, t1);
                    m2 = fmaxf(fminf(m1, t1), fmaxf(m2, t2));
                    m1 = n1;
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&acc_empty[acc]);
                acc_it++;
            }
            if (!ok) break;
            // merge the two column halves of each row, then decide the row
            if (half == 1) {
                ok = mbar_wait(merge_empty, (m_it & 1) ^ 1, p.status, 9);
                if (!ok) break;
                merge[q * 32 + lane] = make_float4(m1, m2, __int_as_float(c1), 0.f);
                __syncwarp();
                if (lane == 0) mbar_arrive(merge_full);
            } else {
                ok = mbar_wait(merge_full, m_it & 1, p.status, 10);
                if (!ok) break;
                const float4 o = merge[q * 32 + lane];
                __syncwarp();
                if (lane == 0) mbar_arrive(merge_empty);
                const int32_t oc = __float_as_int(o.z);
                // keys are distinct (column bits), so only the order matters
                if (o.x > m1) {
                    m2 = fmaxf(m1, o.y);
                    m1 = o.x;
                    c1 = oc;
                } else {
                    m2 = fmaxf(m2, o.x);
                }
                const int32_t ri = ti.r0 + row_in_tile;
                if (ri < ti.nvalid) {
                    const int32_t j = p.row_map ? p.row_map[(int64_t)ti.bh * p.ncap + ri] : ri;
                    const int32_t Lb = seq_len(p.len, ti.bh / p.H, p.ncap);
                    if (j >= 0 && j < Lb) {
                        const int64_t out = (int64_t)ti.bh * p.ncap + j;
                        const bool skip = p.skip && p.skip[out];
                        const bool near = p.window > 0 && (Lb - 1 - j) < p.window;
                        // bound on |v_hat - v| for every centroid, plus the
                        // perturbation of the column bits in both keys
                        const float cmax = p.head[h * 4 + 0], hmax = p.head[h * 4 + 1];
                        const float e = p.err_coef * (sqrtf(nrm) * 1.0001f * cmax + hmax) +
                                        p.head[h * 4 + 3] * sqrtf(nrm);
                        const float mag = fmaxf(fabsf(m1), fabsf(m2));
                        const float tau = 2.f * e + 64.f * mag * 1.1920929e-07f;
                        if (!skip) {
                            if (near || !(m1 - m2 > tau)) {
                                const int32_t slot = atomicAdd(p.exact_count, 1);
                                p.exact_list[slot] = out;
                            } else {
                                p.codes[out] = c1 * 32 + (31 - (int32_t)(__float_as_uint(m1) & 31u));
                            }
                        }
                    }
                }
            }
            m_it++;
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "r"(2 * BN)
                     : "memory");
    }
}

// -------------------------------------------------- codebook preparation --
// In place on chat [H, K, d] fp32: optional rotation by -far_offset (so far
// keys can enter the contraction unrotated), then per-head maxima into
// head_bits [H, 4] (uint bits of non-negative floats; zeroed by the caller):
// max |chat_j|, max h_j, max |element|.
__global__ void codebook_stats_kernel(float* __restrict__ chat, int64_t HK, int64_t K,
                                      int32_t d, const RopeArgs ra, int32_t rotate,
                                      const float* __restrict__ half_norm,
                                      uint32_t* __restrict__ head_bits) {
    const int lane = threadIdx.x & 31;
    for (int64_t j = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; j < HK;
         j += ((int64_t)gridDim.x * blockDim.x) >> 5) {
        float* row = chat + j * d;
        if (rotate) {
            const int halfd = d / 2;
            for (int i = lane; i < halfd; i += 32) {
                float s, c;
                rope_angle(-ra.far_offset, ra.omega_hi[i], ra.omega_lo[i], ra, s, c);
                const int a = ra.interleaved ? 2 * i : i;
                const int b = ra.interleaved ? 2 * i + 1 : i + halfd;
                const float xa = row[a], xb = row[b];
                row[a] = fmaf(xa, c, -__fmul_rn(xb, s));
                row[b] = fmaf(xa, s, __fmul_rn(xb, c));
            }
            __syncwarp();
        }
        Dot2 n;
        float mx = 0.f;
        for (int a = lane; a < d; a += 32) {
            const float v = row[a];
            n.add_prod(v, v);
            mx = fmaxf(mx, fabsf(v));
        }
        for (int m = 16; m; m >>= 1) {
            n.merge(shfl_xor(n, m));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, m));
        }
        if (lane == 0) {
            const int64_t h = j / K;
            atomicMax(&head_bits[h * 4 + 0], __float_as_uint(sqrtf(n.value()) * 1.000001f));
            atomicMax(&head_bits[h * 4 + 1], __float_as_uint(fmaxf(half_norm[j], 0.f)));
            atomicMax(&head_bits[h * 4 + 2], __float_as_uint(mx));
        }
    }
}

// head [H, 4] floats from the raw maxima: max |chat|, max h, 1/scale, abs err.
// bf16 planes: scale 1.  fp16 planes: a power of two that puts the largest
// element near 2^14; elements that fall into the fp16 subnormal range are
// covered by the absolute error term (per unit of |x|).
__global__ void head_finish_kernel(const uint32_t* __restrict__ head_bits, int32_t H, int32_t d,
                                   int32_t unit_scale, float* __restrict__ head,
                                   float* __restrict__ scale) {
    const int h = blockIdx.x * blockDim.x + threadIdx.x;
    if (h >= H) return;
    const float cmax = __uint_as_float(head_bits[h * 4 + 0]);
    const float hmax = __uint_as_float(head_bits[h * 4 + 1]);
    const float emax = __uint_as_float(head_bits[h * 4 + 2]);
    float sc = 1.f;
    float abs_err = 0.f;
    if (!unit_scale) {
        int e = 0;
        frexpf(emax > 0.f ? emax : 1.f, &e);  // emax < 2^e
        sc = ldexpf(1.f, 14 - e);
        // each element carries at most 2^-25 absolute error (fp16 subnormal
        // spacing of the last plane), i.e. 2^-25 / sc unscaled, over d terms
        abs_err = sqrtf((float)d) * ldexpf(1.f, -24) / sc;
    }
    head[h * 4 + 0] = cmax;
    head[h * 4 + 1] = hmax;
    head[h * 4 + 2] = 1.f / sc;
    head[h * 4 + 3] = abs_err;
    scale[h] = sc;
}

// planes [H, P, K, d] (16-bit) of chat * scale: plane p is the rounding of
// what the planes before it leave over (each difference is exact in fp32).
template <bool BF16>
__global__ void codebook_planes_kernel(const float* __restrict__ chat, int64_t K, int32_t d,
                                       int32_t P, int32_t H, const float* __restrict__ scale,
                                       uint16_t* __restrict__ planes) {
    const int64_t n = (int64_t)H * K * d;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t h = i / (K * d);
        const int64_t rest = i % (K * d);
        float r = chat[i] * scale[h];
        for (int pl = 0; pl < P; pl++) {
            uint16_t bits;
            float back;
            if (BF16) {
                const __nv_bfloat16 v = __float2bfloat16_rn(r);
                bits = __bfloat16_as_ushort(v);
                back = __bfloat162float(v);
            } else {
                const __half v = __float2half_rn(r);
                bits = __half_as_ushort(v);
                back = __half2float(v);
            }
            planes[(h * P + pl) * K * d + rest] = bits;
            r = r - back;
        }
    }
}

// ------------------------------------------------------- row gathering --
// Compact copy of the retrieval rows of each (b, h): row i of the compact
// block is row perm[i] of the keys (16-byte vectors), row_map[i] = perm[i].
__global__ void gather_rows_kernel(const void* __restrict__ x, int32_t esize, int32_t H,
                                   int32_t ncap, int32_t d, const int32_t* __restrict__ len,
                                   const int32_t* __restrict__ perm,
                                   const int32_t* __restrict__ count, void* __restrict__ compact,
                                   int32_t* __restrict__ row_map) {
    const int bh = blockIdx.y;
    const int32_t L = seq_len(len, bh / H, ncap);
    const int32_t cnt = min(max(count[bh], 0), L);
    const int vec = d * esize / 16;  // 16-byte vectors per row
    const uint4* src = reinterpret_cast<const uint4*>(x);
    uint4* dst = reinterpret_cast<uint4*>(compact);
    for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < (int64_t)cnt * vec;
         e += (int64_t)gridDim.x * blockDim.x) {
        const int32_t i = (int32_t)(e / vec), v = (int32_t)(e % vec);
        int32_t j = perm[(int64_t)bh * ncap + i];
        const bool valid = j >= 0 && j < L;
        if (v == 0) row_map[(int64_t)bh * ncap + i] = valid ? j : -1;
        dst[((int64_t)bh * ncap + i) * vec + v] =
            valid ? src[((int64_t)bh * ncap + j) * vec + v] : make_uint4(0, 0, 0, 0);
    }
}

// skip[bh*ncap + perm[i]] = 1 for the retrieval rows (bulk mode leaves them alone)
__global__ void mark_rows_kernel(int32_t H, int32_t ncap, const int32_t* __restrict__ len,
                                 const int32_t* __restrict__ perm,
                                 const int32_t* __restrict__ count, uint8_t* __restrict__ skip) {
    const int bh = blockIdx.y;
    const int32_t L = seq_len(len, bh / H, ncap);
    const int32_t cnt = min(max(count[bh], 0), L);
    for (int32_t i = blockIdx.x * blockDim.x + threadIdx.x; i < cnt; i += gridDim.x * blockDim.x) {
        const int32_t j = perm[(int64_t)bh * ncap + i];
        if (j >= 0 && j < L) skip[(int64_t)bh * ncap + j] = 1;
    }
}

// ------------------------------------------------------ exact list kernel --
// One warp per listed row: windowed RoPE in fp32, z = x L (compensated), then
// the direct distance to every cp_j = c_j L, ties to the lowest index.
template <int DT>
__global__ void __launch_bounds__(256)
exact_list_kernel(const void* __restrict__ x, int32_t H, int32_t ncap, int32_t d,
                  const int32_t* __restrict__ len, const RopeArgs ra, const float* __restrict__ L,
                  const float* __restrict__ cp, int64_t K, const int64_t* __restrict__ list,
                  const int32_t* __restrict__ list_count, int32_t* __restrict__ codes) {
    __shared__ float xs[8][kMaxD];
    __shared__ float zs[8][kMaxD];
    const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n = *list_count;
    for (int e = blockIdx.x * 8 + w; e < n; e += gridDim.x * 8) {
        const int64_t out = list[e];
        const int64_t bh = out / ncap;
        const int32_t j = (int32_t)(out % ncap);
        const int64_t h = bh % H;
        const int32_t Lb = seq_len(len, (int32_t)(bh / H), ncap);
        float* xv = xs[w];
        float* zv = zs[w];
        for (int a = lane; a < d; a += 32) xv[a] = load1<DT>(x, out * d + a);
        __syncwarp();
        if (ra.enabled) {
            const int32_t pos = rope_position(j, Lb - 1, ra);
            if (pos != 0) {
                const int halfd = d / 2;
                for (int i = lane; i < halfd; i += 32) {
                    float s, c;
                    rope_angle(pos, ra.omega_hi[i], ra.omega_lo[i], ra, s, c);
                    const int a = ra.interleaved ? 2 * i : i;
                    const int b = ra.interleaved ? 2 * i + 1 : i + halfd;
                    const float xa = xv[a], xb = xv[b];
                    xv[a] = fmaf(xa, c, -__fmul_rn(xb, s));
                    xv[b] = fmaf(xa, s, __fmul_rn(xb, c));
                }
            }
            __syncwarp();
        }
        const float* zr = xv;
        if (L) {
            const float* Lh = L + h * d * d;
            for (int b = lane; b < d; b += 32) {
                Dot2 acc;
                for (int a = 0; a < d; a++) acc.add_prod(xv[a], Lh[(int64_t)a * d + b]);
                zv[b] = acc.value();
            }
            __syncwarp();
            zr = zv;
        }
        float best = INFINITY;
        int32_t bj = 0;
        const float* cph = cp + h * K * d;
        for (int64_t jj = lane; jj < K; jj += 32) {
            const float4* c4 = reinterpret_cast<const float4*>(cph + jj * d);
            float acc[4] = {0.f, 0.f, 0.f, 0.f};
            for (int a = 0; a < d / 4; a++) {
                const float4 cv = __ldg(c4 + a);
                const float t0 = zr[4 * a] - cv.x, t1 = zr[4 * a + 1] - cv.y;
                const float t2 = zr[4 * a + 2] - cv.z, t3 = zr[4 * a + 3] - cv.w;
                acc[0] = fmaf(t0, t0, acc[0]);
                acc[1] = fmaf(t1, t1, acc[1]);
                acc[2] = fmaf(t2, t2, acc[2]);
                acc[3] = fmaf(t3, t3, acc[3]);
            }
            const float v = (acc[0] + acc[1]) + (acc[2] + acc[3]);
            if (v < best) { best = v; bj = (int32_t)jj; }
        }
        for (int m = 16; m; m >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, best, m);
            const int32_t oj = __shfl_xor_sync(0xffffffffu, bj, m);
            if (ov < best || (ov == best && oj < bj)) { best = ov; bj = oj; }
        }
        if (lane == 0) codes[out] = bj;
        __syncwarp();
    }
}

__global__ void transpose_kernel(const float* __restrict__ in, int64_t H, int32_t d,
                                 float* __restrict__ out) {
    const int64_t n = H * d * d;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t h = i / ((int64_t)d * d);
        const int a = (int)((i / d) % d), b = (int)(i % d);
        out[(h * d + b) * d + a] = in[i];
    }
}

// ------------------------------------------------------------ host side --
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        cudaDriverEntryPointQueryResult q;
        void* f = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    }
    return fn;
}

int sm_count() {
    int dev = 0, n = 152;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    return n;
}

template <bool BF16, int DK, int AST, int BST>
cudaError_t launch_kernel(const CUtensorMap& ta, const CUtensorMap& tb, const Params& p,
                          cudaStream_t st) {
    using S = Smem<DK, AST, BST>;
    auto k = assign_tc_kernel<BF16, DK, AST, BST>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, S::kTotal);
    if (e != cudaSuccess) return e;
    const int tiles = p.num_bh * p.tiles_per_bh;
    const int grid = tiles < sm_count() ? tiles : sm_count();
    k<<<grid, kThreads, S::kTotal, st>>>(ta, tb, p);
    note_launches(1);
    return cudaGetLastError();
}

template <bool BF16>
cudaError_t launch_by_width(const CUtensorMap& ta, const CUtensorMap& tb, const Params& p,
                            cudaStream_t st) {
    switch (p.d) {
        case 64: return launch_kernel<BF16, 1, 2, 4>(ta, tb, p, st);
        case 128: return launch_kernel<BF16, 2, 2, 4>(ta, tb, p, st);
        case 192: return launch_kernel<BF16, 3, 1, 4>(ta, tb, p, st);
        default: return launch_kernel<BF16, 4, 1, 4>(ta, tb, p, st);
    }
}

}  // namespace tc

bool tc_supported(int dt, int64_t d) {
    return (dt == kBF16 || dt == kF16) && d % 64 == 0 && d >= 64 && d <= 256 &&
           tc::encode_fn() != nullptr;
}

size_t tc_workspace_floats(int64_t H, int64_t K, int64_t d) {
    return (size_t)(H * K * d);  // chat
}

cudaError_t launch_assign_tc(const TcCall& c, cudaStream_t st) {
    using namespace tc;
    const bool bf16 = c.dt == kBF16;
    const int64_t H = c.s.H, K = c.K, d = c.s.d, nbh = c.s.B * c.s.H, ncap = c.s.Ncap;
    const size_t esz = 2;
    cudaError_t e;
    // 1. transformed codebook chat (fp32) unless the raw codebook is exact
    const bool exact_plain = !c.L && !(c.ra.enabled && c.ra.far_offset != 0);
    const int P = exact_plain ? 1 : (bf16 ? 3 : 2);
    e = cudaMemsetAsync(c.head_bits, 0, sizeof(uint32_t) * 4 * H, st);
    if (e != cudaSuccess) return e;
    if (c.L) {
        transpose_kernel<<<(unsigned)((H * d * d + 255) / 256 < 4096 ? (H * d * d + 255) / 256 : 4096),
                           256, 0, st>>>(c.L, H, (int32_t)d, c.Lt);
        note_launches(1);
        e = launch_codebook_transform(c.cp, kF32, H, K, d, c.Lt, c.chat, c.scratch_norm, st);
        if (e != cudaSuccess) return e;
    } else {
        e = cudaMemcpyAsync(c.chat, c.cp, sizeof(float) * H * K * d, cudaMemcpyDeviceToDevice, st);
        if (e != cudaSuccess) return e;
    }
    {
        const int64_t HK = H * K;
        const unsigned blocks = (unsigned)((HK * 32 + 255) / 256 < 4096 ? (HK * 32 + 255) / 256 : 4096);
        codebook_stats_kernel<<<blocks, 256, 0, st>>>(c.chat, HK, K, (int32_t)d, c.ra,
                                                      c.ra.enabled && c.ra.far_offset != 0,
                                                      c.half_norm, c.head_bits);
        note_launches(1);
        head_finish_kernel<<<(unsigned)((H + 63) / 64), 64, 0, st>>>(
            c.head_bits, (int32_t)H, (int32_t)d, (bf16 || exact_plain) ? 1 : 0, c.head, c.scale);
        note_launches(1);
    }
    const void* bsrc = c.codebook;
    if (!exact_plain) {
        const int64_t n = H * K * d;
        const unsigned blocks = (unsigned)((n + 255) / 256 < 8192 ? (n + 255) / 256 : 8192);
        if (bf16)
            codebook_planes_kernel<true><<<blocks, 256, 0, st>>>(c.chat, K, (int32_t)d, P,
                                                                 (int32_t)H, c.scale, c.planes);
        else
            codebook_planes_kernel<false><<<blocks, 256, 0, st>>>(c.chat, K, (int32_t)d, P,
                                                                  (int32_t)H, c.scale, c.planes);
        note_launches(1);
        bsrc = c.planes;
    }
    // 2. row selection
    const void* asrc = c.x;
    const int32_t* row_map = nullptr;
    const int32_t* count = nullptr;
    const uint8_t* skip = nullptr;
    if (c.sel.mode == 1) {
        dim3 g((unsigned)((ncap * (d * esz / 16) + 255) / 256 < 256 ? (ncap * (d * esz / 16) + 255) / 256 : 256),
               (unsigned)nbh);
        gather_rows_kernel<<<g, 256, 0, st>>>(c.x, (int32_t)esz, (int32_t)H, (int32_t)ncap,
                                              (int32_t)d, c.len, c.sel.perm, c.sel.count,
                                              c.compact, c.row_map);
        note_launches(1);
        asrc = c.compact;
        row_map = c.row_map;
        count = c.sel.count;
    } else if (c.sel.mode == 2) {
        e = cudaMemsetAsync(c.skip, 0, (size_t)(nbh * ncap), st);
        if (e != cudaSuccess) return e;
        dim3 g((unsigned)((ncap + 255) / 256 < 64 ? (ncap + 255) / 256 : 64), (unsigned)nbh);
        mark_rows_kernel<<<g, 256, 0, st>>>((int32_t)H, (int32_t)ncap, c.len, c.sel.perm,
                                            c.sel.count, c.skip);
        note_launches(1);
        skip = c.skip;
    }
    e = cudaMemsetAsync(c.exact_count, 0, sizeof(int32_t) * 2, st);  // count and status
    if (e != cudaSuccess) return e;
    // 3. tensor maps
    CUtensorMap ta, tb;
    {
        const cuuint64_t dims[2] = {(cuuint64_t)d, (cuuint64_t)(nbh * ncap)};
        const cuuint64_t strides[1] = {(cuuint64_t)(d * esz)};
        const cuuint32_t box[2] = {BK, BM};
        const cuuint32_t es[2] = {1, 1};
        if (encode_fn()(&ta, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                        2, const_cast<void*>(asrc), dims, strides, box, es,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    {
        const cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)K, (cuuint64_t)(H * P)};
        const cuuint64_t strides[2] = {(cuuint64_t)(d * esz), (cuuint64_t)(K * d * esz)};
        const cuuint32_t box[3] = {BK, BN, 1};
        const cuuint32_t es[3] = {1, 1, 1};
        if (encode_fn()(&tb, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                        3, const_cast<void*>(bsrc), dims, strides, box, es,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    // 4. the contraction
    Params p;
    p.H = (int32_t)H;
    p.ncap = (int32_t)ncap;
    p.d = (int32_t)d;
    p.K = (int32_t)K;
    p.P = P;
    p.num_bh = (int32_t)nbh;
    p.tiles_per_bh = (int32_t)((ncap + BM - 1) / BM);
    p.nchunks = (int32_t)((K + BN - 1) / BN);
    p.len = c.len;
    p.count = count;
    p.row_map = row_map;
    p.skip = skip;
    p.window = c.ra.enabled ? c.ra.window : 0;
    p.half_norm = c.half_norm;
    p.head = c.head;
    // products are exact; the tensor core adds (d/16 per plane) partial sums
    // into fp32, each addition off by at most 2^-23 of the running magnitude,
    // which |x| max|chat| bounds; plus the rounding of chat (fp32) and of the
    // planes that are dropped, and of h and of acc - h.
    const double steps = (double)P * (double)(d / 16);
    double coef = (steps + 8.0) * 0x1p-22;
    if (!exact_plain) coef += bf16 ? 0x1p-20 : (0x1p-21 + 0x1p-20);
    p.err_coef = (float)coef;
    p.codes = c.codes;
    p.exact_list = c.exact_list;
    p.exact_count = c.exact_count;
    p.status = c.exact_count + 1;
    if (p.num_bh * p.tiles_per_bh > 0) {
        e = bf16 ? launch_by_width<true>(ta, tb, p, st) : launch_by_width<false>(ta, tb, p, st);
        if (e != cudaSuccess) return e;
    }
    // 5. rows the contraction could not decide
    const unsigned lg = (unsigned)(sm_count() * 4);
    if (bf16)
        exact_list_kernel<kBF16><<<lg, 256, 0, st>>>(c.x, (int32_t)H, (int32_t)ncap, (int32_t)d,
                                                     c.len, c.ra, c.L, c.cp, K, c.exact_list,
                                                     c.exact_count, c.codes);
    else
        exact_list_kernel<kF16><<<lg, 256, 0, st>>>(c.x, (int32_t)H, (int32_t)ncap, (int32_t)d,
                                                    c.len, c.ra, c.L, c.cp, K, c.exact_list,
                                                    c.exact_count, c.codes);
    note_launches(1);
    return cudaGetLastError();
}

}  // namespace a2ats
