// calib_tc.cu -- the query second moment H = (1/M) Q^T Q + ridge I on the
// tensor cores (API page "veloxquant_mlx.quantizers.a2ats module",
// a2ats_query_second_moment, paper Eq. 10) for 16-bit queries with d = 128.
//
// One CTA per (slice of the M queries, head).  The CTA's 256 threads load
// the slice 128 rows at a time, transpose 8 x 8 blocks in registers and store
// the tile as Q^T in the 128-byte swizzled K-major layout tcgen05.mma reads;
// the one stored tile is both operands of D = Q^T Q (D[i][j] = sum over rows
// of Q[r][i] Q[r][j]), so every product is exact.  The fp32 accumulation is
// bounded by giving each of four TMEM accumulators a quarter of the slice (at
// most 512 rows, 32 k-steps); at the end the four are added with compensated
// sums and written as the hi / lo planes the compensated reduce of the SIMT
// path folds over the slices.
#include "kernels.cuh"
#include "tc_ptx.cuh"

namespace a2ats {
namespace {

using namespace tc;

constexpr int kQd = 128;       // head width this kernel serves
constexpr int kQt = 128;       // query rows per tile (two 64-row k-blocks)
constexpr int kNacc = 4;       // TMEM accumulators of kQd columns
constexpr int kSmThreadsTc = 256;
constexpr int kTileBytes = 2 * kQd * 128;  // two k-blocks of kQd rows x 128 bytes
constexpr int kSmemTc = 2 * kTileBytes + 1024;

// Rows per accumulator above which the SIMT kernel is used instead (the
// error of an fp32 accumulator grows with its k-steps).
constexpr int64_t kMaxAccRows = 512;

template <bool BF16>
__global__ void __launch_bounds__(kSmThreadsTc, 1)
second_moment_tc_kernel(const uint16_t* __restrict__ q, int64_t M, int64_t splits,
                        float* __restrict__ partial, int32_t* __restrict__ status) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
    __shared__ uint64_t stage_free[2];
    __shared__ uint64_t done;
    __shared__ uint32_t tmem_holder;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int split = blockIdx.x, h = blockIdx.y, H = gridDim.y;
    const int64_t m0 = M * split / splits, m1 = M * (split + 1) / splits;
    const int T = (int)((m1 - m0 + kQt - 1) / kQt);   // tiles of the slice
    const int nacc = T < kNacc ? T : kNacc;

    if (tid == 0) {
        mbar_init(&stage_free[0], 1);
        mbar_init(&stage_free[1], 1);
        mbar_init(&done, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         su32(&tmem_holder)),
                     "r"(kNacc * kQd)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_holder;

    // this thread's 8 x 8 block of a tile: rows 8 rb .. + 7, columns 8 cb .. + 7;
    // a warp covers 8 distinct rb % 8 (conflict-free stores) and 4 adjacent cb
    // (64 contiguous bytes of each row per load)
    const int rb = (lane & 7) + 8 * (warp & 1);
    const int cb = (lane >> 3) + 4 * (warp >> 1);
    const uint16_t* qh = q + (int64_t)h * M * kQd;
    uint4 cur[8], nxt[8];
    auto load = [&](int it, uint4* r) {
        const int64_t base = m0 + (int64_t)it * kQt + 8 * rb;
#pragma unroll
        for (int k = 0; k < 8; k++) {
            const int64_t m = base + k;
            r[k] = m < m1 ? __ldg(reinterpret_cast<const uint4*>(qh + m * kQd + 8 * cb))
                          : make_uint4(0u, 0u, 0u, 0u);
        }
    };
    const uint32_t idesc = (1u << 4) | ((BF16 ? 1u : 0u) << 7) | ((BF16 ? 1u : 0u) << 10) |
                           ((uint32_t)(kQd >> 3) << 17) | ((uint32_t)(128 >> 4) << 24);
    if (T > 0) load(0, cur);
    for (int it = 0; it < T; it++) {
        if (it + 1 < T) load(it + 1, nxt);
        const int s = it & 1;
        // the MMAs that read this stage two tiles ago have completed
        mbar_wait(&stage_free[s], ((it >> 1) & 1) ^ 1, status, 21);
        uint8_t* stage = sm + s * kTileBytes;
        // column i = 8 cb + c of the block holds rows 8 rb .. + 7: its 16 bytes
        // are chunk rb % 8 of row i in k-block rb / 8 (swizzled by i % 8 = c)
        uint8_t* kblk = stage + (rb >> 3) * (kQd * 128);
#pragma unroll
        for (int c = 0; c < 8; c++) {
            const int i = 8 * cb + c;
            const uint32_t sel = (c & 1) ? 0x7632u : 0x5410u;
            uint4 o;
            o.x = __byte_perm((&cur[0].x)[c >> 1], (&cur[1].x)[c >> 1], sel);
            o.y = __byte_perm((&cur[2].x)[c >> 1], (&cur[3].x)[c >> 1], sel);
            o.z = __byte_perm((&cur[4].x)[c >> 1], (&cur[5].x)[c >> 1], sel);
            o.w = __byte_perm((&cur[6].x)[c >> 1], (&cur[7].x)[c >> 1], sel);
            *reinterpret_cast<uint4*>(kblk + i * 128 + 16 * ((rb & 7) ^ c)) = o;
        }
        // the generic-proxy stores are visible to the tensor core's reads
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncthreads();
        if (tid == 0) {
            tc_fence_after();
            // accumulator a takes tiles [a T / nacc, (a + 1) T / nacc)
            int a = 0;
            while ((a + 1) * T / nacc <= it) a++;
            const bool first = it == a * T / nacc;
            const uint32_t d_tmem = tmem + (uint32_t)(a * kQd);
#pragma unroll
            for (int kb = 0; kb < 2; kb++) {
                const uint64_t desc = sw128_desc(su32(stage + kb * (kQd * 128)));
#pragma unroll
                for (int ks = 0; ks < 4; ks++)
                    tc_mma(d_tmem, desc + 2 * ks, desc + 2 * ks, idesc,
                           (first && kb == 0 && ks == 0) ? 0u : 1u);
            }
            tc_commit(&stage_free[s]);
        }
#pragma unroll
        for (int k = 0; k < 8; k++) cur[k] = nxt[k];
    }
    if (tid == 0) tc_commit(&done);
    mbar_wait(&done, 0, status, 22);
    tc_fence_after();

    // read-out: warp (quarter qd, half) takes rows 32 qd + lane (TMEM lanes)
    // and columns 64 half .. + 63; the accumulators are added with
    // compensated sums into the hi / lo planes
    const int qd = warp & 3, half = warp >> 2;
    const int i = 32 * qd + lane;
    float* hi = partial + ((int64_t)split * H + h) * kQd * kQd + (int64_t)i * kQd;
    float* lo = hi + splits * H * kQd * kQd;
    for (int g = 0; g < 4; g++) {
        const int col = 64 * half + 16 * g;
        Dot2 acc[16];
        for (int a = 0; a < nacc; a++) {
            uint32_t r[16];
            const uint32_t taddr = tmem + ((uint32_t)(32 * qd) << 16) + (uint32_t)(a * kQd + col);
            asm volatile(
                "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, "
                "%10, %11, %12, %13, %14, %15}, [%16];"
                : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
                  "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]),
                  "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
                : "r"(taddr));
            tmem_wait_ld();
#pragma unroll
            for (int u = 0; u < 16; u++) acc[u].add(__uint_as_float(r[u]));
        }
#pragma unroll
        for (int u = 0; u < 16; u += 4) {
            *reinterpret_cast<float4*>(hi + col + u) =
                make_float4(acc[u].s, acc[u + 1].s, acc[u + 2].s, acc[u + 3].s);
            *reinterpret_cast<float4*>(lo + col + u) =
                make_float4(acc[u].c, acc[u + 1].c, acc[u + 2].c, acc[u + 3].c);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "r"(kNacc * kQd)
                     : "memory");
    }
}

}  // namespace

bool second_moment_tc_supported(int dt, int64_t H, int64_t M, int64_t d) {
    if ((dt != kBF16 && dt != kF16) || d != kQd || M < 1) return false;
    const int64_t splits = second_moment_splits(M, H);
    const int64_t rows = (M + splits - 1) / splits;
    const int64_t tiles = (rows + kQt - 1) / kQt;
    return (tiles + kNacc - 1) / kNacc * kQt <= kMaxAccRows;
}

cudaError_t launch_second_moment_tc(const void* q, int dt, int64_t H, int64_t M, float* partial,
                                    int32_t* status, cudaStream_t st) {
    const int64_t splits = second_moment_splits(M, H);
    auto k = dt == kBF16 ? second_moment_tc_kernel<true> : second_moment_tc_kernel<false>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemTc);
    if (e != cudaSuccess) return e;
    dim3 grid((unsigned)splits, (unsigned)H);
    k<<<grid, kSmThreadsTc, kSmemTc, st>>>(static_cast<const uint16_t*>(q), M, splits, partial,
                                          status);
    note_launches(1);
    return cudaGetLastError();
}

}  // namespace a2ats
