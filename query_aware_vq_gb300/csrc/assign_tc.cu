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
// Kernel layout (one persistent CTA per SM, 11 warps):
//   warp 10    TMA producer of the key tiles (kept for all centroids), a tile
//              ahead: 256 rows as two 128-row blocks at d <= 128 with one
//              operand plane, else 128 rows;
//   warp 0     TMA producer of the codebook by the accumulator width (128
//              centroids with two row blocks, else 256): a stage holds both
//              64-element k-blocks of a plane up to d = 128 (one k-block
//              above), and a chunk's first stage also the bf16 planes of
//              -|c'|^2/2 (fp16: a ring of its own, read by the epilogue);
//   warp 1     TMEM allocation and tcgen05.mma issue (M = 128 per row
//              block, bf16/fp16 -> fp32) into two accumulators per row block
//              (the 512 TMEM columns), so the epilogue of one centroid chunk
//              overlaps the MMAs of the next.  With bf16 operands the first
//              MMA of a chunk is one more K = 16 step, a constant tile of
//              ones against three bf16 planes of -|c'|^2/2, which starts the
//              accumulator at -h_j exactly;
//   warps 2-9  epilogue, one per (TMEM lane quarter, row block or 128-column
//              part): tcgen05.ld of the accumulator, v = acc - |c'|^2/2 (the
//              accumulator itself with bf16 operands; fp16 planes carry a
//              scale and add -h_j here), and
//              per 16-column group only its largest value (a three-input max
//              tree); the values of the best group so far are kept in
//              registers, and the position and second value inside it are
//              found once per row after the sweep.  Column parts of a row
//              meet in shared memory, and a rigorous error bound sends rows
//              whose top two are closer than the bound to the exact SIMT
//              kernels through a list.  Each warp loads the next 32 columns
//              from TMEM while it reduces the current ones.
// Every mbarrier wait is bounded; on time-out the kernel records an error
// code and leaves.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <float.h>

#include "kernels.cuh"
#include "tc_ptx.cuh"

namespace a2ats {
namespace tc {

constexpr int BM = 128;   // rows per row block (UMMA M)
constexpr int BK = 64;    // 16-bit elements per 128-byte swizzle atom
constexpr int kPadCols = 256;  // -|c L|^2 / 2 rows are padded to a multiple of this
constexpr int kEpiWarps = 8;   // 4 TMEM lane quarters x 2 (row blocks or column parts)
constexpr int kAWarp = 2 + kEpiWarps;          // the key-tile producer
constexpr int kThreads = 32 * (kAWarp + 1);

struct Params {
    int32_t H, d, K, P;        // P: codebook planes the pass multiplies
    int32_t pstride;           // planes stored per head in the B tensor map
    int32_t num_bh, seg, tiles_per_bh, nchunks, kpad;
    int32_t out_ncap;          // rows per (b, h) of the keys and of codes
    int64_t plane_rows;        // rows of one A plane in the A tensor map
    const int32_t* len;        // [B] or null
    const int32_t* count;      // compact list: rows per (b, h); null = natural order
    // compact list, two row planes: per 128-row tile, nonzero when a row of
    // it was rotated (else every second plane is zero and its MMAs are
    // skipped), [num_bh, tiles128]; or null
    const int32_t* tile_rot;
    int32_t tiles128;
    const int32_t* row_map;    // compact list: row of the keys each entry stands for,
                               // | kUnrotated when it was not rotated (its second
                               // plane is zero: the row operand is exact)
    const uint8_t* skip;       // rows to leave untouched (bulk mode), or null
    int32_t skip_near;         // natural order: rows with t - j < skip_near belong to
                               // the compact pass (0 = none)
    const float* hneg;         // [H, kpad]: -|c_j L|^2 / 2, -FLT_MAX past K (fp16)
    const uint16_t* hplanes;   // [H, kpad, 16]: the same as bf16 planes of the -h step (bf16)
    const float* head;         // [H, 4]: max |chat_j|, max h_j, 1/scale, abs error
    float err_coef;            // relative error bound of the contraction (host)
    float err_coef_unrot;      // the same for a compact row stored unrotated
    float norm_slack;          // |x| from plane 0 times this bounds |x|
    int32_t* codes;            // [num_bh * out_ncap]
    int64_t* exact_list;       // rows for the exact kernel
    int32_t* exact_count;
    int32_t* status;           // 0, or the code of a timed-out wait
    const int32_t* max_rows;   // compact list: longest list over (b, h), or null
    // per group of kTcGroup centroids: (max |chat_j|, max h_j), [H, ngroups]
    const float2* gstat;
    int32_t ngroups;
    // natural order over stored keys only (else null): the cosine of every
    // row of the pass with the query of its (b, h), and a copy of the row
    const float* sq;           // [num_bh, d] fp32 query
    const float* sqn;          // [num_bh] |query|
    float* scores;             // [num_bh * out_ncap], or null
    void* kcopy;               // [num_bh * out_ncap, d] 16-bit, or null
    int32_t kcopy_tma;         // tiles whose rows are all valid are copied by TMA
                               // stores through the third tensor map
};

// Flag in a compact row-map entry: the row was stored as it is (no rotation).
constexpr int32_t kUnrotated = 1 << 30;

__device__ __forceinline__ float max3f(float a, float b, float c) {
    float r;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}
// (bits & ~15) | pos: a column position in the four low mantissa bits, so
// that the top-2 network below also yields where the largest value sits; the
// key is within 15 units in the last place of the value.
__device__ __forceinline__ float embed_pos(float v, uint32_t pos) {
    return __uint_as_float((__float_as_uint(v) & ~15u) | pos);
}

// Largest of 16 values: a tree of three-input maxima (8 instructions).
__device__ __forceinline__ float max_16(const float* v) {
    const float a0 = max3f(v[0], v[1], v[2]), a1 = max3f(v[3], v[4], v[5]);
    const float a2 = max3f(v[6], v[7], v[8]), a3 = max3f(v[9], v[10], v[11]);
    const float a4 = max3f(v[12], v[13], v[14]);
    return fmaxf(max3f(a0, a1, a2), max3f(a3, a4, v[15]));
}

// Top two of 16 keys: min/max of pairs, then a merge tree of (max, second)
// pairs where each merge is max(h1, h2) and max3(min(h1, h2), l1, l2).
__device__ __forceinline__ void top2_16(const float* k, float& t1, float& t2) {
    float hi[8], lo[8];
#pragma unroll
    for (int i = 0; i < 8; i++) {
        hi[i] = fmaxf(k[2 * i], k[2 * i + 1]);
        lo[i] = fminf(k[2 * i], k[2 * i + 1]);
    }
#pragma unroll
    for (int w = 4; w >= 1; w >>= 1) {
#pragma unroll
        for (int i = 0; i < w; i++) {
            const float h = fmaxf(hi[i], hi[i + w]);
            lo[i] = max3f(fminf(hi[i], hi[i + w]), lo[i], lo[i + w]);
            hi[i] = h;
        }
    }
    t1 = hi[0];
    t2 = lo[0];
}

// The decision for one row of a pass.  Every value the contraction yields is
// off from the exact x . chat_j - h_j by at most err_coef (|x| |chat_j| + h_j)
// (plus the absolute fp16 term), which is bounded group by group with the
// group maxima of |chat_j| and h_j: s_g = alpha max|chat| + beta max h over
// group g of kTcGroup centroids.  The row carries m1, its best value, at
// centroid code (group code / kTcGroup) whose group bound is s1; U, an upper
// bound of the exact value of every other centroid (the largest t1_g + s_g
// over the other groups, and the second value of the code's own group plus
// its s); the code is certified when m1 - s1 still exceeds U, with room for
// the rounding of the comparison and the absolute term (abs_xn: the absolute
// fp16 term for this row), else the row joins the exact list.  Lb: the
// sequence length of the row's (b, h).
__device__ __forceinline__ void decide_row(const Params& p, int32_t bh, int32_t ri, int32_t Lb,
                                           float m1, float U, int32_t code, float s1,
                                           float abs_xn) {
    const int32_t j = p.row_map ? (p.row_map[(int64_t)bh * p.seg + ri] & ~kUnrotated) : ri;
    if (j < 0 || j >= Lb) return;
    const int64_t out = (int64_t)bh * p.out_ncap + j;
    if (p.skip && p.skip[out]) return;
    const float mag = fmaxf(fabsf(m1), fabsf(U));
    const float tau = s1 + 2.f * abs_xn + 4.f * mag * 1.1920929e-07f;
    if (!(m1 - U > tau)) {
        const int32_t slot = atomicAdd(p.exact_count, 1);
        p.exact_list[slot] = out;
    } else {
        p.codes[out] = code;
    }
}

struct TileInfo {
    int32_t bh, r0, nvalid;
    bool skip;
};

// Tile t of a pass covers rows r0 .. r0 + rows - 1 of (b, h) bh.
__device__ __forceinline__ TileInfo tile_info(const Params& p, int t, int tpb, int rows) {
    TileInfo ti;
    ti.bh = t / tpb;
    ti.r0 = (t % tpb) * rows;
    if (p.count) {
        ti.nvalid = min(max(p.count[ti.bh], 0), p.seg);
    } else {
        ti.nvalid = seq_len(p.len, ti.bh / p.H, p.out_ncap);
        // rows of the compact pass never enter this tile
        if (p.skip_near > 0) ti.nvalid = max(ti.nvalid - p.skip_near, 0);
    }
    ti.skip = ti.r0 >= ti.nvalid;
    return ti;
}

// RB row blocks of BM rows share each codebook stage: with RB = 2 a tile is
// 256 rows, and the accumulators are 128 columns wide (RB x 2 buffers x BN
// columns fill the 512 TMEM columns).
template <int RB>
struct Geo {
    static constexpr int kBN = RB == 2 ? 128 : 256;  // centroids per accumulator (UMMA N)
    static constexpr int kParts = 2 / RB;             // column parts of a chunk
    static constexpr int kSubs = kBN / 32 / kParts;   // 32-column loads per part per chunk
    static constexpr int kRows = BM * RB;             // rows per tile
};

// -|c'|^2/2 per chunk.  Folded (bf16 operands): the B operand of one more
// K = 16 step, kBN rows of 32 bytes holding -h_j as three bf16 planes
// (elements 0-2, zeros after), copied into the chunk's first codebook stage;
// the MMA issuer multiplies it by a constant tile of ones so that each
// accumulator starts at -h_j.  Else kBN floats per chunk in a ring of their
// own, added by the epilogue, which lets the codebook stream run ahead of
// the epilogue.
template <bool FOLD, int RB>
struct HRing {
    static constexpr int kSlots = FOLD ? 0 : 8;
    static constexpr int kSlotBytes = Geo<RB>::kBN * 4;
};

template <bool FOLD, int DK, int PA, int AST, int BST, int RB>
struct Smem {
    using G = Geo<RB>;
    using R = HRing<FOLD, RB>;
    static constexpr int kA = BM * 128;        // one 64-element k-block of one A plane
    // a codebook stage holds KS k-blocks of one plane (all of them up to
    // d = 128: one handshake per chunk and plane), and in a chunk's first
    // stage the folded -h tile after them
    static constexpr int KS = DK <= 2 ? DK : 1;
    static constexpr int kBk = G::kBN * 128;   // one k-block of one plane
    static constexpr int kHT = FOLD ? G::kBN * 32 : 0;
    static constexpr int kB = (KS * kBk + kHT + 1023) / 1024 * 1024;  // one B stage
    static constexpr int kABytes = AST * RB * PA * DK * kA;
    static constexpr int kBBytes = BST * kB;
    static constexpr int kHOff = kABytes + kBBytes;          // the -h ring (unfolded)
    static constexpr int kOnesOff = kHOff + R::kSlots * R::kSlotBytes;  // folded: BM x 32 bytes
    static constexpr int kBarOff = kOnesOff + (FOLD ? BM * 32 : 0);
    static constexpr int kBars = 2 * AST + 2 * BST + 10 + 2 * R::kSlots;
    static constexpr int kMergeOff = kBarOff + kBars * 8 + 16;
    static constexpr int kNrmOff = kMergeOff + (G::kParts - 1) * 2 * 4 * 32 * 16;
    static constexpr int kQOff = kNrmOff + 2 * G::kParts * BM * 8;  // [AST][kMaxD] fp32 queries
    static constexpr int kTotal = kQOff + AST * kMaxD * 4 + 1024;  // + alignment slack
};

template <bool BF16, int DK, int PA, int AST, int BST, int RB>
__global__ void __launch_bounds__(kThreads, 1)
assign_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                 const __grid_constant__ CUtensorMap tmK, const Params p) {
    // bf16 operands take -h_j into the MMAs (an exact three-plane split);
    // fp16 planes carry a per-head scale, and their epilogue adds -h_j
    constexpr bool FOLD = BF16;
    static_assert(PA == 1 || RB == 1, "two row planes take one row block per tile");
    using S = Smem<FOLD, DK, PA, AST, BST, RB>;
    using G = Geo<RB>;
    constexpr int BN = G::kBN, kParts = G::kParts, kSubs = G::kSubs, kRows = G::kRows;
    constexpr int kHS = HRing<FOLD, RB>::kSlots, kHBytes = HRing<FOLD, RB>::kSlotBytes;
    constexpr int KS = S::KS, kGroups = DK / KS;  // k-blocks per stage, stages per plane
    constexpr int kHSd = kHS > 0 ? kHS : 1;       // the h ring's size as a divisor
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
    uint8_t* smA = sm;
    uint8_t* smB = sm + S::kABytes;
    uint8_t* smH = sm + S::kHOff;
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + S::kBarOff);
    uint64_t* a_full = bars;
    uint64_t* a_empty = bars + AST;
    uint64_t* b_full = bars + 2 * AST;
    uint64_t* b_empty = bars + 2 * AST + BST;
    uint64_t* acc_full = bars + 2 * AST + 2 * BST;
    uint64_t* acc_empty = acc_full + 2;
    uint64_t* h_full = acc_full + 4;
    uint64_t* h_empty = h_full + kHS;
    uint64_t* merge_full = h_empty + kHS;  // column-part handoff, after the h ring
    uint64_t* merge_empty = merge_full + 1;
    uint64_t* nrm_full = merge_full + 2;       // [4] one per TMEM lane quarter: row-norm partials
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + S::kBars);
    float4* merge = reinterpret_cast<float4*>(sm + S::kMergeOff);
    // [2][kParts][BM] partial (|x|^2, x . q) of each row (column parts only)
    float2* nrm_part = reinterpret_cast<float2*>(sm + S::kNrmOff);
    float* smQ = reinterpret_cast<float*>(sm + S::kQOff);  // the tile's query, per A stage
    // k-block kb of plane pa of row block rb in A stage sa
    auto a_block = [&](int sa, int rb, int pa, int kb) {
        return smA + (((sa * RB + rb) * PA + pa) * DK + kb) * S::kA;
    };

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // tiles per (b, h): the host's bound, cut to the longest compact list
    // when its length is on the device (the tiles past it hold no row)
    int tpb = p.tiles_per_bh;
    if (p.max_rows) tpb = min(tpb, (max(*p.max_rows, 0) + kRows - 1) / kRows);
    const int total_tiles = p.num_bh * tpb;

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
        for (int i = 0; i < kHS; i++) {
            mbar_init(&h_full[i], 1);
            mbar_init(&h_empty[i], FOLD ? 1 : kEpiWarps);  // folded: released by an MMA commit
        }
        mbar_init(merge_full, 4);   // the part-1 warps hand over (two column parts)
        mbar_init(merge_empty, 4);  // the part-0 warps take the handoff
        for (int i = 0; i < 4; i++) mbar_init(&nrm_full[i], kParts);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if constexpr (FOLD) {
        // the A operand of the -h step: BM rows whose elements 0-2 are 1 (bf16)
        // and the rest 0, in the 32-byte swizzle
        uint4* ones = reinterpret_cast<uint4*>(sm + S::kOnesOff);
        for (int i = threadIdx.x; i < BM * 2; i += kThreads) {
            const int r = i >> 1, half = i & 1;
            ones[i] = half == ((r >> 2) & 1) ? make_uint4(0x3F803F80u, 0x3F80u, 0u, 0u)
                                             : make_uint4(0u, 0u, 0u, 0u);
        }
        // the generic-proxy stores are visible to the tensor core's reads
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         su32(tmem_holder)),
                     "r"(2 * RB * BN)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;

    if (warp == kAWarp) {
        // ---------------------------------------------- key-tile producer --
        // the rows of each tile (and its query), issued as soon as a stage
        // is free, a whole tile ahead of the MMAs that read them
        if (lane == 0) {
            uint32_t a_it = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < total_tiles && ok; t += gridDim.x) {
                const TileInfo ti = tile_info(p, t, tpb, kRows);
                if (ti.skip) continue;
                const int sa = a_it % AST;
                ok = mbar_wait(&a_empty[sa], ((a_it / AST) & 1) ^ 1, p.status, 1);
                if (!ok) break;
                mbar_expect_tx(&a_full[sa], RB * PA * DK * S::kA + (p.sq ? p.d * 4 : 0));
                const int row0 = ti.bh * p.seg + ti.r0;
#pragma unroll
                for (int rb = 0; rb < RB; rb++)
#pragma unroll
                    for (int pa = 0; pa < PA; pa++)
#pragma unroll
                        for (int kb = 0; kb < DK; kb++)
                            tma_2d(a_block(sa, rb, pa, kb), &tmA, &a_full[sa], kb * BK,
                                   (int)(pa * p.plane_rows) + row0 + rb * BM);
                if (p.sq)
                    asm volatile(
                        "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], "
                        "[%1], %2, [%3];" ::"r"(su32(smQ + sa * kMaxD)),
                        "l"(p.sq + (int64_t)ti.bh * p.d), "r"(p.d * 4), "r"(su32(&a_full[sa]))
                        : "memory");
                a_it++;
            }
            // every issued copy has landed before the CTA may leave
            for (int s = 0; s < AST; s++)
                if (a_it > (uint32_t)s) {
                    const uint32_t last = a_it - 1 - ((a_it - 1 - s) % AST);
                    mbar_wait(&a_full[last % AST], (last / AST) & 1, p.status, 3);
                }
        }
    } else if (warp == 0) {
        // ---------------------------------------------- codebook producer --
        if (lane == 0) {
            uint32_t b_it = 0, h_it = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < total_tiles && ok; t += gridDim.x) {
                const TileInfo ti = tile_info(p, t, tpb, kRows);
                if (ti.skip) continue;
                const int h = ti.bh % p.H;
                for (int c = 0; c < p.nchunks && ok; c++) {
                    const int64_t hrow = (int64_t)h * p.kpad + c * BN;
                    if constexpr (!FOLD) {
                        const int hs = h_it % kHSd;
                        ok = mbar_wait(&h_empty[hs], ((h_it / kHSd) & 1) ^ 1, p.status, 11);
                        if (!ok) break;
                        mbar_expect_tx(&h_full[hs], kHBytes);
                        asm volatile(
                            "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], "
                            "[%1], %2, [%3];" ::"r"(su32(smH + hs * kHBytes)),
                            "l"(p.hneg + hrow), "r"(kHBytes), "r"(su32(&h_full[hs]))
                            : "memory");
                        h_it++;
                    }
                    for (int pl = 0; pl < p.P && ok; pl++)
                        for (int g = 0; g < kGroups; g++) {
                            const int sb = b_it % BST;
                            ok = mbar_wait(&b_empty[sb], ((b_it / BST) & 1) ^ 1, p.status, 2);
                            if (!ok) break;
                            // the chunk's first stage also carries the -h tile
                            const bool with_h = FOLD && pl == 0 && g == 0;
                            mbar_expect_tx(&b_full[sb], KS * S::kBk + (with_h ? S::kHT : 0));
                            uint8_t* stage = smB + sb * S::kB;
#pragma unroll
                            for (int k = 0; k < KS; k++)
                                tma_3d(stage + k * S::kBk, &tmB, &b_full[sb], (g * KS + k) * BK,
                                       c * BN, h * p.pstride + pl);
                            if (with_h)
                                asm volatile(
                                    "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes "
                                    "[%0], [%1], %2, [%3];" ::"r"(su32(stage + KS * S::kBk)),
                                    "l"(p.hplanes + hrow * 16), "r"(S::kHT),
                                    "r"(su32(&b_full[sb]))
                                    : "memory");
                            b_it++;
                        }
                }
            }
            // every issued copy has landed before the CTA may leave
            for (int s = 0; s < BST; s++)
                if (b_it > (uint32_t)s) {
                    const uint32_t last = b_it - 1 - ((b_it - 1 - s) % BST);
                    mbar_wait(&b_full[last % BST], (last / BST) & 1, p.status, 3);
                }
            for (int s = 0; s < kHS; s++)
                if (h_it > (uint32_t)s) {
                    const uint32_t last = h_it - 1 - ((h_it - 1 - s) % kHSd);
                    mbar_wait(&h_full[last % kHSd], (last / kHSd) & 1, p.status, 3);
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
                const TileInfo ti = tile_info(p, t, tpb, kRows);
                if (ti.skip) continue;
                const int sa = a_it % AST;
                ok = mbar_wait(&a_full[sa], (a_it / AST) & 1, p.status, 4);
                if (!ok) break;
                tc_fence_after();
                uint64_t a_desc[RB][PA][DK];
#pragma unroll
                for (int rb = 0; rb < RB; rb++)
#pragma unroll
                    for (int pa = 0; pa < PA; pa++)
#pragma unroll
                        for (int kb = 0; kb < DK; kb++)
                            a_desc[rb][pa][kb] = sw128_desc(su32(a_block(sa, rb, pa, kb)));
                // each row block of valid rows only is copied out whole by
                // TMA stores (rows ti.r0 + rb BM .. + BM of (b, h) ti.bh; the
                // coordinates are non-negative and x is a multiple of 64
                // elements)
                bool stored = false;
                if (p.kcopy_tma) {
#pragma unroll
                    for (int rb = 0; rb < RB; rb++) {
                        if (ti.r0 + (rb + 1) * BM > ti.nvalid) continue;
                        if (!stored) asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                        stored = true;
#pragma unroll
                        for (int kb = 0; kb < DK; kb++)
                            tma_store_3d(&tmK, a_block(sa, rb, 0, kb), kb * BK, ti.r0 + rb * BM,
                                         ti.bh);
                    }
                    if (stored) bulk_commit();
                }
                // the row's second plane is needed only when the tile holds a
                // rotated row (one 128-row block per tile with two planes)
                const bool lo_needed =
                    PA == 1 || !p.tile_rot ||
                    p.tile_rot[(int64_t)ti.bh * p.tiles128 + ti.r0 / BM] != 0;
                for (int c = 0; c < p.nchunks && ok; c++) {
                    const int acc = acc_it & 1;
                    ok = mbar_wait(&acc_empty[acc], ((acc_it >> 1) & 1) ^ 1, p.status, 5);
                    if (!ok) break;
                    tc_fence_after();
                    uint32_t accumulate[RB];
#pragma unroll
                    for (int rb = 0; rb < RB; rb++) accumulate[rb] = 0;
                    for (int pl = 0; pl < p.P && ok; pl++)
#pragma unroll
                        for (int g = 0; g < kGroups; g++) {
                            const int sb = b_it % BST;
                            ok = mbar_wait(&b_full[sb], (b_it / BST) & 1, p.status, 6);
                            if (!ok) break;
                            tc_fence_after();
                            uint8_t* stage = smB + sb * S::kB;
                            if (FOLD && pl == 0 && g == 0) {
                                // D = ones x (-h planes)^T starts each
                                // accumulator at -h_j
                                const uint64_t od = sw32_desc(su32(sm + S::kOnesOff));
                                const uint64_t hd = sw32_desc(su32(stage + KS * S::kBk));
#pragma unroll
                                for (int rb = 0; rb < RB; rb++) {
                                    tc_mma(tmem + (uint32_t)((acc * RB + rb) * BN), od, hd, idesc,
                                           0u);
                                    accumulate[rb] = 1;
                                }
                            }
#pragma unroll
                            for (int k = 0; k < KS; k++) {
                                const int kb = g * KS + k;
                                // descriptors of the k-block's start; the k-steps of
                                // 16 elements are 32 bytes apart, i.e. +2 in the
                                // address field (no carry: shared addresses are
                                // below 2^18)
                                const uint64_t bd = sw128_desc(su32(stage + k * S::kBk));
#pragma unroll
                                for (int rb = 0; rb < RB; rb++) {
                                    const uint32_t d_tmem = tmem + (uint32_t)((acc * RB + rb) * BN);
#pragma unroll
                                    for (int pa = 0; pa < PA; pa++) {
                                        // the row's second plane multiplies chat's
                                        // first only (the bound counts the rest)
                                        if (pa > 0 && (pl > 0 || !lo_needed)) continue;
                                        const uint64_t ad = a_desc[rb][pa][kb];
#pragma unroll
                                        for (int ks = 0; ks < BK / 16; ks++) {
                                            tc_mma(d_tmem, ad + 2 * ks, bd + 2 * ks, idesc,
                                                   accumulate[rb]);
                                            accumulate[rb] = 1;
                                        }
                                    }
                                }
                            }
                            tc_commit(&b_empty[sb]);
                            b_it++;
                        }
                    tc_commit(&acc_full[acc]);
                    acc_it++;
                }
                // the stores have read the tile before the stage is released
                if (stored) bulk_wait_read();
                tc_commit(&a_empty[sa]);
                a_it++;
            }
            bulk_wait_all();
        }
    } else if (warp < kAWarp) {
        // ------------------------------------------------------ epilogue --
        // warp (quarter q, e): with two row blocks, e is the row block and
        // the warp takes every column; with one, e is the column part
        const int ew = warp - 2;
        const int q = warp & 3;          // TMEM lane quarter this warp may access
        const int rb = RB == 2 ? (ew >> 2) : 0;
        const int part = RB == 2 ? 0 : (ew >> 2);
        const int row_in_tile = rb * BM + 32 * q + lane;
        uint32_t a_it = 0, acc_it = 0, m_it = 0, t_it = 0;
        bool ok = true;
        for (int t = blockIdx.x; t < total_tiles && ok; t += gridDim.x) {
            const TileInfo ti = tile_info(p, t, tpb, kRows);
            if (ti.skip) continue;
            const int h = ti.bh % p.H;
            const int sa = a_it % AST;
            ok = mbar_wait(&a_full[sa], (a_it / AST) & 1, p.status, 7);
            if (!ok) break;
            // |x|^2 of this row from the swizzled tile of plane 0: each column
            // part sums its share of the row's 16-byte chunks, the partials
            // meet in shared memory (an mbarrier per lane quarter) and every
            // part adds them in the same order.  With scores on, the same pass
            // takes x . q and copies the row's chunks out.
            const int32_t ri = ti.r0 + row_in_tile;
            const bool sc = p.scores != nullptr;
            float nrm = 0.f, dot = 0.f;
            {
                constexpr int kChunks = 8 * DK / kParts;  // 16-byte chunks per part
                // rows of a block that the TMA stores do not copy
                const bool by_tma = p.kcopy_tma && ti.r0 + (rb + 1) * BM <= ti.nvalid;
                uint8_t* kc = (p.kcopy && !by_tma && ri < ti.nvalid)
                                  ? reinterpret_cast<uint8_t*>(p.kcopy) +
                                        ((int64_t)ti.bh * p.out_ncap + ri) * p.d * 2
                                  : nullptr;
                const float* qrow = smQ + sa * kMaxD;
                const int rr_in_block = 32 * q + lane;
                float2 nrm2 = make_float2(0.f, 0.f), dot2 = make_float2(0.f, 0.f);
#pragma unroll 4
                for (int ci = part * kChunks; ci < (part + 1) * kChunks; ci++) {
                    const int kb = ci >> 3, c = ci & 7;
                    const uint8_t* rowp = a_block(sa, rb, 0, kb) + rr_in_block * 128;
                    const uint4 raw =
                        *reinterpret_cast<const uint4*>(rowp + 16 * (c ^ (rr_in_block & 7)));
                    if (kc) __stcs(reinterpret_cast<uint4*>(kc + (kb * 64 + c * 8) * 2), raw);
                    float qv[8];
                    if (sc) {
                        const float4* q4 = reinterpret_cast<const float4*>(qrow + kb * 64 + c * 8);
                        const float4 qa = q4[0], qb = q4[1];
                        qv[0] = qa.x; qv[1] = qa.y; qv[2] = qa.z; qv[3] = qa.w;
                        qv[4] = qb.x; qv[5] = qb.y; qv[6] = qb.z; qv[7] = qb.w;
                    }
                    const uint32_t w4[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
                    for (int u = 0; u < 4; u++) {
                        float2 f;
                        if (BF16) {
                            f = make_float2(__uint_as_float(w4[u] << 16),
                                            __uint_as_float(w4[u] & 0xFFFF0000u));
                        } else {
                            f = __half22float2(*reinterpret_cast<const __half2*>(&w4[u]));
                        }
                        nrm2 = __ffma2_rn(f, f, nrm2);
                        if (sc) dot2 = __ffma2_rn(f, make_float2(qv[2 * u], qv[2 * u + 1]), dot2);
                    }
                }
                nrm = nrm2.x + nrm2.y;
                dot = dot2.x + dot2.y;
                if (kParts > 1) {
                    float2* np = nrm_part + (t_it & 1) * kParts * BM;
                    np[part * BM + rr_in_block] = make_float2(nrm, dot);
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&nrm_full[q]);
                    ok = mbar_wait(&nrm_full[q], t_it & 1, p.status, 13);
                    nrm = 0.f;
                    dot = 0.f;
#pragma unroll
                    for (int pp = 0; pp < kParts; pp++) {
                        const float2 v = np[pp * BM + rr_in_block];
                        nrm += v.x;
                        dot += v.y;
                    }
                    t_it++;
                }
            }
            // cosine of the row with its query; 0 when either norm is 0
            if (ok && sc && part == kParts - 1 && ri < ti.nvalid) {
                const float qn = p.sqn[ti.bh];
                const float kn = sqrtf(nrm);
                p.scores[(int64_t)ti.bh * p.out_ncap + ri] =
                    (kn > 0.f && qn > 0.f) ? dot / (kn * qn) : 0.f;
            }
            if (!ok) break;
            __syncwarp();
            if (lane == 0) mbar_arrive(&a_empty[sa]);
            a_it++;

            // Per group g of kTcGroup columns this warp takes only t1_g, the
            // largest value (a three-input max tree), and b_g = t1_g + s_g.  It
            // keeps m1 / c1, the best t1 so far and its group, with that
            // group's values (best), and ub1 / gb1 / ub2, the two largest b_g
            // and the group of the first.  The position of m1 inside its group
            // and the group's second value are worked out once, after the sweep.
            constexpr int kG = kTcGroup;
            constexpr int kGroupsPerPart = kSubs * 32 / kG;
            float m1 = -INFINITY, ub1 = -FLT_MAX, ub2 = -FLT_MAX, s1 = 0.f;
            int32_t c1 = 0, gb1 = -1;
            float best[kG];
            const float xn = sqrtf(nrm) * p.norm_slack;
            // a compact row stored without rotation is exact in its first
            // plane (the second is zero), so only the contraction's own
            // rounding and chat's count
            float coef = p.err_coef;
            if (p.row_map && ri < ti.nvalid) {
                const int32_t rm = p.row_map[(int64_t)ti.bh * p.seg + ri];
                if (rm >= 0 && (rm & kUnrotated)) coef = p.err_coef_unrot;
            }
            const float alpha = coef * xn, beta = coef;
            // per-tile values of the decision, loaded ahead of the sweep
            const int32_t Lb = seq_len(p.len, ti.bh / p.H, p.out_ncap);
            const float abs_xn = p.head[h * 4 + 3] * xn;
            const float2* gst = p.gstat + (int64_t)h * p.ngroups;
            const float inv_scale = FOLD ? 1.f : p.head[h * 4 + 2];
            const float2 inv2 = make_float2(inv_scale, inv_scale);
            for (int c = 0; c < p.nchunks && ok; c++) {
                const int acc = acc_it & 1;
                // this part's group bounds s_g for the chunk, loaded ahead
                const int g0 = (c * BN + part * kSubs * 32) / kG;
                float sg[kGroupsPerPart];
#pragma unroll
                for (int i = 0; i < kGroupsPerPart; i++) {
                    const float2 gs = __ldg(gst + g0 + i);
                    sg[i] = fmaf(alpha, gs.x, beta * gs.y);
                }
                const int hs = acc_it % kHSd;
                ok = (FOLD || mbar_wait(&h_full[hs], (acc_it / kHSd) & 1, p.status, 12)) &&
                     mbar_wait(&acc_full[acc], (acc_it >> 1) & 1, p.status, 8);
                if (!ok) break;
                tc_fence_after();
                const float* hrow = reinterpret_cast<const float*>(smH + hs * kHBytes);
                const uint32_t tbase =
                    tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)((acc * RB + rb) * BN);
                // the next 32 columns are loaded while the current ones are
                // reduced (the wait covers the load issued before it)
                uint32_t rr[2][32];
                A2ATS_TMEM_LD32(tbase + (uint32_t)(part * kSubs * 32), rr[0]);
                tmem_wait_ld();
                tmem_regs_ready(rr[0]);
#pragma unroll
                for (int sub = 0; sub < kSubs; sub++) {
                    const int col = (part * kSubs + sub) * 32;
                    if (sub + 1 < kSubs)
                        A2ATS_TMEM_LD32(tbase + (uint32_t)(col + 32), rr[(sub + 1) & 1]);
                    const uint32_t* r = rr[sub & 1];
                    const float4* h4 = reinterpret_cast<const float4*>(hrow + col);
                    float v[32];
                    if constexpr (FOLD) {
                        // the accumulator already holds x . chat_j - h_j
#pragma unroll
                        for (int u = 0; u < 32; u++) v[u] = __uint_as_float(r[u]);
                    } else {
#pragma unroll
                        for (int u = 0; u < 8; u++) {
                            const float4 hv = h4[u];
                            const float2 v01 = __ffma2_rn(
                                make_float2(__uint_as_float(r[4 * u]), __uint_as_float(r[4 * u + 1])),
                                inv2, make_float2(hv.x, hv.y));
                            const float2 v23 = __ffma2_rn(
                                make_float2(__uint_as_float(r[4 * u + 2]), __uint_as_float(r[4 * u + 3])),
                                inv2, make_float2(hv.z, hv.w));
                            v[4 * u + 0] = v01.x;
                            v[4 * u + 1] = v01.y;
                            v[4 * u + 2] = v23.x;
                            v[4 * u + 3] = v23.y;
                        }
                    }
#pragma unroll
                    for (int half = 0; half < 32 / kG; half++) {
                        const float* vg = v + half * kG;
                        const int gi = sub * (32 / kG) + half;
                        const float t1 = max_16(vg);
                        const float b1 = t1 + sg[gi];
                        if (b1 > ub1) {
                            ub2 = ub1;
                            ub1 = b1;
                            gb1 = g0 + gi;
                        } else {
                            ub2 = fmaxf(ub2, b1);
                        }
                        // a strictly larger group maximum replaces the kept
                        // group (equal ones keep the earlier columns);
                        // branch-free, so the work of consecutive groups
                        // interleaves
                        const bool upd = t1 > m1;
#pragma unroll
                        for (int i = 0; i < kG; i++) best[i] = upd ? vg[i] : best[i];
                        if (upd) {
                            m1 = t1;
                            c1 = g0 + gi;
                            s1 = sg[gi];
                        }
                    }
                    if (sub + 1 < kSubs) {
                        tmem_wait_ld();
                        tmem_regs_ready(rr[(sub + 1) & 1]);
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(&acc_empty[acc]);
                    if (!FOLD) mbar_arrive(&h_empty[hs]);
                }
                acc_it++;
            }
            if (!ok) break;
            // the kept group: the position of m1 (lowest index on equal
            // values) and w2, a bound of its other values plus s of the group
            int32_t code;
            float w2;
            {
                float key[kG];
#pragma unroll
                for (int i = 0; i < kG; i++) key[i] = embed_pos(best[i], kG - 1 - i);
                float k1, k2;
                top2_16(key, k1, k2);
                code = c1 * kG + (kG - 1 - (int32_t)(__float_as_uint(k1) & (kG - 1)));
                // the second value is within 15 units in the last place of k2
                w2 = k2 + 16.f * 1.1920929e-07f * fabsf(k2) + s1;
            }
            if (kParts == 1) {
                const float U = fmaxf(gb1 == code / kTcGroup ? ub2 : ub1, w2);
                if (ri < ti.nvalid) decide_row(p, ti.bh, ri, Lb, m1, U, code, s1, abs_xn);
            } else if (part != 0) {
                // merge the column parts of each row, then decide the row
                ok = mbar_wait(merge_empty, (m_it & 1) ^ 1, p.status, 9);
                if (!ok) break;
                float4* mg = merge + (q * 32 + lane) * 2;
                mg[0] = make_float4(m1, w2, __int_as_float(code), s1);
                mg[1] = make_float4(ub1, ub2, __int_as_float(gb1), 0.f);
                __syncwarp();
                if (lane == 0) mbar_arrive(merge_full);
            } else {
                ok = mbar_wait(merge_full, m_it & 1, p.status, 10);
                if (!ok) break;
                const float4* mg = merge + (q * 32 + lane) * 2;
                const float4 o0 = mg[0], o1 = mg[1];
                __syncwarp();
                if (lane == 0) mbar_arrive(merge_empty);
                // part 1 holds the later columns of each chunk: it takes the
                // row only with a strictly larger value
                if (o0.x > m1) {
                    m1 = o0.x;
                    w2 = o0.y;
                    code = __float_as_int(o0.z);
                    s1 = o0.w;
                }
                if (o1.x > ub1) {
                    ub2 = fmaxf(ub1, o1.y);
                    ub1 = o1.x;
                    gb1 = __float_as_int(o1.z);
                } else {
                    ub2 = fmaxf(ub2, o1.x);
                }
                const float U = fmaxf(gb1 == code / kTcGroup ? ub2 : ub1, w2);
                if (ri < ti.nvalid) decide_row(p, ti.bh, ri, Lb, m1, U, code, s1, abs_xn);
            }
            m_it++;
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "r"(2 * RB * BN)
                     : "memory");
    }
}

// -------------------------------------------------- codebook preparation --
// rot = RoPE(chat, -far_offset) for every centroid (far keys enter the
// contraction unrotated, so their shared rotation moves to the codebook).
__global__ void rotate_rows_kernel(const float* __restrict__ in, int64_t rows, int32_t d,
                                   const RopeArgs ra, float* __restrict__ out) {
    const int halfd = d / 2;
    for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < rows * halfd;
         e += (int64_t)gridDim.x * blockDim.x) {
        const int64_t r = e / halfd;
        const int i = (int)(e % halfd);
        const int a = ra.interleaved ? 2 * i : i;
        const int b = ra.interleaved ? 2 * i + 1 : i + halfd;
        float s, c;
        rope_angle(-ra.far_offset, ra.omega_hi[i], ra.omega_lo[i], ra, s, c);
        const float xa = in[r * d + a], xb = in[r * d + b];
        out[r * d + a] = fmaf(xa, c, -__fmul_rn(xb, s));
        out[r * d + b] = fmaf(xa, s, __fmul_rn(xb, c));
    }
}

// Per-head maxima into head_bits [H, 4] (uint bits of non-negative floats,
// zeroed by the caller): max |chat_j|, max h_j, max |element|.
__global__ void __launch_bounds__(256)
codebook_stats_kernel(const float* __restrict__ chat, int64_t K, int32_t d,
                      const float* __restrict__ half_norm, uint32_t* __restrict__ head_bits,
                      uint32_t* __restrict__ group_bits, int32_t ngroups) {
    // one warp per centroid, one head per block row; the block's maxima are
    // combined in shared memory first, so a head takes one atomic per block
    __shared__ float red[3][8];
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int64_t h = blockIdx.y;
    const int64_t j = (int64_t)blockIdx.x * 8 + w;
    float cm = 0.f, hm = 0.f, em = 0.f;
    if (j < K) {
        const float* row = chat + (h * K + j) * d;
        Dot2 n;
        for (int a = lane; a < d; a += 32) {
            const float v = row[a];
            n.add_prod(v, v);
            em = fmaxf(em, fabsf(v));
        }
        for (int m = 16; m; m >>= 1) {
            n.merge(shfl_xor(n, m));
            em = fmaxf(em, __shfl_xor_sync(0xffffffffu, em, m));
        }
        cm = sqrtf(n.value()) * 1.000001f;
        hm = fmaxf(half_norm[h * K + j], 0.f);
        // the same maxima per group of kTcGroup centroids (bits of
        // non-negative floats)
        if (lane == 0) {
            uint32_t* gb = group_bits + 2 * (h * ngroups + j / kTcGroup);
            atomicMax(gb, __float_as_uint(cm));
            atomicMax(gb + 1, __float_as_uint(hm));
        }
    }
    if (lane == 0) {
        red[0][w] = cm;
        red[1][w] = hm;
        red[2][w] = em;
    }
    __syncthreads();
    if (threadIdx.x < 3) {
        float v = 0.f;
        for (int ww = 0; ww < 8; ww++) v = fmaxf(v, red[threadIdx.x][ww]);
        atomicMax(&head_bits[h * 4 + threadIdx.x], __float_as_uint(v));
    }
}

// head [H, 4] floats from the raw maxima: max |chat|, max h, 1/scale, abs err.
// unit_scale: planes are bf16 or the raw 16-bit codebook (scale 1).  fp16
// planes: a power of two that puts the largest element near 2^14; elements in
// the fp16 subnormal range are covered by the absolute error term (per unit
// of |x|).
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

// hneg [H, kpad] = -half_norm, and -FLT_MAX past K (those columns never win).
// For bf16 operands the same values go into hplanes [H, kpad, 16] instead, as
// the B operand of the K = 16 step that starts each accumulator at -h_j:
// elements 0-2 of row j are three bf16 planes, each the truncation toward
// zero of what the planes before it leave (8 significant bits each, so their
// sum is the fp32 value exactly, -FLT_MAX included), elements 3-15 are zero,
// and the two 16-byte halves of row j are swapped when bit 2 of j is set: the
// 32-byte swizzle, so that a chunk of rows (a multiple of 8) copies into
// shared memory as the MMA reads it.
__global__ void hneg_planes_kernel(const float* __restrict__ half_norm, int64_t H, int64_t K,
                                   int64_t kpad, uint16_t* __restrict__ hplanes) {
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < H * kpad;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t h = i / kpad, j = i % kpad;
        float v = j < K ? -half_norm[h * K + j] : -FLT_MAX;
        uint32_t pl[3];
#pragma unroll
        for (int k = 0; k < 3; k++) {
            const uint32_t top = __float_as_uint(v) & 0xFFFF0000u;
            pl[k] = top >> 16;
            v = v - __uint_as_float(top);  // exact: the low 16 bits of the significand
        }
        const uint4 lo = make_uint4(pl[0] | (pl[1] << 16), pl[2], 0u, 0u);
        const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
        uint4* row = reinterpret_cast<uint4*>(hplanes + i * 16);
        const bool swap = (j >> 2) & 1;
        row[0] = swap ? zero : lo;
        row[1] = swap ? lo : zero;
    }
}
__global__ void pad_half_norm_kernel(const float* __restrict__ half_norm, int64_t H, int64_t K,
                                     int64_t kpad, float* __restrict__ hneg) {
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < H * kpad;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t h = i / kpad, j = i % kpad;
        hneg[i] = j < K ? -half_norm[h * K + j] : -FLT_MAX;
    }
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

// ------------------------------------------------------ compact rows --
// The rows of one pass that cannot use the stored keys as they are: rows
// inside the RoPE window (natural order), every retrieval row (routed mode 1)
// or the decode row (mode 3).  Each is rotated in fp32 and split into two 16-bit planes
// hi = rn(k~), lo = rn(k~ - hi); planes [2][nbh * ncap][d].  Rows whose fp16
// planes would overflow go to the exact list instead.
//
// Eight lanes take a row, 16 bytes at a time: with the two-halves layout lane
// e of the octet holds elements 8 ch .. 8 ch + 7 (ch = e, e + 8, ...) of both
// halves, i.e. whole rotation pairs; interleaved pairs sit inside one 16-byte
// chunk.  A block takes 32 rows per sweep, so a few thousand rows per (b, h)
// are one or two sweeps of a single wave of blocks.
constexpr int kCompactRows = 32;  // rows per block per sweep (8 warps x 4)

template <int DT>
__device__ __forceinline__ bool split_store8(const float* v, uint16_t* hi_p, uint16_t* lo_p) {
    uint32_t hw[4], lw[4];
    bool over = false;
#pragma unroll
    for (int u = 0; u < 8; u += 2) {
        uint16_t hb[2], lb[2];
#pragma unroll
        for (int k = 0; k < 2; k++) {
            const float x = v[u + k];
            if (DT == kBF16) {
                const __nv_bfloat16 hv = __float2bfloat16_rn(x);
                const __nv_bfloat16 lv = __float2bfloat16_rn(x - __bfloat162float(hv));
                hb[k] = __bfloat16_as_ushort(hv);
                lb[k] = __bfloat16_as_ushort(lv);
            } else {
                const __half hv = __float2half_rn(x);
                const __half lv = __float2half_rn(x - __half2float(hv));
                over |= !(fabsf(x) <= 65504.f);
                hb[k] = __half_as_ushort(hv);
                lb[k] = __half_as_ushort(lv);
            }
        }
        hw[u / 2] = (uint32_t)hb[0] | ((uint32_t)hb[1] << 16);
        lw[u / 2] = (uint32_t)lb[0] | ((uint32_t)lb[1] << 16);
    }
    *reinterpret_cast<uint4*>(hi_p) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
    *reinterpret_cast<uint4*>(lo_p) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
    return over;
}

template <int DT>
__global__ void __launch_bounds__(256)
compact_rows_kernel(const void* __restrict__ x, int32_t H, int32_t ncap, int32_t d,
                    const int32_t* __restrict__ len, const RopeArgs ra, int32_t mode,
                    const int32_t* __restrict__ perm, const int32_t* __restrict__ count,
                    uint16_t* __restrict__ planes, int32_t* __restrict__ row_map,
                    int32_t* __restrict__ ccount, int64_t* __restrict__ exact_list,
                    int32_t* __restrict__ exact_count, int32_t* __restrict__ tile_rot) {
    const int bh = blockIdx.y;
    const int32_t L = seq_len(len, bh / H, ncap);
    int32_t n;
    if (mode == 1) {
        n = min(max(count[bh], 0), L);
    } else if (mode == 3) {
        n = L > 0 ? 1 : 0;  // the decode row
    } else {
        n = (ra.enabled && ra.window > 0) ? min(L, ra.window) : 0;
    }
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        ccount[bh] = n;
        atomicMax(exact_count + 2, n);  // the longest list, for the contraction's tile bound
    }
    const int lane = threadIdx.x & 31, e = lane & 7;
    const int halfd = d / 2;
    const int64_t plane_rows = (int64_t)gridDim.y * ncap;
    uint16_t* lo_planes = planes + plane_rows * d;
    // i0 is the same for the whole block, so every warp runs each sweep whole
    // (the ballot below takes all its lanes)
    for (int32_t i0 = blockIdx.x * kCompactRows; i0 < n; i0 += gridDim.x * kCompactRows) {
        const int32_t i = i0 + (int32_t)(threadIdx.x >> 3);
        const bool active = i < n;
        int32_t j = -1;
        if (active) j = mode == 1 ? perm[(int64_t)bh * ncap + i] : L - n + i;  // mode 3: L - 1
        const bool valid = active && j >= 0 && j < L;
        bool over = false;
        int32_t pos_row = 0;
        if (valid) {
            const int64_t src = ((int64_t)bh * ncap + j) * d;
            const int64_t dst = ((int64_t)bh * ncap + i) * d;
            const int32_t pos = ra.enabled ? rope_position(j, L - 1, ra) : 0;
            pos_row = pos;
            if (!ra.interleaved) {
                for (int ch = e; ch < halfd / 8; ch += 8) {
                    float va[8], vb[8];
                    load_vec<DT>(x, src + 8 * ch, va);
                    load_vec<DT>(x, src + halfd + 8 * ch, vb);
                    if (pos != 0) {
#pragma unroll
                        for (int u = 0; u < 8; u++) {
                            float s, c;
                            rope_angle(pos, ra.omega_hi[8 * ch + u], ra.omega_lo[8 * ch + u], ra, s,
                                       c);
                            const float ya = fmaf(va[u], c, -__fmul_rn(vb[u], s));
                            const float yb = fmaf(va[u], s, __fmul_rn(vb[u], c));
                            va[u] = ya;
                            vb[u] = yb;
                        }
                    }
                    over |= split_store8<DT>(va, planes + dst + 8 * ch, lo_planes + dst + 8 * ch);
                    over |= split_store8<DT>(vb, planes + dst + halfd + 8 * ch,
                                             lo_planes + dst + halfd + 8 * ch);
                }
            } else {
                for (int ch = e; ch < d / 8; ch += 8) {
                    float v[8];
                    load_vec<DT>(x, src + 8 * ch, v);
                    if (pos != 0) {
#pragma unroll
                        for (int u = 0; u < 4; u++) {
                            const int pi = 4 * ch + u;
                            float s, c;
                            rope_angle(pos, ra.omega_hi[pi], ra.omega_lo[pi], ra, s, c);
                            const float xa = v[2 * u], xb = v[2 * u + 1];
                            v[2 * u] = fmaf(xa, c, -__fmul_rn(xb, s));
                            v[2 * u + 1] = fmaf(xa, s, __fmul_rn(xb, c));
                        }
                    }
                    over |= split_store8<DT>(v, planes + dst + 8 * ch, lo_planes + dst + 8 * ch);
                }
            }
        }
        // any lane of the row's octet
        over = ((__ballot_sync(0xffffffffu, over) >> (lane & ~7)) & 0xFFu) != 0;
        if (e == 0 && active) {
            if (!valid) {
                row_map[(int64_t)bh * ncap + i] = -1;
            } else if (over) {
                row_map[(int64_t)bh * ncap + i] = -1;
                exact_list[atomicAdd(exact_count, 1)] = (int64_t)bh * ncap + j;
            } else {
                row_map[(int64_t)bh * ncap + i] = j | (pos_row == 0 ? kUnrotated : 0);
                if (pos_row != 0) tile_rot[(int64_t)bh * ((ncap + 127) / 128) + i / 128] = 1;
            }
        }
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

// ------------------------------------------------------ exact list kernels --
// Rows the contraction could not decide, in two short launches so that a
// handful of rows still spreads over the whole GPU:
//   exact_rows_kernel   one block per listed row: windowed RoPE in fp32 and
//                       z = x L (compensated) into zbuf; best <- +inf; the
//                       row joins its head's list
//   exact_scan_kernel   one block per (head, slice of centroids, chunk of the
//                       head's rows): the slice is staged in shared memory
//                       once and every row of the chunk takes the direct
//                       distance sum_b (z_b - cp_jb)^2 to each cp_j = c_j L;
//                       a 64-bit atomicMin on (distance bits, j) merges the
//                       slices, so ties go to the lowest index, and the
//                       slice that finishes a row last writes its code
constexpr int kExactThreads = 256;

template <int DT>
__global__ void __launch_bounds__(kExactThreads)
exact_rows_kernel(const void* __restrict__ x, int32_t H, int32_t ncap, int32_t d,
                  const int32_t* __restrict__ len, const RopeArgs ra, const float* __restrict__ L,
                  const int64_t* __restrict__ list, const int32_t* __restrict__ list_count,
                  float* __restrict__ zbuf, unsigned long long* __restrict__ best,
                  int32_t* __restrict__ done, int32_t* __restrict__ head_count,
                  int32_t* __restrict__ head_rows, int64_t head_cap) {
    __shared__ __align__(16) float xv[kMaxD];
    __shared__ Dot2 part[kExactThreads];
    const int tid = threadIdx.x;
    const int n = *list_count;
    for (int e = blockIdx.x; e < n; e += gridDim.x) {
        const int64_t out = list[e];
        const int64_t bh = out / ncap;
        const int32_t j = (int32_t)(out % ncap);
        const int64_t h = bh % H;
        const int32_t Lb = seq_len(len, (int32_t)(bh / H), ncap);
        for (int a = tid; a < d; a += blockDim.x) xv[a] = load1<DT>(x, out * d + a);
        __syncthreads();
        if (ra.enabled) {
            const int32_t pos = rope_position(j, Lb - 1, ra);
            const int halfd = d / 2;
            if (pos != 0 && tid < halfd) {
                float sn, cs;
                rope_angle(pos, ra.omega_hi[tid], ra.omega_lo[tid], ra, sn, cs);
                const int a = ra.interleaved ? 2 * tid : tid;
                const int b = ra.interleaved ? 2 * tid + 1 : tid + halfd;
                const float xa = xv[a], xb = xv[b];
                xv[a] = fmaf(xa, cs, -__fmul_rn(xb, sn));
                xv[b] = fmaf(xa, sn, __fmul_rn(xb, cs));
            }
            __syncthreads();
        }
        float* z = zbuf + (int64_t)e * d;
        if (L) {
            // P groups of threads split the rows of L into spans of a
            // multiple of 32 rows; group g sums rows [g d / P, (g + 1) d / P)
            // of column b (d % 32 == 0)
            const int P = min((int)blockDim.x / d, d / 32);
            const int g = tid / d, b = tid - g * d;
            const int span = d / P;
            if (g < P) {
                const float* Lh = L + h * d * d + b;
                Dot2 acc;
                for (int a0 = g * span; a0 < (g + 1) * span; a0 += 32) {
                    float l[32];
#pragma unroll
                    for (int u = 0; u < 32; u++) l[u] = __ldg(Lh + (int64_t)(a0 + u) * d);
#pragma unroll
                    for (int u = 0; u < 32; u++) acc.add_prod(xv[a0 + u], l[u]);
                }
                part[g * d + b] = acc;
            }
            __syncthreads();
            if (tid < d) {
                Dot2 acc = part[tid];
                for (int gg = 1; gg < P; gg++) acc.merge(part[gg * d + tid]);
                z[tid] = acc.value();
            }
        } else {
            for (int b = tid; b < d; b += blockDim.x) z[b] = xv[b];
        }
        if (tid == 0) {
            best[e] = ~0ull;
            done[e] = 0;
            head_rows[h * head_cap + atomicAdd(head_count + h, 1)] = e;
        }
        __syncthreads();
    }
}

// Rows of a warp per chunk of a head's rows for long lists: four with the
// 64-centroid slices of d > 128 (an LDS serves four rows); two with
// 128-centroid slices, where more rows would cost a block per SM (eight were
// slower on the long-context workload); a head whose list fits the grid's
// chunk groups in chunks of two rows per warp takes those.
template <int S> struct ScanTile { static constexpr int kRT = S == 128 ? 2 : 4; };

// One warp's rows r0 .. r0 + nr - 1 of head list `rows` against the staged
// slice (see exact_scan_kernel): z staged transposed in zT, then per pair of
// centroids (l + 64 m, l + 64 m + 32) packed differences and squares.
template <int S, int RT>
__device__ __forceinline__ void scan_rows(const float* cT, float* zT, int d, int nc, int64_t j0,
                                          const int32_t* rows, int r0, int nr, const float* zbuf,
                                          unsigned long long* best, int32_t* done,
                                          const int64_t* list, int32_t* codes, int lane) {
    constexpr int CT = S / 32;
    // z of the warp's rows, transposed (a missing row repeats the first)
    for (int i = lane; i < RT * d; i += 32) {
        const int r = i / d, a = i - r * d;
        const int64_t e = rows[r0 + (r < nr ? r : 0)];
        zT[a * RT + r] = __ldg(zbuf + e * d + a);
    }
    __syncwarp();
    // acc[r][m]: distances of row r to l + 64 m and l + 64 m + 32
    float2 acc[RT][CT / 2];
#pragma unroll
    for (int r = 0; r < RT; r++)
#pragma unroll
        for (int m = 0; m < CT / 2; m++) acc[r][m] = make_float2(0.f, 0.f);
    const float2 neg1 = make_float2(-1.f, -1.f);
    constexpr int kUnroll = RT <= 2 ? 4 : 2;  // registers of the row tile
#pragma unroll kUnroll
    for (int a = 0; a < d; a++) {
        const float* col = cT + a * (S + 1) + lane;
        float2 cv[CT / 2];
#pragma unroll
        for (int m = 0; m < CT / 2; m++) cv[m] = make_float2(col[64 * m], col[64 * m + 32]);
        const float2* z2 = reinterpret_cast<const float2*>(zT + a * RT);
#pragma unroll
        for (int q = 0; q < RT / 2; q++) {
            const float2 zq = z2[q];
#pragma unroll
            for (int u = 0; u < 2; u++) {
                const float zr = u ? zq.y : zq.x;
                const float2 za = make_float2(zr, zr);
#pragma unroll
                for (int m = 0; m < CT / 2; m++) {
                    const float2 t = __ffma2_rn(cv[m], neg1, za);  // za - c, exact negation
                    acc[2 * q + u][m] = __ffma2_rn(t, t, acc[2 * q + u][m]);
                }
            }
        }
    }
    __syncwarp();  // zT is rewritten by the warp's next rows
#pragma unroll
    for (int r = 0; r < RT; r++) {
        if (r >= nr) break;
        const int64_t e = rows[r0 + r];
        float bv = INFINITY;
        int32_t bj = 0;
#pragma unroll
        for (int k = 0; k < CT; k++) {  // ascending j: strict < keeps the lowest
            const float v = (k & 1) ? acc[r][k >> 1].y : acc[r][k >> 1].x;
            const int c = lane + 32 * k;
            if (c < nc && v < bv) {
                bv = v;
                bj = (int32_t)(j0 + c);
            }
        }
        for (int m = 16; m; m >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, bv, m);
            const int32_t oj = __shfl_xor_sync(0xffffffffu, bj, m);
            if (ov < bv || (ov == bv && oj < bj)) { bv = ov; bj = oj; }
        }
        if (lane == 0) {
            if (bv < INFINITY)
                atomicMin(best + e, ((unsigned long long)__float_as_uint(bv) << 32) | (uint32_t)bj);
            __threadfence();
            if (atomicAdd(done + e, 1) == (int)gridDim.x - 1)
                codes[list[e]] = (int32_t)(uint32_t)(atomicOr(best + e, 0ull) & 0xffffffffull);
        }
    }
}

// The slice [j0, j0 + S) of head h's cp is staged transposed, cT[a][c] with a
// padded stride S + 1 (few bank conflicts when it is written along a, none
// when lanes read along c).  Each warp takes a few rows of the chunk at a
// time, their z staged transposed (zT[a][r]: one vector load gives two rows'
// element a to every lane), and lane l owns centroids l, l + 32, ... of the
// slice, in pairs whose differences and squares run as packed two-float
// instructions (each rounded as the scalar one); every centroid value read
// from shared memory serves all of the warp's rows.  The row's code is
// written by the slice block that adds the last of the gridDim.x partial
// minima (a counter per row).
template <int S>
__global__ void __launch_bounds__(kExactThreads)
exact_scan_kernel(int32_t d, const float* __restrict__ cp, int64_t K,
                  const int32_t* __restrict__ head_count, const int32_t* __restrict__ head_rows,
                  int64_t head_cap, const float* __restrict__ zbuf,
                  unsigned long long* __restrict__ best, int32_t* __restrict__ done,
                  const int64_t* __restrict__ list, int32_t* __restrict__ codes) {
    static_assert(S % 64 == 0, "centroids come in pairs of lanes' columns");
    constexpr int kWarps = kExactThreads / 32;
    constexpr int RT = ScanTile<S>::kRT;
    extern __shared__ float cT[];  // [d][S + 1], then [warps][d][RT] for the rows' z
    const int h = blockIdx.y;
    const int64_t j0 = (int64_t)blockIdx.x * S;
    const int n = head_count[h];
    // chunks of two rows per warp when they fit the chunk groups once
    const bool narrow = n <= 2 * kWarps * (int)gridDim.z;
    const int kChunk = kWarps * (narrow ? 2 : RT);
    const int nchunks = (n + kChunk - 1) / kChunk;
    if ((int)blockIdx.z >= nchunks || j0 >= K) return;
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int nc = (int)(K - j0 < S ? K - j0 : S);
    // 16-byte loads, eight in flight per thread before their stores
    const float4* src4 = reinterpret_cast<const float4*>(cp + ((int64_t)h * K + j0) * d);
    const int d4 = d / 4, n4 = S * d4;
    for (int i0 = threadIdx.x; i0 < n4; i0 += 8 * kExactThreads) {
        float4 v[8];
#pragma unroll
        for (int u = 0; u < 8; u++) {
            const int i = i0 + u * kExactThreads;
            const int c = i / d4;
            v[u] = (i < n4 && c < nc) ? __ldg(src4 + i) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int u = 0; u < 8; u++) {
            const int i = i0 + u * kExactThreads;
            if (i < n4) {
                const int c = i / d4, a = (i - c * d4) * 4;
                float* dst = cT + a * (S + 1) + c;
                dst[0] = v[u].x;
                dst[S + 1] = v[u].y;
                dst[2 * (S + 1)] = v[u].z;
                dst[3 * (S + 1)] = v[u].w;
            }
        }
    }
    __syncthreads();
    const int32_t* rows = head_rows + (int64_t)h * head_cap;
    float* zT = cT + d * (S + 1) + w * d * RT;  // this warp's rows, [a][r]
    for (int chunk = blockIdx.z; chunk < nchunks; chunk += gridDim.z) {
        const int rt = narrow ? 2 : RT;
        const int r0 = chunk * kChunk + w * rt;
        const int nr = min(rt, n - r0);  // the warp's rows in this chunk
        if (nr <= 0) continue;
        if (narrow)
            scan_rows<S, 2>(cT, zT, d, nc, j0, rows, r0, nr, zbuf, best, done, list, codes, lane);
        else
            scan_rows<S, RT>(cT, zT, d, nc, j0, rows, r0, nr, zbuf, best, done, list, codes, lane);
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

unsigned blocks_for(int64_t n, int per, unsigned cap) {
    const int64_t b = (n + per - 1) / per;
    return (unsigned)(b < 1 ? 1 : (b > cap ? cap : b));
}

template <bool BF16, int DK, int PA, int AST, int BST, int RB>
cudaError_t launch_kernel(const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& tk,
                          const Params& p, cudaStream_t st) {
    using S = Smem<BF16, DK, PA, AST, BST, RB>;
    static_assert(S::kTotal <= 232448, "shared memory budget");
    auto k = assign_tc_kernel<BF16, DK, PA, AST, BST, RB>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, S::kTotal);
    if (e != cudaSuccess) return e;
    const int tiles = p.num_bh * p.tiles_per_bh;
    const int grid = tiles < sm_count() ? tiles : sm_count();
    k<<<grid, kThreads, S::kTotal, st>>>(ta, tb, tk, p);
    note_launches(1);
    return cudaGetLastError();
}

// Row blocks per tile: two (256 rows sharing every codebook stage, N = 128
// accumulators) for the one-plane pass at d <= 128, where two A stages of
// both blocks fit in shared memory, while the codebook has few chunks; with
// many chunks (K above 2048) one block and N = 256 accumulators, which issue
// half as many MMAs per centroid, do better (measured on GB300: 0.090 against
// 0.094 ms at K = 1024, 3.84 against 4.02 ms at K = 4096).
int row_blocks(int PA, int64_t d, int64_t K) { return PA == 1 && d <= 128 && K <= 2048 ? 2 : 1; }

template <bool BF16, int PA>
cudaError_t launch_by_width(const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& tk,
                            const Params& p, int rb, cudaStream_t st) {
    if constexpr (PA == 1) {
        switch (p.d) {
            case 64:
                return rb == 2 ? launch_kernel<BF16, 1, PA, 2, 6, 2>(ta, tb, tk, p, st)
                               : launch_kernel<BF16, 1, PA, 2, 4, 1>(ta, tb, tk, p, st);
            case 128:  // stages of both k-blocks
                return rb == 2 ? launch_kernel<BF16, 2, PA, 2, 2, 2>(ta, tb, tk, p, st)
                               : launch_kernel<BF16, 2, PA, 2, 2, 1>(ta, tb, tk, p, st);
            case 192: return launch_kernel<BF16, 3, PA, 1, 4, 1>(ta, tb, tk, p, st);
            // bf16 stages carry room for the -h tile: one stage fewer
            default: return launch_kernel<BF16, 4, PA, 1, BF16 ? 3 : 4, 1>(ta, tb, tk, p, st);
        }
    }
    else {
        switch (p.d) {
            case 64: return launch_kernel<BF16, 1, PA, 2, BF16 ? 3 : 4, 1>(ta, tb, tk, p, st);
            case 128: return launch_kernel<BF16, 2, PA, 1, 2, 1>(ta, tb, tk, p, st);
            case 192: return launch_kernel<BF16, 3, PA, 1, BF16 ? 2 : 3, 1>(ta, tb, tk, p, st);
            default: return launch_kernel<BF16, 4, PA, 1, 2, 1>(ta, tb, tk, p, st);
        }
    }
}

bool encode(CUtensorMap* m, bool bf16, int rank, const void* base, const cuuint64_t* dims,
            const cuuint64_t* strides, const cuuint32_t* box) {
    const cuuint32_t es[3] = {1, 1, 1};
    return encode_fn()(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                       (cuuint32_t)rank, const_cast<void*>(base), dims, strides, box, es,
                       CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                       CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                       CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// One codebook operand: the planes (or the raw codebook) and its head table.
struct BSide {
    const void* src;
    int P;
    bool exact;           // products exact without planes (raw 16-bit codebook)
    const float* head;
    const float2* gstat;  // [H, ngroups] group maxima of |chat_j| and h_j
};

// The codebook operand (variant v: 0 as is, 1 rotated by -far_offset) and,
// when launch is set, the launches that build it: per-head statistics, the
// head table and the 16-bit planes.  Without launch only the description is
// filled in, for a call that reuses an earlier call's preparation.
cudaError_t prepare_b(const TcCall& c, const float* chat, int v, bool raw, BSide& out,
                      cudaStream_t st, bool launch = true) {
    const bool bf16 = c.dt == kBF16;
    const int64_t H = c.s.H, K = c.K, d = c.s.d;
    const int64_t ngroups = (K + kPadCols - 1) / kPadCols * kPadCols / kTcGroup;
    out.gstat = c.gstat + v * H * ngroups;
    if (launch) {
        codebook_stats_kernel<<<dim3((unsigned)((K + 7) / 8), (unsigned)H), 256, 0, st>>>(
            chat, K, (int32_t)d, c.half_norm, c.head_bits + v * H * 4,
            reinterpret_cast<uint32_t*>(c.gstat + v * H * ngroups), (int32_t)ngroups);
        note_launches(1);
        head_finish_kernel<<<(unsigned)((H + 63) / 64), 64, 0, st>>>(
            c.head_bits + v * H * 4, (int32_t)H, (int32_t)d, (bf16 || raw) ? 1 : 0,
            c.head + v * H * 4, c.scale + v * H);
        note_launches(1);
    }
    out.head = c.head + v * H * 4;
    out.exact = raw;
    if (raw) {
        out.src = c.codebook;
        out.P = 1;
    } else {
        out.P = bf16 ? 3 : 2;
        uint16_t* planes = c.planes + (size_t)v * H * 3 * K * d;
        out.src = planes;
        if (!launch) return cudaSuccess;
        if (bf16)
            codebook_planes_kernel<true><<<blocks_for(H * K * d, 256, 8192), 256, 0, st>>>(
                chat, K, (int32_t)d, out.P, (int32_t)H, c.scale + v * H, planes);
        else
            codebook_planes_kernel<false><<<blocks_for(H * K * d, 256, 8192), 256, 0, st>>>(
                chat, K, (int32_t)d, out.P, (int32_t)H, c.scale + v * H, planes);
        note_launches(1);
    }
    return cudaGetLastError();
}

// max_rows: a bound on the rows of any (b, h) in this pass (the tiles past it
// are not visited).
cudaError_t run_pass(const TcCall& c, const BSide& b, int PA, const void* asrc, int64_t plane_rows,
                     const int32_t* count, const int32_t* row_map, const uint8_t* skip,
                     int32_t skip_near, int64_t max_rows, cudaStream_t st,
                     bool with_scores = false) {
    const bool bf16 = c.dt == kBF16;
    const int64_t H = c.s.H, K = c.K, d = c.s.d, nbh = c.s.B * c.s.H, ncap = c.s.Ncap;
    const int rb = row_blocks(PA, d, K);
    const int64_t bn = rb == 2 ? 128 : 256, tile_rows = BM * rb;
    CUtensorMap ta, tb;
    {
        const cuuint64_t dims[2] = {(cuuint64_t)d, (cuuint64_t)(PA * nbh * ncap)};
        const cuuint64_t strides[1] = {(cuuint64_t)(d * 2)};
        const cuuint32_t box[2] = {BK, BM};
        if (!encode(&ta, bf16, 2, asrc, dims, strides, box)) return cudaErrorInvalidValue;
    }
    {
        const cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)K, (cuuint64_t)(H * b.P)};
        const cuuint64_t strides[2] = {(cuuint64_t)(d * 2), (cuuint64_t)(K * d * 2)};
        const cuuint32_t box[3] = {BK, (cuuint32_t)bn, 1};
        if (!encode(&tb, bf16, 3, b.src, dims, strides, box)) return cudaErrorInvalidValue;
    }
    Params p;
    p.H = (int32_t)H;
    p.d = (int32_t)d;
    p.K = (int32_t)K;
    // two row planes: the first against every plane of chat, the second
    // against chat's first plane only
    p.P = b.P;
    p.pstride = b.P;
    p.num_bh = (int32_t)nbh;
    p.seg = (int32_t)ncap;
    p.tiles_per_bh = (int32_t)(((max_rows < ncap ? max_rows : ncap) + tile_rows - 1) / tile_rows);
    p.nchunks = (int32_t)((K + bn - 1) / bn);
    p.kpad = (int32_t)((K + kPadCols - 1) / kPadCols * kPadCols);  // row stride of hneg
    p.out_ncap = (int32_t)ncap;
    p.plane_rows = plane_rows;
    p.len = c.len;
    p.count = count;
    p.row_map = row_map;
    p.tile_rot = PA == 2 && row_map ? c.tile_rot : nullptr;
    p.tiles128 = (int32_t)((ncap + 127) / 128);
    p.skip = skip;
    p.skip_near = skip_near;
    p.hneg = c.hneg;
    p.hplanes = c.hplanes;
    p.head = b.head;
    p.gstat = b.gstat;
    p.ngroups = p.kpad / kTcGroup;
    // The products are exact; the tensor core adds (d/16 per operand pair)
    // partial sums into fp32, each addition off by at most 2^-23 of the
    // running magnitude, which |x| max|chat| + max h bounds; plus the rounding
    // of chat and of the planes that are dropped, of the two-plane row
    // operand, and of h and of acc - h.  A k-step whose products are all
    // zero (the second plane of a row stored unrotated) adds nothing.
    const int pairs = p.P + (PA == 2 ? 1 : 0);
    // bf16: one more k-step, the one that starts the accumulator at -h_j
    const double fixed = bf16 ? 9.0 : 8.0;
    double coef = ((double)pairs * (double)(d / 16) + fixed) * 0x1p-22;
    double coef_unrot = ((double)p.P * (double)(d / 16) + fixed) * 0x1p-22;
    if (!b.exact) {
        coef += bf16 ? 0x1p-21 : 0x1p-20;
        coef_unrot += bf16 ? 0x1p-21 : 0x1p-20;
    }
    if (PA == 2) coef += bf16 ? 0x1p-15 : 0x1p-20;
    // the dropped products, elementwise within a relative 2^-16 (bf16; 2^-22
    // fp16) of |x| |chat|: the row's second plane (|lo| <= 2^-8 |x|) against
    // chat's second (|c1| <= 2^-8 |chat|) and, for bf16, third plane
    if (PA == 2 && !b.exact) coef += bf16 ? 0x1.1p-16 : 0x1p-20;
    p.err_coef = (float)coef;
    p.err_coef_unrot = (float)coef_unrot;
    p.norm_slack = PA == 2 ? 1.01f : 1.0001f;
    p.codes = c.codes;
    p.exact_list = c.exact_list;
    p.exact_count = c.exact_count;
    p.status = c.exact_count + 1;
    p.max_rows = count ? c.exact_count + 2 : nullptr;
    // scores and the row copy: the stored keys in natural order only
    const bool sc = with_scores && PA == 1 && !count && !row_map && c.scores;
    p.sq = sc ? c.score_q : nullptr;
    p.sqn = sc ? c.score_qn : nullptr;
    p.scores = sc ? c.scores : nullptr;
    p.kcopy = sc ? c.kcopy : nullptr;
    // the copy's tensor map: [nbh][ncap][d] with the A tile's box and
    // swizzle, so the staged tile is stored as it landed (a 3-d map keeps
    // every box inside its (b, h))
    CUtensorMap tk = ta;
    p.kcopy_tma = 0;
    if (p.kcopy) {
        const cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)ncap, (cuuint64_t)nbh};
        const cuuint64_t strides[2] = {(cuuint64_t)(d * 2), (cuuint64_t)(ncap * d * 2)};
        const cuuint32_t box[3] = {BK, BM, 1};
        if (encode(&tk, bf16, 3, p.kcopy, dims, strides, box)) p.kcopy_tma = 1;
        else tk = ta;
    }
    if (p.num_bh * p.tiles_per_bh == 0) return cudaSuccess;
    if (PA == 1)
        return bf16 ? launch_by_width<true, 1>(ta, tb, tk, p, rb, st)
                    : launch_by_width<false, 1>(ta, tb, tk, p, rb, st);
    return bf16 ? launch_by_width<true, 2>(ta, tb, tk, p, rb, st)
                : launch_by_width<false, 2>(ta, tb, tk, p, rb, st);
}

}  // namespace tc

bool tc_supported(int dt, int64_t d) {
    return (dt == kBF16 || dt == kF16) && d % 64 == 0 && d >= 64 && d <= 256 &&
           tc::encode_fn() != nullptr;
}

cudaError_t launch_assign_tc(const TcCall& c, cudaStream_t st) {
    using namespace tc;
    const int64_t H = c.s.H, K = c.K, d = c.s.d, nbh = c.s.B * c.s.H, ncap = c.s.Ncap;
    const int64_t kpad = (K + kPadCols - 1) / kPadCols * kPadCols;
    const bool rot = c.ra.enabled && c.ra.far_offset != 0;
    const bool natural = c.sel.mode == 0 || c.sel.mode == 2;
    const bool compact = !natural || (c.ra.enabled && c.ra.window > 0);
    const bool need_u = compact || (natural && !rot);
    const bool need_r = natural && rot;
    cudaError_t e;

    // count, status, longest list, (unused), then the per-head list lengths
    // and the compact tiles' flags (they follow exact_count in the workspace)
    e = cudaMemsetAsync(c.exact_count, 0, sizeof(int32_t) * (4 + H + nbh * ((ncap + 127) / 128)),
                        st);
    if (e != cudaSuccess) return e;
    // the codebook side, unless an earlier call left it in this workspace:
    // chat = c L L^T (c itself when L is the identity), -|c L|^2 / 2 padded,
    // and the operand planes
    const bool build = !c.prepared;
    if (build) {
        e = cudaMemsetAsync(c.head_bits, 0, sizeof(uint32_t) * 2 * 4 * H, st);
        if (e != cudaSuccess) return e;
        e = cudaMemsetAsync(c.gstat, 0, sizeof(float2) * 2 * H * (kpad / kTcGroup), st);
        if (e != cudaSuccess) return e;
        if (c.dt == kBF16)
            hneg_planes_kernel<<<blocks_for(H * kpad, 256, 4096), 256, 0, st>>>(c.half_norm, H, K,
                                                                              kpad, c.hplanes);
        else
            pad_half_norm_kernel<<<blocks_for(H * kpad, 256, 4096), 256, 0, st>>>(
                c.half_norm, H, K, kpad, c.hneg);
        note_launches(1);
    }
    const float* chat = c.L ? c.chat : c.cp;
    BSide bu{}, br{};
    if (need_u && (e = prepare_b(c, chat, 0, c.L == nullptr, bu, st, build)) != cudaSuccess)
        return e;
    if (need_r) {
        if (build) {
            rotate_rows_kernel<<<blocks_for(H * K * (d / 2), 256, 8192), 256, 0, st>>>(
                chat, H * K, (int32_t)d, c.ra, c.chat_rot);
            note_launches(1);
        }
        if ((e = prepare_b(c, c.chat_rot, 1, false, br, st, build)) != cudaSuccess) return e;
    }
    const uint8_t* skip = nullptr;
    if (c.sel.mode == 2) {
        e = cudaMemsetAsync(c.skip, 0, (size_t)(nbh * ncap), st);
        if (e != cudaSuccess) return e;
        dim3 g(blocks_for(ncap, 256, 64), (unsigned)nbh);
        mark_rows_kernel<<<g, 256, 0, st>>>((int32_t)H, (int32_t)ncap, c.len, c.sel.perm,
                                            c.sel.count, c.skip);
        note_launches(1);
        skip = c.skip;
    }
    // far rows in stored order: the keys themselves are the row operand
    if (natural) {
        const int32_t skip_near = (c.ra.enabled && c.ra.window > 0) ? c.ra.window : 0;
        timing_begin(st);
        e = run_pass(c, rot ? br : bu, 1, c.x, 0, nullptr, nullptr, skip, skip_near, ncap, st,
                     !rot && !skip);
        timing_end(st);
        if (e != cudaSuccess) return e;
    }
    if (c.after_natural && (e = c.after_natural(c.after_ctx, st)) != cudaSuccess) return e;
    // rotated rows (the RoPE window, or every routed row) as two 16-bit planes
    if (compact) {
        // rows per (b, h): at most the window (natural order), one (decode),
        // or the retrieval count (not known here; grid-stride)
        const int cmode = c.sel.mode == 2 ? 0 : c.sel.mode;
        const int64_t most = cmode == 0 ? (c.ra.window < ncap ? c.ra.window : ncap)
                                        : (cmode == 3 ? 1 : ncap);
        // one wave of blocks (eight per SM) over all (b, h); each block
        // sweeps kCompactRows rows at a time
        const int64_t per_bh = 8 * (int64_t)sm_count() / (nbh > 0 ? nbh : 1);
        dim3 g(blocks_for(most, kCompactRows, (unsigned)(per_bh > 1 ? per_bh : 1)), (unsigned)nbh);
        if (c.dt == kBF16)
            compact_rows_kernel<kBF16><<<g, 256, 0, st>>>(
                c.x, (int32_t)H, (int32_t)ncap, (int32_t)d, c.len, c.ra, c.sel.mode == 2 ? 0 : c.sel.mode,
                c.sel.perm, c.sel.count, c.compact, c.row_map, c.ccount, c.exact_list,
                c.exact_count, c.tile_rot);
        else
            compact_rows_kernel<kF16><<<g, 256, 0, st>>>(
                c.x, (int32_t)H, (int32_t)ncap, (int32_t)d, c.len, c.ra, c.sel.mode == 2 ? 0 : c.sel.mode,
                c.sel.perm, c.sel.count, c.compact, c.row_map, c.ccount, c.exact_list,
                c.exact_count, c.tile_rot);
        note_launches(1);
        e = run_pass(c, bu, 2, c.compact, nbh * ncap, c.ccount, c.row_map, skip, 0, most, st);
        if (e != cudaSuccess) return e;
    }
    // rows the contraction could not decide
    const unsigned sms = (unsigned)sm_count();
    float* zbuf = reinterpret_cast<float*>(c.compact);   // the planes are no longer read
    int32_t* head_rows = c.row_map;                      // nor the compact row map
    const int64_t head_cap = c.s.B * ncap;
    if (c.dt == kBF16)
        exact_rows_kernel<kBF16><<<sms * 4, kExactThreads, 0, st>>>(
            c.x, (int32_t)H, (int32_t)ncap, (int32_t)d, c.len, c.ra, c.L, c.exact_list,
            c.exact_count, zbuf, c.exact_best, c.exact_done, c.head_count, head_rows, head_cap);
    else
        exact_rows_kernel<kF16><<<sms * 4, kExactThreads, 0, st>>>(
            c.x, (int32_t)H, (int32_t)ncap, (int32_t)d, c.len, c.ra, c.L, c.exact_list,
            c.exact_count, zbuf, c.exact_best, c.exact_done, c.head_count, head_rows, head_cap);
    {
        // slices of 128 centroids (64 at d > 128) keep the staged slice near
        // 66 KB; with few centroids (K <= 2048) slices of 64, whose blocks
        // stage half as much each and spread the short lists over twice as
        // many blocks (0.1504 against 0.1521 ms per step at K = 1024; at
        // K = 4096, with long lists, 128 is faster: 4.20 against 4.25 ms)
        const int S = (d > 128 || K <= 2048) ? 64 : 128;
        const int RT = S == 128 ? ScanTile<128>::kRT : ScanTile<64>::kRT;
        const size_t smem = sizeof(float) * (size_t)d * (S + 1 + RT * (kExactThreads / 32));
        auto scan = S == 128 ? exact_scan_kernel<128> : exact_scan_kernel<64>;
        e = cudaFuncSetAttribute(scan, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        // chunks of a head's rows run side by side in z: up to 8, about 2048
        // blocks in all (the blocks past a head's last chunk leave at once,
        // and a block takes the chunks z, z + zc, ... of its head, staging
        // its slice once)
        const int64_t slices = (K + S - 1) / S;
        int64_t zc = 2048 / (slices * H);
        zc = zc < 1 ? 1 : (zc > 8 ? 8 : zc);
        dim3 g((unsigned)slices, (unsigned)H, (unsigned)zc);
        scan<<<g, kExactThreads, smem, st>>>((int32_t)d, c.cp, K, c.head_count, head_rows, head_cap,
                                             zbuf, c.exact_best, c.exact_done, c.exact_list,
                                             c.codes);
    }
    note_launches(2);
    return cudaGetLastError();
}

}  // namespace a2ats
