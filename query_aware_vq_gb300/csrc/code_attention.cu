// code_attention.cu -- code-based attention scores and the top tokens.
//
// Deploy-preview "A2ATS-adapted" page, paper-fidelity section, "Windowed
// RoPE (Eq. 11-12)": far keys stay in the unrotated frame and the constant
// far relative position b rides on the query (u_ij = q_i R_b k_j^T); keys
// inside the window keep exact RoPE.  The paper's abstract: the attention
// score is approximated through the vector-quantised keys so that the top-K
// tokens are retrieved.  With q the decode query before RoPE and t = len - 1:
//   near row j (0 <= t - j < window):  u_j = RoPE(q, t) . RoPE(k_j, j)
//   far row j:                         u_j = RoPE(q, b) . c_{code_j}
// (0 for a code outside [0, K)); the top ceil(fraction len) rows by
// (u desc, index asc) are then split off as the retrieval split orders its
// set.
//
// The far rows, nearly all of the cache, cost one 4-byte code read, one
// lookup in a per-(b, h) table of K entries (q R_b . c_k) and one 4-byte
// score write each: the pass is bound by HBM bandwidth at 8 bytes per key.
#include "kernels.cuh"

namespace a2ats {
namespace {

constexpr int kTableThreads = 256;  // 32 centroids x 8 lanes
constexpr int kRowThreads = 256;

// Blocks (x, bh): each forms RoPE(q, t) and RoPE(q, b) of its (b, h) in
// shared memory (block x = 0 stores the first for the near rows), then fills
// its share of the table lut[bh][k] = RoPE(q, b) . c_k, 8 lanes per centroid.
template <int DT>
__global__ void __launch_bounds__(kTableThreads)
query_table_kernel(const void* __restrict__ query, const void* __restrict__ codebook, int32_t H,
                   int32_t ncap, int32_t d, int64_t K, const int32_t* __restrict__ len,
                   const RopeArgs ra, int32_t far_b, float* __restrict__ q_near,
                   float* __restrict__ lut) {
    __shared__ __align__(16) float qn[kMaxD];
    __shared__ __align__(16) float qf[kMaxD];
    const int bh = blockIdx.y;
    const int h = bh % H;
    const int32_t L = seq_len(len, bh / H, ncap);
    const int32_t t = L > 0 ? L - 1 : 0;
    const int tid = threadIdx.x;
    for (int a = tid; a < d; a += blockDim.x) {
        const float v = load1<DT>(query, (int64_t)bh * d + a);
        qn[a] = v;
        qf[a] = v;
    }
    __syncthreads();
    const int half = d / 2;
    for (int i = tid; i < half; i += blockDim.x) {
        const int a = ra.interleaved ? 2 * i : i;
        const int b = ra.interleaved ? 2 * i + 1 : i + half;
        float sn, cs;
        if (t != 0) {
            rope_angle(t, ra.omega_hi[i], ra.omega_lo[i], ra, sn, cs);
            const float xa = qn[a], xb = qn[b];
            qn[a] = fmaf(xa, cs, -__fmul_rn(xb, sn));
            qn[b] = fmaf(xa, sn, __fmul_rn(xb, cs));
        }
        if (far_b != 0) {
            rope_angle(far_b, ra.omega_hi[i], ra.omega_lo[i], ra, sn, cs);
            const float xa = qf[a], xb = qf[b];
            qf[a] = fmaf(xa, cs, -__fmul_rn(xb, sn));
            qf[b] = fmaf(xa, sn, __fmul_rn(xb, cs));
        }
    }
    __syncthreads();
    if (blockIdx.x == 0)
        for (int a = tid; a < d; a += blockDim.x) q_near[(int64_t)bh * d + a] = qn[a];
    const int grp = tid >> 3, seg = tid & 7;
    // uniform trip count: the shuffles below need every lane
    for (int64_t j0 = (int64_t)blockIdx.x * 32; j0 < K; j0 += (int64_t)gridDim.x * 32) {
        const int64_t j = j0 + grp;
        const bool ok = j < K;
        float acc = 0.f;
        if (ok) {
            const int64_t base = ((int64_t)h * K + j) * d;
            for (int a = seg; a < d; a += 8) acc = fmaf(qf[a], load1<DT>(codebook, base + a), acc);
        }
        for (int m = 4; m; m >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, m);
        if (ok && seg == 0) lut[(int64_t)bh * K + j] = acc;
    }
}

// Far rows: scores[row] = lut[bh][code]; one thread per row, grid-stride,
// with (bh, j) advanced by the stride without 64-bit divisions.  Rows past
// len and the near rows are left alone.
__global__ void __launch_bounds__(kRowThreads)
far_score_kernel(const int32_t* __restrict__ codes, int64_t rows, int32_t H, int32_t ncap,
                 int64_t K, const int32_t* __restrict__ len, int32_t window,
                 const float* __restrict__ lut, float* __restrict__ scores) {
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    const int64_t qs = stride / ncap;
    const int32_t rs = (int32_t)(stride - qs * ncap);
    int64_t row = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    int64_t bh = row / ncap;
    int32_t j = (int32_t)(row - bh * ncap);
    for (; row < rows; row += stride) {
        const int32_t L = seq_len(len, (int32_t)(bh / H), ncap);
        const int32_t dist = L - 1 - j;
        if (j < L && !(window > 0 && dist < window)) {
            const int32_t c = codes[row];
            scores[row] = (c >= 0 && c < K) ? lut[bh * K + c] : 0.f;
        }
        j += rs;
        bh += qs;
        if (j >= ncap) {
            j -= ncap;
            bh++;
        }
    }
}

// Near rows j in [len - W, len) of each (b, h): one warp per row, the key
// rotated at its own position and dotted with RoPE(q, t).
template <int DT>
__global__ void __launch_bounds__(kRowThreads)
near_score_kernel(const void* __restrict__ keys, int64_t nbh, int32_t H, int32_t ncap, int32_t d,
                  int32_t win, const int32_t* __restrict__ len, const RopeArgs ra,
                  const float* __restrict__ q_near, float* __restrict__ scores) {
    __shared__ float buf[kRowThreads / 32][kMaxD];
    const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t rows = nbh * win;
    for (int64_t r = (int64_t)blockIdx.x * (kRowThreads / 32) + w; r < rows;
         r += (int64_t)gridDim.x * (kRowThreads / 32)) {
        const int64_t bh = r / win;
        const int32_t L = seq_len(len, (int32_t)(bh / H), ncap);
        const int32_t j = L - win + (int32_t)(r - bh * win);
        if (j < 0 || j >= L) continue;
        const int64_t row = bh * ncap + j;
        float* v = buf[w];
        for (int i = lane; i < d; i += 32) v[i] = load1<DT>(keys, row * d + i);
        __syncwarp();
        if (j != 0) {
            const int half = d / 2;
            for (int i = lane; i < half; i += 32) {
                const int a = ra.interleaved ? 2 * i : i;
                const int b = ra.interleaved ? 2 * i + 1 : i + half;
                float sn, cs;
                rope_angle(j, ra.omega_hi[i], ra.omega_lo[i], ra, sn, cs);
                const float xa = v[a], xb = v[b];
                v[a] = fmaf(xa, cs, -__fmul_rn(xb, sn));
                v[b] = fmaf(xa, sn, __fmul_rn(xb, cs));
            }
        }
        __syncwarp();
        float dot = 0.f;
        for (int i = lane; i < d; i += 32) dot = fmaf(v[i], q_near[bh * d + i], dot);
        for (int m = 16; m; m >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, m);
        if (lane == 0) scores[row] = dot;
        __syncwarp();
    }
}

// Dequantisation (v0.39.0 page, "How it works", step 3: a key is
// reconstructed from its assigned centroid): row j of out = codebook row
// codes[j] of its head, zeros for a code outside [0, K).  vec lanes per row,
// one 16-byte chunk each; grid-stride over rows with (bh, j) advanced by the
// stride without divisions; rows past len are left alone.
__global__ void __launch_bounds__(kRowThreads)
dequantize_kernel(const int32_t* __restrict__ codes, const uint4* __restrict__ cb,
                  uint4* __restrict__ out, int64_t rows, int32_t H, int32_t ncap, int32_t vec,
                  int64_t K, const int32_t* __restrict__ len) {
    const int rpb = kRowThreads / vec;
    const int lane = threadIdx.x % vec, rl = threadIdx.x / vec;
    if (rl >= rpb) return;  // vec need not divide the block
    const int64_t stride = (int64_t)gridDim.x * rpb;
    const int64_t qs = stride / ncap;
    const int32_t rs = (int32_t)(stride - qs * ncap);
    int64_t row = (int64_t)blockIdx.x * rpb + rl;
    int32_t bh = (int32_t)(row / ncap);  // B H <= 65535
    int32_t j = (int32_t)(row - (int64_t)bh * ncap);
    for (; row < rows; row += stride) {
        if (j < seq_len(len, bh / H, ncap)) {
            const int32_t c = codes[row];
            uint4 v = make_uint4(0u, 0u, 0u, 0u);
            if (c >= 0 && c < K) v = cb[((int64_t)(bh % H) * K + c) * vec + lane];
            out[row * vec + lane] = v;
        }
        j += rs;
        bh += (int32_t)qs;
        if (j >= ncap) {
            j -= ncap;
            bh++;
        }
    }
}

int device_sms() {
    int dev = 0, sms = 152;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    return sms;
}

}  // namespace

cudaError_t launch_code_attention(const void* keys, int dt, const Shape& s, const int32_t* len,
                                  const int32_t* codes, const void* codebook, int64_t K,
                                  const void* query, const RopeArgs& ra, int32_t far_b,
                                  float* q_near, float* lut, float* scores, cudaStream_t st) {
    const int64_t nbh = s.B * s.H;
    if (nbh == 0 || s.Ncap == 0) return cudaSuccess;
    const int d = (int)s.d;
    const int sms = device_sms();
    {
        int64_t per = (K + 31) / 32;
        const int64_t cap = (2 * (int64_t)sms + nbh - 1) / nbh;
        if (per > cap) per = cap;
        if (per < 1) per = 1;
        const dim3 g((unsigned)per, (unsigned)nbh);
        if (dt == kBF16)
            query_table_kernel<kBF16><<<g, kTableThreads, 0, st>>>(
                query, codebook, (int32_t)s.H, (int32_t)s.Ncap, d, K, len, ra, far_b, q_near, lut);
        else if (dt == kF16)
            query_table_kernel<kF16><<<g, kTableThreads, 0, st>>>(
                query, codebook, (int32_t)s.H, (int32_t)s.Ncap, d, K, len, ra, far_b, q_near, lut);
        else
            query_table_kernel<kF32><<<g, kTableThreads, 0, st>>>(
                query, codebook, (int32_t)s.H, (int32_t)s.Ncap, d, K, len, ra, far_b, q_near, lut);
        note_launches(1);
    }
    {
        const int64_t rows = nbh * s.Ncap;
        int64_t blocks = (rows + kRowThreads - 1) / kRowThreads;
        if (blocks > 8 * (int64_t)sms) blocks = 8 * (int64_t)sms;
        far_score_kernel<<<(unsigned)blocks, kRowThreads, 0, st>>>(
            codes, rows, (int32_t)s.H, (int32_t)s.Ncap, K, len, ra.window, lut, scores);
        note_launches(1);
    }
    const int64_t win = ra.window > 0 ? (ra.window < s.Ncap ? ra.window : s.Ncap) : 0;
    if (win > 0) {
        int64_t blocks = (nbh * win + kRowThreads / 32 - 1) / (kRowThreads / 32);
        if (blocks > 8 * (int64_t)sms) blocks = 8 * (int64_t)sms;
        if (dt == kBF16)
            near_score_kernel<kBF16><<<(unsigned)blocks, kRowThreads, 0, st>>>(
                keys, nbh, (int32_t)s.H, (int32_t)s.Ncap, d, (int32_t)win, len, ra, q_near, scores);
        else if (dt == kF16)
            near_score_kernel<kF16><<<(unsigned)blocks, kRowThreads, 0, st>>>(
                keys, nbh, (int32_t)s.H, (int32_t)s.Ncap, d, (int32_t)win, len, ra, q_near, scores);
        else
            near_score_kernel<kF32><<<(unsigned)blocks, kRowThreads, 0, st>>>(
                keys, nbh, (int32_t)s.H, (int32_t)s.Ncap, d, (int32_t)win, len, ra, q_near, scores);
        note_launches(1);
    }
    return cudaGetLastError();
}

cudaError_t launch_dequantize(const int32_t* codes, const void* codebook, int dt, const Shape& s,
                              int64_t K, const int32_t* len, void* out, cudaStream_t st) {
    const int64_t rows = s.B * s.H * s.Ncap;
    if (rows == 0) return cudaSuccess;
    const int32_t vec = (int32_t)(s.d * (dt == kF32 ? 4 : 2) / 16);
    const int64_t rpb = kRowThreads / vec;
    int64_t blocks = (rows + rpb - 1) / rpb;
    const int64_t cap = 16 * (int64_t)device_sms();
    if (blocks > cap) blocks = cap;
    dequantize_kernel<<<(unsigned)blocks, kRowThreads, 0, st>>>(
        codes, reinterpret_cast<const uint4*>(codebook), reinterpret_cast<uint4*>(out), rows,
        (int32_t)s.H, (int32_t)s.Ncap, vec, K, len);
    note_launches(1);
    return cudaGetLastError();
}

}  // namespace a2ats
