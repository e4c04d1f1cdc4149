// aux_kernels.cu -- the centroid-norm kernel and the key-finalize kernel.
//
// Norms (flashlib PR #22 "Optimize Blackwell k-means assignment reduction",
// Summary: the centroid norms applied to every score tile):
//   cnorm[j] = sum_d c_jd^2, fp32, one warp per centroid row.  Each lane
//   reads 16 contiguous bytes (8 bf16) of the row, so a warp reads a 512-byte
//   row in one coalesced sweep; D <= 256 means one load per lane.  Each lane
//   sums its 8 exact squares in order, then a fixed xor-shuffle tree adds the
//   lanes, so the result is deterministic.  The kernel is bound by HBM
//   bandwidth (2*D bytes read, 4 written per centroid).
//
// Finalize: turns the packed (ordered score << 32 | index) keys left by the
// split-centroid path into idx and minscore.  A key still at its initial
// all-ones value means no number was seen for that point (every score NaN):
// idx 0, minscore NaN.
#include "internal.h"

#include <cuda_bf16.h>

#include <algorithm>

namespace kma {
namespace {

constexpr int kNormWarps = 8;

__global__ void __launch_bounds__(32 * kNormWarps)
    norms_kernel(const uint4 *__restrict__ C, int64_t K, int32_t D, float *__restrict__ cnorm)
{
    const int lane = threadIdx.x & 31;
    const int64_t j = static_cast<int64_t>(blockIdx.x) * kNormWarps + (threadIdx.x >> 5);
    if (j >= K)
        return;
    const int vec_per_row = D >> 3;   // 16-byte vectors per row (D % 16 == 0)
    float acc = 0.0f;
    if (lane < vec_per_row) {
        const uint4 q = __ldg(C + j * vec_per_row + lane);
        const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float lo = __uint_as_float(w[i] << 16);
            const float hi = __uint_as_float(w[i] & 0xffff0000u);
            acc = fmaf(lo, lo, acc);
            acc = fmaf(hi, hi, acc);
        }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
        acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (lane == 0)
        cnorm[j] = acc;
}

__global__ void finalize_kernel(const unsigned long long *__restrict__ keys, int64_t N,
                                int32_t *__restrict__ idx, float *__restrict__ minscore)
{
    const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (i >= N)
        return;
    const unsigned long long key = keys[i];
    int32_t ix;
    float ms;
    if (key == ~0ull) {
        ix = 0;
        ms = __int_as_float(0x7fc00000);
    } else {
        ix = static_cast<int32_t>(key & 0xffffffffull);
        const uint32_t o = static_cast<uint32_t>(key >> 32);
        const uint32_t u = (o & 0x80000000u) ? (o & 0x7fffffffu) : ~o;
        ms = __uint_as_float(u);
    }
    idx[i] = ix;
    if (minscore != nullptr)
        minscore[i] = ms;
}

// The update step of a Lloyd iteration, which follows the assignment (not
// part of flashlib PR #22, which covers the assignment; the textbook update):
// counts[j] += |{i : idx[i] == j}|, sums[j][d] += sum of x_id over them, fp32.
// A group of D/8 lanes takes one point: each lane widens 8 bf16 values and
// adds them with two 16-byte vector reductions into L2.  The order in which
// points reach a centroid is not fixed, so fp32 sums of non-integer data can
// differ in their last bits between runs; integer-valued data whose sums stay
// below 2^24 is exact.  Ids outside [0, K) are skipped.
__global__ void __launch_bounds__(256)
    update_kernel(const uint4 *__restrict__ X, const int32_t *__restrict__ idx, int64_t N,
                  int32_t K, int32_t D, float *__restrict__ sums, int32_t *__restrict__ counts)
{
    const int lane = threadIdx.x & 31;
    const int vec = D >> 3;                 // 16-byte vectors per row
    const int per_warp = 32 / vec;          // points per warp per step; spare lanes idle
    const int slot = lane / vec;
    const int part = lane - slot * vec;
    const int64_t warp = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
    for (int64_t i0 = warp * per_warp; i0 < N; i0 += nwarps * per_warp) {
        const int64_t i = i0 + slot;
        if (slot >= per_warp || i >= N)
            continue;
        const int32_t j = __ldg(idx + i);
        if (j < 0 || j >= K)
            continue;
        if (part == 0)
            atomicAdd(counts + j, 1);
        const uint4 q = __ldg(X + i * vec + part);
        const uint32_t w[4] = {q.x, q.y, q.z, q.w};
        float f[8];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            f[2 * e] = __uint_as_float(w[e] << 16);
            f[2 * e + 1] = __uint_as_float(w[e] & 0xffff0000u);
        }
        float *dst = sums + static_cast<int64_t>(j) * D + part * 8;
        asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(dst), "f"(f[0]),
                     "f"(f[1]), "f"(f[2]), "f"(f[3])
                     : "memory");
        asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(dst + 4), "f"(f[4]),
                     "f"(f[5]), "f"(f[6]), "f"(f[7])
                     : "memory");
    }
}

// New centroids from the sums: mean (fp32, correctly rounded division) where
// a centroid has points, written as bf16 (round to nearest even) and, when
// asked, as fp32; a centroid without points keeps its old value.  One thread
// per 8 dimensions.  C_new may alias C_old.
__global__ void centroids_kernel(const float *__restrict__ sums, const int32_t *__restrict__ counts,
                                 const uint4 *C_old, int64_t K, int32_t D, uint4 *C_new,
                                 float *__restrict__ means)
{
    const int vec = D >> 3;
    const int64_t t = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (t >= K * vec)
        return;
    const int64_t j = t / vec;
    const int part = static_cast<int>(t - j * vec);
    const int32_t n = counts[j];
    if (n <= 0) {
        const uint4 q = C_old[t];
        if (C_new != C_old)
            C_new[t] = q;
        if (means != nullptr) {
            const uint32_t w[4] = {q.x, q.y, q.z, q.w};
            float *m = means + j * D + part * 8;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                m[2 * e] = __uint_as_float(w[e] << 16);
                m[2 * e + 1] = __uint_as_float(w[e] & 0xffff0000u);
            }
        }
        return;
    }
    const float count = static_cast<float>(n);
    const float *s = sums + j * D + part * 8;
    float m[8];
#pragma unroll
    for (int e = 0; e < 8; ++e)
        m[e] = __fdiv_rn(s[e], count);
    uint32_t w[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const uint32_t lo = __bfloat16_as_ushort(__float2bfloat16_rn(m[2 * e]));
        const uint32_t hi = __bfloat16_as_ushort(__float2bfloat16_rn(m[2 * e + 1]));
        w[e] = lo | (hi << 16);
    }
    C_new[t] = make_uint4(w[0], w[1], w[2], w[3]);
    if (means != nullptr) {
        float *mo = means + j * D + part * 8;
#pragma unroll
        for (int e = 0; e < 8; ++e)
            mo[e] = m[e];
    }
}

// Squared distances from the assignment's scores: d = ||x||^2 + s in fp32,
// a negative (rounding) result written as 0, NaN kept.
__global__ void add_norms_kernel(float *__restrict__ score, const float *__restrict__ xnorm,
                                 int64_t N)
{
    const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (i >= N)
        return;
    const float d = xnorm[i] + score[i];
    score[i] = d < 0.0f ? 0.0f : d;
}

}  // namespace

cudaError_t launch_add_norms(float *score, const float *xnorm, int64_t N, cudaStream_t stream)
{
    const int threads = 256;
    const int64_t blocks = (N + threads - 1) / threads;
    add_norms_kernel<<<static_cast<unsigned>(blocks), threads, 0, stream>>>(score, xnorm, N);
    return cudaGetLastError();
}

cudaError_t launch_update(const void *X, const int32_t *idx, int64_t N, int64_t K, int64_t D,
                          float *sums, int32_t *counts, int sms, cudaStream_t stream)
{
    const int threads = 256;
    const int64_t per_block = (threads / 32) * (32 / (D / 8));
    const int64_t want = (N + per_block - 1) / per_block;
    const int64_t blocks = std::max<int64_t>(1, std::min<int64_t>(want, int64_t(sms) * 16));
    update_kernel<<<static_cast<unsigned>(blocks), threads, 0, stream>>>(
        static_cast<const uint4 *>(X), idx, N, static_cast<int32_t>(K), static_cast<int32_t>(D),
        sums, counts);
    return cudaGetLastError();
}

cudaError_t launch_centroids(const float *sums, const int32_t *counts, const void *C_old, int64_t K,
                             int64_t D, void *C_new, float *means, cudaStream_t stream)
{
    const int threads = 256;
    const int64_t total = K * (D / 8);
    const int64_t blocks = (total + threads - 1) / threads;
    centroids_kernel<<<static_cast<unsigned>(blocks), threads, 0, stream>>>(
        sums, counts, static_cast<const uint4 *>(C_old), K, static_cast<int32_t>(D),
        static_cast<uint4 *>(C_new), means);
    return cudaGetLastError();
}

cudaError_t launch_norms(const void *C, int64_t K, int64_t D, float *cnorm, cudaStream_t stream)
{
    const int64_t blocks = (K + kNormWarps - 1) / kNormWarps;
    norms_kernel<<<static_cast<unsigned>(blocks), 32 * kNormWarps, 0, stream>>>(
        static_cast<const uint4 *>(C), K, static_cast<int32_t>(D), cnorm);
    return cudaGetLastError();
}

cudaError_t launch_finalize(const unsigned long long *keys, int64_t N, int32_t *idx,
                            float *minscore, cudaStream_t stream)
{
    const int threads = 256;
    const int64_t blocks = (N + threads - 1) / threads;
    finalize_kernel<<<static_cast<unsigned>(blocks), threads, 0, stream>>>(keys, N, idx, minscore);
    return cudaGetLastError();
}

}  // namespace kma
