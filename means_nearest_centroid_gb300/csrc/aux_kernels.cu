// aux_kernels.cu -- the centroid-norm kernel, the key-finalize kernel, the
// new-centroid kernel of the update step and the distance fix-up.
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
