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

}  // namespace

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
