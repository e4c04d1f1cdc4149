// aux_kernels.cu -- the centroid-norm kernel, the preparation kernel of an
// assignment call, the new-centroid kernel of the update step and the
// distance fix-up.
//
// Norms (flashlib PR #22 "Optimize Blackwell k-means assignment reduction",
// Summary: the centroid norms applied to every score tile):
//   cnorm[j] = sum_d c_jd^2, fp32, one warp per centroid row (warp_row_norm:
//   a fixed summation order, so the result is deterministic).  Each lane
//   reads 16 contiguous bytes (8 bf16) of the row, so a warp reads a 512-byte
//   row in one coalesced sweep.  Bound by HBM bandwidth (2*D bytes read, 4
//   written per centroid).
//
// Preparation: everything an assignment call needs before its main kernel,
// in one launch -- the norms (when the caller gave none), the CTA pair's fold
// operand (when the plan folds the norms on CTA pairs), and the all-ones
// initial value of the packed keys and arrival counters of split rows.
#include "internal.h"
#include "norm_math.cuh"

#include <cuda_bf16.h>

#include <algorithm>

namespace kma {
namespace {

constexpr int kNormWarps = 8;

__global__ void __launch_bounds__(32 * kNormWarps)
    norms_kernel(const uint4 *__restrict__ C, int64_t K, int32_t D, float *__restrict__ cnorm)
{
    const int lane = threadIdx.x & 31;
    const int rpw = rows_per_warp(D);
    const int64_t row0 =
        (static_cast<int64_t>(blockIdx.x) * kNormWarps + (threadIdx.x >> 5)) * rpw;
    if (row0 >= K)
        return;   // uniform across the warp
    const float acc = warp_rows_norm(C, row0, K, D, lane);
    const int vpr = rpw == 1 ? 32 : D >> 3;
    const int64_t j = row0 + lane / vpr;
    if (lane % vpr == 0 && j < K)
        cnorm[j] = acc;
}

struct PrepArgs {
    const uint4 *C;          // centroids, or nullptr when the norms are given
    const float *cnorm_in;   // the caller's norms, or nullptr
    float *cnorm_out;        // norms computed here, or nullptr
    uint4 *fold;             // fold operand ([block][2][128] rows of 16 bytes), or nullptr
    uint4 *fill;             // 16-byte words set to all-ones, or nullptr
    int64_t K, rows, fill_words;
    int64_t row_blocks;      // blocks [0, row_blocks) work on centroid rows
    int32_t D;
    int32_t rpw;             // rows per warp: 32 with the caller's norms, else rows_per_warp(D)
};

// Rows: one warp per centroid row j < rows (rows covers K, and the fold
// operand's padding to whole blocks of 128 centroids per CTA, whose rows
// hold NaN so that they never win).  The fold operand of centroid j is row r
// = j % 128 of block b = j / 128: its first K half holds the three bf16 parts
// of -cnorm[j] / 2, its second half zeros.  Fill: the remaining blocks write
// all-ones words.
__global__ void __launch_bounds__(32 * kNormWarps) prep_kernel(const PrepArgs a)
{
    // The assignment kernel that follows may start its set-up now; its warps
    // that read these outputs wait for this kernel to complete.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if (blockIdx.x >= a.row_blocks) {
        const int64_t stride = (static_cast<int64_t>(gridDim.x) - a.row_blocks) * blockDim.x;
        for (int64_t t = (static_cast<int64_t>(blockIdx.x) - a.row_blocks) * blockDim.x +
                         threadIdx.x;
             t < a.fill_words; t += stride)
            a.fill[t] = make_uint4(~0u, ~0u, ~0u, ~0u);
        return;
    }
    const int lane = threadIdx.x & 31;
    const int64_t row0 =
        (static_cast<int64_t>(blockIdx.x) * kNormWarps + (threadIdx.x >> 5)) * a.rpw;
    if (row0 >= a.rows)
        return;   // uniform across the warp
    // lanes per row: one with the caller's norms, else D / 8 (the whole warp
    // for a single row)
    const int lpr = a.cnorm_in != nullptr ? 1 : (a.rpw == 1 ? 32 : a.D >> 3);
    const int64_t j = row0 + lane / lpr;
    float norm = __int_as_float(0x7fc00000);
    if (a.cnorm_in != nullptr) {
        if (j < a.K)
            norm = __ldg(a.cnorm_in + j);
    } else {
        const float acc = warp_rows_norm(a.C, row0, a.K, a.D, lane);
        if (j < a.K)
            norm = acc;
    }
    if (lane % lpr != 0 || j >= a.rows)
        return;
    if (a.cnorm_out != nullptr && j < a.K)
        a.cnorm_out[j] = norm;
    if (a.fold != nullptr) {
        uint32_t w0, w1;
        fold_split(norm, w0, w1);
        const int64_t b = j >> 7;
        const int64_t r = j & 127;
        a.fold[b * 256 + r] = make_uint4(w0, w1, 0u, 0u);
        a.fold[b * 256 + 128 + r] = make_uint4(0u, 0u, 0u, 0u);
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

// rows_per_warp on the host
static int rows_per_warp_host(int D)
{
    const int v = D >> 3;
    return (v < 32 && (v & (v - 1)) == 0) ? 32 / v : 1;
}

cudaError_t launch_norms(const void *C, int64_t K, int64_t D, float *cnorm, cudaStream_t stream)
{
    const int64_t rows_per_block = int64_t(kNormWarps) * rows_per_warp_host(static_cast<int>(D));
    const int64_t blocks = (K + rows_per_block - 1) / rows_per_block;
    norms_kernel<<<static_cast<unsigned>(blocks), 32 * kNormWarps, 0, stream>>>(
        static_cast<const uint4 *>(C), K, static_cast<int32_t>(D), cnorm);
    return cudaGetLastError();
}

cudaError_t launch_prep(const void *C, int64_t K, int64_t D, const float *cnorm_in,
                        float *cnorm_out, void *fold, void *fill, size_t fill_bytes,
                        cudaStream_t stream, bool *launched)
{
    *launched = false;
    PrepArgs a{};
    a.C = static_cast<const uint4 *>(C);
    a.cnorm_in = cnorm_in;
    a.cnorm_out = cnorm_out;
    a.fold = static_cast<uint4 *>(fold);
    a.fill = static_cast<uint4 *>(fill);
    a.K = K;
    a.D = static_cast<int32_t>(D);
    a.rows = std::max<int64_t>(cnorm_out != nullptr ? K : 0,
                               fold != nullptr ? fold_operand_blocks(K) * 128 : 0);
    a.fill_words = fill != nullptr ? static_cast<int64_t>(fill_bytes / 16) : 0;
    a.rpw = cnorm_in != nullptr ? 32 : rows_per_warp_host(static_cast<int>(D));
    const int64_t rows_per_block = int64_t(kNormWarps) * a.rpw;
    a.row_blocks = (a.rows + rows_per_block - 1) / rows_per_block;
    const int64_t fill_blocks =
        std::min<int64_t>((a.fill_words + 32 * kNormWarps - 1) / (32 * kNormWarps), 1024);
    const int64_t blocks = a.row_blocks + fill_blocks;
    if (blocks == 0)
        return cudaSuccess;
    prep_kernel<<<static_cast<unsigned>(blocks), 32 * kNormWarps, 0, stream>>>(a);
    *launched = true;
    return cudaGetLastError();
}

}  // namespace kma
