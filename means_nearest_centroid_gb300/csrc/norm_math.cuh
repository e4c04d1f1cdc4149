// norm_math.cuh -- per-centroid arithmetic shared by the kernels that form
// the norms and by those that fold them into the tensor-core accumulator.
//
// What it computes (flashlib PR #22 "Optimize Blackwell k-means assignment
// reduction", Summary: the centroid norms applied to every score tile):
//   * ||c_j||^2 as an fp32 sum of the exact bf16 squares in one fixed order
//     (each lane of a warp squares and sums its 8 values in order, then a
//     fixed xor-shuffle tree adds the lanes), so every kernel that forms a
//     norm gets the same bits;
//   * -||c_j||^2 / 2 split into three bf16 parts h + m + l, each the
//     rounding of what the previous parts leave, so the parts carry all 24
//     bits of the fp32 value; they enter the accumulator as one more K = 16
//     tensor-core step against a tile of ones.
#pragma once

#include <cuda_bf16.h>

#include <cstdint>

namespace kma {
namespace {

// ||row||^2 of one bf16 row of D values (D a multiple of 16, at most 256) by
// a whole warp: lane l reads the row's l-th 16-byte vector.  Every lane
// returns the sum.
__device__ __forceinline__ float warp_row_norm(const uint4 *__restrict__ row, int D, int lane)
{
    const int vec_per_row = D >> 3;
    float acc = 0.0f;
    if (lane < vec_per_row) {
        const uint4 q = __ldg(row + lane);
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
    return acc;
}

// Rows of a warp: 32 / (D / 8) rows when D / 8 is a power of two below 32
// (D = 16, 32, 64, 128), one otherwise.
__device__ __forceinline__ int rows_per_warp(int D)
{
    const int v = D >> 3;
    return (v < 32 && (v & (v - 1)) == 0) ? 32 / v : 1;
}

// ||c_j||^2 for the rows_per_warp(D) rows row0 .. of a warp, D / 8 lanes per
// row (lane l: row row0 + l / (D / 8), vector l % (D / 8)); rows at or past K
// sum nothing.  The lanes of a row combine by the same xor tree as
// warp_row_norm restricted to the row's lanes -- the offsets it leaves out
// only add +0 there -- so the bits are warp_row_norm's.  Every lane returns
// its row's sum.
__device__ __forceinline__ float warp_rows_norm(const uint4 *__restrict__ C, int64_t row0, int64_t K,
                                                int D, int lane)
{
    const int vpr = D >> 3;
    if (rows_per_warp(D) == 1)
        return row0 < K ? warp_row_norm(C + row0 * vpr, D, lane) : 0.0f;
    const int64_t j = row0 + lane / vpr;
    float acc = 0.0f;
    if (j < K) {
        const uint4 q = __ldg(C + j * vpr + lane % vpr);
        const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float lo = __uint_as_float(w[i] << 16);
            const float hi = __uint_as_float(w[i] & 0xffff0000u);
            acc = fmaf(lo, lo, acc);
            acc = fmaf(hi, hi, acc);
        }
    }
    for (int off = vpr >> 1; off > 0; off >>= 1)
        acc += __shfl_xor_sync(0xffffffffu, acc, off);
    return acc;
}

__device__ __forceinline__ uint32_t bf16_bits(float v)
{
    return static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(v)));
}

// -c / 2 (c a centroid norm, NaN past K) split into three bf16 parts
// h + m + l, each the rounding of what the previous parts leave, so that
// the sum carries the fp32 value's 24 bits; w0 = h | m << 16, w1 = l: the
// first three K positions of the centroid's fold-operand row.  A non-finite
// value goes whole into h.
__device__ __forceinline__ void fold_split(float c, uint32_t &w0, uint32_t &w1)
{
    const float v = -0.5f * c;
    if (isfinite(v)) {
        const float h = __bfloat162float(__float2bfloat16_rn(v));
        const float r = v - h;
        const float m = __bfloat162float(__float2bfloat16_rn(r));
        w0 = bf16_bits(h) | (bf16_bits(m) << 16);
        w1 = bf16_bits(r - m);
    } else {
        w0 = bf16_bits(v);
        w1 = 0u;
    }
}

}  // namespace
}  // namespace kma
