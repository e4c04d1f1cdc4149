// update.cu -- the update step of a Lloyd iteration, which follows the
// assignment (not part of flashlib PR #22, which covers the assignment; the
// textbook update): counts[j] += |{i : idx[i] == j}| and sums[j][d] += the sum
// of x_id over those points, in fp32.  Ids outside [0, K) are skipped.
//
// Two ways to form the sums:
//   * atomic: every point adds its row into L2 with 16-byte vector
//     reductions.  One launch, but N * D / 4 reductions: the L2 atomic units,
//     not HBM, bound it (about a sixth of the copy bandwidth for D = 256).
//   * sorted: a counting sort groups the points by centroid (histogram, whose
//     last block runs the exclusive scan; scatter of (point, centroid)
//     pairs; when each block sees far more points than there are centroids,
//     blocks count in shared memory first and touch global counters once per
//     bin), then groups of D / 8 lanes walk runs of the sorted order,
//     gathering each point's row (one 16-byte load per lane) into registers
//     and adding the run's total and its number of points into L2 once per
//     centroid met.  About (N / R + K) * D / 4 reductions for runs of R
//     points, and X is read once, row by row.
// Either way the order in which a centroid's points are added is not fixed,
// so fp32 sums of non-integer data can differ in their last bits between
// runs; integer-valued data whose sums stay below 2^24 is exact.
#include "internal.h"

#include <algorithm>

namespace kma {
namespace {

__device__ __forceinline__ void red_add_v4(float *dst, float a, float b, float c, float d)
{
    asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(dst), "f"(a), "f"(b),
                 "f"(c), "f"(d)
                 : "memory");
}

__device__ __forceinline__ void widen8(const uint4 &q, float (&f)[8])
{
    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        f[2 * e] = __uint_as_float(w[e] << 16);
        f[2 * e + 1] = __uint_as_float(w[e] & 0xffff0000u);
    }
}

// Atomic form: a group of D/8 lanes takes one point at a time.
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
        float f[8];
        widen8(__ldg(X + i * vec + part), f);
        float *dst = sums + static_cast<int64_t>(j) * D + part * 8;
        red_add_v4(dst, f[0], f[1], f[2], f[3]);
        red_add_v4(dst + 4, f[4], f[5], f[6], f[7]);
    }
}

// ---- sorted form ----------------------------------------------------------

constexpr int kScanThreads = 1024;
constexpr int kScanPer = 4;                           // elements per thread
constexpr int kScanTile = kScanThreads * kScanPer;    // elements per block tile
constexpr int64_t kSmallScanMax = 65536;              // centroids scanned by one block
constexpr int kBinsPerThread = 16;                    // one-block scan: four 16-byte loads
constexpr int kBinTile = kScanThreads * kBinsPerThread;
constexpr int64_t kLocalMaxBins = 12288;              // 48 KiB of shared counters per block

// Points per thread in the scatter pass: its atomics are independent, so a
// thread keeps this many in flight.  The histogram pass runs 1024-thread
// blocks (its last block scans) with 2 points per thread, so that it still
// spreads over the SMs.
constexpr int kPerThread = 8;
constexpr int kHistPerThread = 2;

// Counters are padded to a multiple of 16 bins, so the one-block scan reads
// and writes them with 16-byte accesses.
inline int64_t padded_bins(int64_t K) { return (K + 15) / 16 * 16; }

// Exclusive scan of one value per thread over a block of kScanThreads;
// *block_total receives the sum.  Uses 33 int64 of shared memory.
__device__ __forceinline__ int64_t block_exclusive_scan(int64_t v, int64_t *warp_sums,
                                                        int64_t *block_total)
{
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    int64_t incl = v;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int64_t t = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off)
            incl += t;
    }
    if (lane == 31)
        warp_sums[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        const int64_t w = warp_sums[lane];
        int64_t wi = w;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int64_t t = __shfl_up_sync(0xffffffffu, wi, off);
            if (lane >= off)
                wi += t;
        }
        warp_sums[lane] = wi - w;   // exclusive prefix of warp totals
        if (lane == 31)
            warp_sums[32] = wi;
    }
    __syncthreads();
    const int64_t out = incl - v + warp_sums[warp];
    *block_total = warp_sums[32];
    __syncthreads();   // warp_sums is reused by the caller's next scan
    return out;
}

// cursor[j] = sum of hist[0, j) over the Kp padded bins (K <= kSmallScanMax),
// by one whole block of kScanThreads threads in tiles of kBinTile bins;
// *total_out = the sum of all bins.  hist is read at L2 (it was written by
// other blocks' atomics).  hist and cursor are 16-byte aligned.
__device__ void scan_bins_block(const int32_t *hist, int64_t Kp, int32_t *cursor,
                                int32_t *total_out, int64_t *warp_sums)
{
    int64_t carry = 0;
    for (int64_t t0 = 0; t0 < Kp; t0 += kBinTile) {
        const int64_t base = t0 + static_cast<int64_t>(threadIdx.x) * kBinsPerThread;
        const bool mine = base < Kp;   // Kp and base are multiples of 16
        int4 h[4] = {};
        if (mine) {
#pragma unroll
            for (int q = 0; q < 4; ++q)
                h[q] = __ldcg(reinterpret_cast<const int4 *>(hist + base) + q);
        }
        int64_t v = 0;
#pragma unroll
        for (int q = 0; q < 4; ++q)
            v += static_cast<int64_t>(h[q].x) + h[q].y + h[q].z + h[q].w;
        int64_t total;
        int64_t run = carry + block_exclusive_scan(v, warp_sums, &total);
        if (mine) {
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                int4 c;
                c.x = static_cast<int32_t>(run);
                run += h[q].x;
                c.y = static_cast<int32_t>(run);
                run += h[q].y;
                c.z = static_cast<int32_t>(run);
                run += h[q].z;
                c.w = static_cast<int32_t>(run);
                run += h[q].w;
                reinterpret_cast<int4 *>(cursor + base)[q] = c;
            }
        }
        carry += total;
    }
    if (threadIdx.x == 0)
        *total_out = static_cast<int32_t>(carry);
}

// Called by every thread of a counting block after its last atomic on hist:
// the block that finishes last runs the scan, so the histogram and the scan
// take one launch.  Each thread's fence orders its atomics before the
// block's ticket; the last block's fence orders the ticket before its reads.
__device__ void last_block_scans(uint32_t *ticket, const int32_t *hist, int64_t Kp,
                                 int32_t *cursor, int32_t *total_out)
{
    __shared__ int64_t warp_sums[33];
    __shared__ int is_last;
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0)
        is_last = atomicAdd(ticket, 1u) == gridDim.x - 1;
    __syncthreads();
    if (!is_last)
        return;
    __threadfence();
    scan_bins_block(hist, Kp, cursor, total_out, warp_sums);
}

// The scan alone, by one block (K <= kSmallScanMax), when the histogram was
// formed elsewhere (by the assignment kernel in the Lloyd loop).
__global__ void __launch_bounds__(kScanThreads)
    scan_kernel(const int32_t *hist, int64_t Kp, int32_t *cursor, int32_t *total)
{
    __shared__ int64_t warp_sums[33];
    scan_bins_block(hist, Kp, cursor, total, warp_sums);
}

// hist[j] += 1 for every point with a valid id; with scan, the last block
// then scans the bins.
__global__ void __launch_bounds__(kScanThreads)
    hist_kernel(const int32_t *__restrict__ idx, int64_t N, int32_t K, int32_t *hist, bool scan,
                int64_t Kp, uint32_t *ticket, int32_t *cursor, int32_t *total)
{
    const int64_t base =
        (static_cast<int64_t>(blockIdx.x) * blockDim.x) * kHistPerThread + threadIdx.x;
    int32_t j[kHistPerThread];
#pragma unroll
    for (int u = 0; u < kHistPerThread; ++u) {
        const int64_t i = base + static_cast<int64_t>(u) * blockDim.x;
        j[u] = i < N ? __ldg(idx + i) : -1;
    }
#pragma unroll
    for (int u = 0; u < kHistPerThread; ++u)
        if (j[u] >= 0 && j[u] < K)
            atomicAdd(hist + j[u], 1);
    if (scan)
        last_block_scans(ticket, hist, Kp, cursor, total);
}

// Phase A (many tiles only): tile_sum[b] = sum of hist over tile b.
__global__ void __launch_bounds__(kScanThreads)
    tile_sum_kernel(const int32_t *__restrict__ hist, int32_t K, int64_t *__restrict__ tile_sum)
{
    __shared__ int64_t warp_sums[33];
    const int64_t base = static_cast<int64_t>(blockIdx.x) * kScanTile + threadIdx.x * kScanPer;
    int64_t v = 0;
#pragma unroll
    for (int e = 0; e < kScanPer; ++e)
        if (base + e < K)
            v += hist[base + e];
    int64_t total;
    block_exclusive_scan(v, warp_sums, &total);
    if (threadIdx.x == 0)
        tile_sum[blockIdx.x] = total;
}

// Phase B (many tiles only, one block): tile_sum -> exclusive tile offsets.
__global__ void __launch_bounds__(kScanThreads)
    tile_offsets_kernel(int64_t *__restrict__ tile_sum, int64_t ntiles)
{
    __shared__ int64_t warp_sums[33];
    int64_t carry = 0;
    for (int64_t b0 = 0; b0 < ntiles; b0 += kScanThreads) {
        const int64_t b = b0 + threadIdx.x;
        const int64_t v = b < ntiles ? tile_sum[b] : 0;
        int64_t total;
        const int64_t ex = block_exclusive_scan(v, warp_sums, &total);
        if (b < ntiles)
            tile_sum[b] = carry + ex;
        carry += total;
    }
}

// Phase C: cursor[j] = first sorted position of centroid j; the block holding
// the last tile writes the number of sorted points.
__global__ void __launch_bounds__(kScanThreads)
    scan_apply_kernel(const int32_t *__restrict__ hist, int32_t K,
                      const int64_t *__restrict__ tile_off, int32_t *__restrict__ cursor,
                      int32_t *__restrict__ total_out)
{
    __shared__ int64_t warp_sums[33];
    const int64_t base = static_cast<int64_t>(blockIdx.x) * kScanTile + threadIdx.x * kScanPer;
    int32_t h[kScanPer];
    int64_t v = 0;
#pragma unroll
    for (int e = 0; e < kScanPer; ++e) {
        h[e] = base + e < K ? hist[base + e] : 0;
        v += h[e];
    }
    int64_t total;
    int64_t run = block_exclusive_scan(v, warp_sums, &total) + tile_off[blockIdx.x];
#pragma unroll
    for (int e = 0; e < kScanPer; ++e) {
        if (base + e < K)
            cursor[base + e] = static_cast<int32_t>(run);
        run += h[e];
    }
    if (blockIdx.x == gridDim.x - 1 && threadIdx.x == 0)
        *total_out = static_cast<int32_t>(tile_off[blockIdx.x] + total);
}

// perm[cursor[j]++] = (i, j) for every point i with a valid id j.
__global__ void __launch_bounds__(256)
    scatter_kernel(const int32_t *__restrict__ idx, int64_t N, int32_t K,
                   int32_t *__restrict__ cursor, int2 *__restrict__ perm)
{
    const int64_t base = (static_cast<int64_t>(blockIdx.x) * blockDim.x) * kPerThread + threadIdx.x;
    int32_t j[kPerThread], pos[kPerThread];
#pragma unroll
    for (int u = 0; u < kPerThread; ++u) {
        const int64_t i = base + static_cast<int64_t>(u) * blockDim.x;
        j[u] = i < N ? __ldg(idx + i) : -1;
    }
#pragma unroll
    for (int u = 0; u < kPerThread; ++u)
        pos[u] = (j[u] >= 0 && j[u] < K) ? atomicAdd(cursor + j[u], 1) : -1;
#pragma unroll
    for (int u = 0; u < kPerThread; ++u)
        if (pos[u] >= 0)
            perm[pos[u]] = make_int2(static_cast<int32_t>(base + static_cast<int64_t>(u) * blockDim.x),
                                     j[u]);
}

// Block-local counting, for K small against each block's share of points
// (the usual k-means regime, N >> K): counts gather in shared memory first,
// so the global atomics drop from one per point to one per (block, bin).
// Block b takes the contiguous points [b*per, (b+1)*per); with scan, the last
// block then scans the bins.
__global__ void __launch_bounds__(kScanThreads)
    block_hist_kernel(const int32_t *__restrict__ idx, int64_t N, int32_t K, int64_t per,
                      int32_t *hist, bool scan, int64_t Kp, uint32_t *ticket, int32_t *cursor,
                      int32_t *total)
{
    extern __shared__ int32_t h[];
    for (int j = threadIdx.x; j < K; j += blockDim.x)
        h[j] = 0;
    __syncthreads();
    const int64_t b0 = static_cast<int64_t>(blockIdx.x) * per;
    const int64_t b1 = min(N, b0 + per);
    for (int64_t i = b0 + threadIdx.x; i < b1; i += blockDim.x) {
        const int32_t j = __ldg(idx + i);
        if (j >= 0 && j < K)
            atomicAdd(h + j, 1);
    }
    __syncthreads();
    for (int j = threadIdx.x; j < K; j += blockDim.x)
        if (h[j] != 0)
            atomicAdd(hist + j, h[j]);
    if (scan)
        last_block_scans(ticket, hist, Kp, cursor, total);
}

// Each block counts its points again, reserves one range per bin in the
// sorted order (one global atomic per non-empty bin), then places its points
// with shared-memory atomics.
__global__ void __launch_bounds__(1024)
    block_scatter_kernel(const int32_t *__restrict__ idx, int64_t N, int32_t K, int64_t per,
                         int32_t *__restrict__ cursor, int2 *__restrict__ perm)
{
    extern __shared__ int32_t h[];
    for (int j = threadIdx.x; j < K; j += blockDim.x)
        h[j] = 0;
    __syncthreads();
    const int64_t b0 = static_cast<int64_t>(blockIdx.x) * per;
    const int64_t b1 = min(N, b0 + per);
    for (int64_t i = b0 + threadIdx.x; i < b1; i += blockDim.x) {
        const int32_t j = __ldg(idx + i);
        if (j >= 0 && j < K)
            atomicAdd(h + j, 1);
    }
    __syncthreads();
    for (int j = threadIdx.x; j < K; j += blockDim.x)
        if (h[j] != 0)
            h[j] = atomicAdd(cursor + j, h[j]);   // first sorted slot of this block's run
    __syncthreads();
    for (int64_t i = b0 + threadIdx.x; i < b1; i += blockDim.x) {
        const int32_t j = __ldg(idx + i);
        if (j >= 0 && j < K)
            perm[atomicAdd(h + j, 1)] = make_int2(static_cast<int32_t>(i), j);
    }
}

// Runs of R sorted points per group of D/8 lanes (R a multiple of kAhead):
// the group gathers kAhead rows at a time and adds a centroid's partial sum
// (and its number of points, to counts) into L2 whenever the centroid
// changes, and at the end of the run.
constexpr int kAhead = 8;

__global__ void __launch_bounds__(256)
    segsum_kernel(const uint4 *__restrict__ X, const int2 *__restrict__ perm,
                  const int32_t *__restrict__ total_p, int32_t D,
                  int32_t R, float *__restrict__ sums, int32_t *__restrict__ counts)
{
    const int lane = threadIdx.x & 31;
    const int vec = D >> 3;
    const int per_warp = 32 / vec;
    const int slot = lane / vec;
    const int part = lane - slot * vec;
    const int64_t warp = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t total = *total_p;
    const int64_t begin = (warp * per_warp + slot) * R;
    if (slot >= per_warp || begin >= total)
        return;   // no collective operations below
    const int64_t end = min(begin + R, total);
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    int32_t cur = -1;
    int32_t n = 0;   // points of centroid cur in this run
    auto flush = [&]() {
        float *dst = sums + static_cast<int64_t>(cur) * D + part * 8;
        red_add_v4(dst, acc[0], acc[1], acc[2], acc[3]);
        red_add_v4(dst + 4, acc[4], acc[5], acc[6], acc[7]);
        if (counts != nullptr && part == 0)
            atomicAdd(counts + cur, n);
    };
    for (int64_t s0 = begin; s0 < end; s0 += kAhead) {
        int32_t i[kAhead], j[kAhead];
        uint4 q[kAhead];
#pragma unroll
        for (int u = 0; u < kAhead; ++u) {
            const int2 ij = s0 + u < end ? __ldg(perm + s0 + u) : make_int2(-1, -1);
            i[u] = ij.x;
            j[u] = ij.y;
        }
#pragma unroll
        for (int u = 0; u < kAhead; ++u)
            if (i[u] >= 0)
                q[u] = __ldg(X + static_cast<int64_t>(i[u]) * vec + part);
#pragma unroll
        for (int u = 0; u < kAhead; ++u) {
            if (i[u] < 0)
                break;
            if (j[u] != cur) {
                if (cur >= 0)
                    flush();
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    acc[e] = 0.f;
                cur = j[u];
                n = 0;
            }
            ++n;
            float f[8];
            widen8(q[u], f);
#pragma unroll
            for (int e = 0; e < 8; ++e)
                acc[e] += f[e];
        }
    }
    if (cur >= 0)
        flush();
}

// The counting sort's placement and the run reductions (counts may be NULL:
// the histogram was formed elsewhere).
cudaError_t scatter_and_sum(const void *X, const int32_t *idx, int64_t N, int64_t K, int64_t D,
                            float *sums, int32_t *counts, int32_t *cursor, int2 *perm,
                            const int32_t *total, bool local, int64_t lblocks, int64_t lper,
                            size_t lsmem, int sms, cudaStream_t stream)
{
    const int threads = 256;
    if (local)
        block_scatter_kernel<<<static_cast<unsigned>(lblocks), 1024, lsmem, stream>>>(
            idx, N, static_cast<int32_t>(K), lper, cursor, perm);
    else
        scatter_kernel<<<static_cast<unsigned>(
                             (N + int64_t(threads) * kPerThread - 1) / (int64_t(threads) * kPerThread)),
                         threads, 0, stream>>>(idx, N, static_cast<int32_t>(K), cursor, perm);
    // Runs of R points: enough groups to give every SM about 48 resident warps.
    const int vec = static_cast<int>(D / 8);
    const int per_warp = 32 / vec;
    const int64_t groups_target = int64_t(sms) * 48 * per_warp;
    int64_t R = (N + groups_target - 1) / groups_target;
    R = std::max<int64_t>(kAhead, (R + kAhead - 1) / kAhead * kAhead);
    const int64_t groups = (N + R - 1) / R;
    const int64_t warps = (groups + per_warp - 1) / per_warp;
    const int64_t sblocks = (warps * 32 + threads - 1) / threads;
    segsum_kernel<<<static_cast<unsigned>(sblocks), threads, 0, stream>>>(
        static_cast<const uint4 *>(X), perm, total, static_cast<int32_t>(D),
        static_cast<int32_t>(R), sums, counts);
    return cudaGetLastError();
}

// counted == nullptr: count, scan, scatter and sum, adding the counts into
// counts.  counted != nullptr: the histogram is given (padded, zero past K);
// scan it, scatter and sum (counts unused).
cudaError_t launch_update_sorted_impl(const void *X, const int32_t *idx, int64_t N, int64_t K,
                                      int64_t D, float *sums, int32_t *counts,
                                      const int32_t *counted, void *scratch, int sms,
                                      cudaStream_t stream)
{
    // scratch: [ticket 16 B][hist Kp][cursor Kp][perm 2N][tile offsets][total]
    const int64_t ntiles = (K + kScanTile - 1) / kScanTile;
    const int64_t Kp = padded_bins(K);
    uint8_t *p = static_cast<uint8_t *>(scratch);
    uint32_t *ticket = reinterpret_cast<uint32_t *>(p);
    int32_t *hist = reinterpret_cast<int32_t *>(p + 16);
    int32_t *cursor = hist + Kp;
    int2 *perm = reinterpret_cast<int2 *>(cursor + Kp);   // Kp is even: 8-byte aligned
    uint8_t *tail = reinterpret_cast<uint8_t *>(perm + N);
    int64_t *tile_off = reinterpret_cast<int64_t *>(
        (reinterpret_cast<uintptr_t>(tail) + 7) & ~uintptr_t(7));
    int32_t *total = reinterpret_cast<int32_t *>(tile_off + ntiles);
    const bool one_block_scan = K <= kSmallScanMax;
    // Block-local counting when blocks of about 4K points each (so nearly
    // every bin of a block is hit, and the global atomics drop about 4x) still
    // give at least 32 blocks.
    const int64_t lblocks = std::min<int64_t>(int64_t(sms) * 2, N / (4 * K));
    const bool local = K <= kLocalMaxBins && lblocks >= 32;
    const int64_t lper = local ? (N + lblocks - 1) / lblocks : 0;
    const size_t lsmem = static_cast<size_t>(K) * 4;
    if (counted != nullptr) {
        if (one_block_scan)
            scan_kernel<<<1, kScanThreads, 0, stream>>>(counted, Kp, cursor, total);
        else {
            tile_sum_kernel<<<static_cast<unsigned>(ntiles), kScanThreads, 0, stream>>>(
                counted, static_cast<int32_t>(K), tile_off);
            tile_offsets_kernel<<<1, kScanThreads, 0, stream>>>(tile_off, ntiles);
            scan_apply_kernel<<<static_cast<unsigned>(ntiles), kScanThreads, 0, stream>>>(
                counted, static_cast<int32_t>(K), tile_off, cursor, total);
        }
        return scatter_and_sum(X, idx, N, K, D, sums, nullptr, cursor, perm, total, local, lblocks,
                               lper, lsmem, sms, stream);
    }
    // One memset clears the ticket and the padded bins.
    cudaError_t e = cudaMemsetAsync(p, 0, 16 + static_cast<size_t>(Kp) * 4, stream);
    if (e != cudaSuccess)
        return e;
    // With K <= kSmallScanMax the counting kernel's last block scans the bins.
    const int64_t blocks =
        (N + int64_t(kScanThreads) * kHistPerThread - 1) / (int64_t(kScanThreads) * kHistPerThread);
    if (local)
        block_hist_kernel<<<static_cast<unsigned>(lblocks), kScanThreads, lsmem, stream>>>(
            idx, N, static_cast<int32_t>(K), lper, hist, one_block_scan, Kp, ticket, cursor,
            total);
    else
        hist_kernel<<<static_cast<unsigned>(blocks), kScanThreads, 0, stream>>>(
            idx, N, static_cast<int32_t>(K), hist, one_block_scan, Kp, ticket, cursor, total);
    if (!one_block_scan) {
        tile_sum_kernel<<<static_cast<unsigned>(ntiles), kScanThreads, 0, stream>>>(
            hist, static_cast<int32_t>(K), tile_off);
        tile_offsets_kernel<<<1, kScanThreads, 0, stream>>>(tile_off, ntiles);
        scan_apply_kernel<<<static_cast<unsigned>(ntiles), kScanThreads, 0, stream>>>(
            hist, static_cast<int32_t>(K), tile_off, cursor, total);
    }
    return scatter_and_sum(X, idx, N, K, D, sums, counts, cursor, perm, total, local, lblocks,
                           lper, lsmem, sms, stream);
}

}  // namespace

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

size_t update_sorted_scratch_bytes(int64_t N, int64_t K)
{
    const int64_t ntiles = (K + kScanTile - 1) / kScanTile;
    return 16 +                                              // ticket
           static_cast<size_t>(padded_bins(K)) * 4 * 2 +     // hist, cursor
           static_cast<size_t>(N) * 8 +                      // perm: (point, centroid)
           8 + static_cast<size_t>(ntiles) * 8 + 64;         // tile offsets, total
}

int64_t update_padded_bins(int64_t K)
{
    return padded_bins(K);
}

cudaError_t launch_update_sorted_counted(const void *X, const int32_t *idx, int64_t N, int64_t K,
                                         int64_t D, float *sums, const int32_t *counts,
                                         void *scratch, int sms, cudaStream_t stream)
{
    return launch_update_sorted_impl(X, idx, N, K, D, sums, nullptr, counts, scratch, sms,
                                     stream);
}

cudaError_t launch_update_sorted(const void *X, const int32_t *idx, int64_t N, int64_t K,
                                 int64_t D, float *sums, int32_t *counts, void *scratch, int sms,
                                 cudaStream_t stream)
{
    return launch_update_sorted_impl(X, idx, N, K, D, sums, counts, nullptr, scratch, sms,
                                     stream);
}

}  // namespace kma
