// pipeline.cuh -- the parts of the assignment pipeline shared by the kernels
// that consume score tiles (the nearest-centroid kernel and the k-nearest
// kernel): barrier layout, bounded waits, the work-unit schedule, the score
// arithmetic of a 32-column chunk, and the roles of the non-consumer warps of
// a single-block kernel (X loader, C producer, MMA issuer, norm stager).
//
// What the pipeline computes (flashlib PR #22 "Optimize Blackwell k-means
// assignment reduction", Summary and Key ideas): score tiles X . C^T on the
// tensor cores into tensor memory, then the centroid norms applied
// (s = ||c||^2 - 2 x.c) by the consumer warps, which differ per kernel.
//
// Each translation unit that includes this header gets its own status word
// (internal linkage) and must expose a host function that reads and clears
// it; the library checks all of them.
#pragma once

#include "internal.h"
#include "norm_math.cuh"
#include "ptx.cuh"

#include "kmassign.h"

#include <cuda_bf16.h>

namespace kma {
namespace {

// Status word of this translation unit's kernels (0 or a kmassign_status).
__device__ int g_status_word = 0;

// Barrier slots (8 bytes each) after the operand and staging buffers.
constexpr int kBarXFull = 0;                          // [kMaxXBufs]
constexpr int kBarXEmpty = kBarXFull + kMaxXBufs;     // [kMaxXBufs]
constexpr int kBarAccFull = kBarXEmpty + kMaxXBufs;   // [2]
constexpr int kBarAccEmpty = kBarAccFull + 2;         // [2]
constexpr int kBarDrain = kBarAccEmpty + 2;           // [1]
constexpr int kBarCFull = kBarDrain + 1;              // [kMaxStages]
constexpr int kBarCEmpty = kBarCFull + kMaxStages;    // [kMaxStages]
constexpr int kCnStages = 4;                          // centroid-norm ring depth
constexpr int kBarCnFull = kBarCEmpty + kMaxStages;   // [kCnStages]
constexpr int kBarCnEmpty = kBarCnFull + kCnStages;   // [kCnStages]
constexpr int kNumBars = kBarCnEmpty + kCnStages;
constexpr uint32_t kMiscBytes = kNumBars * 8 + 16;    // + tmem slot, abort flag, 2 split flags
// Norm folding (every assignment kernel at D <= 128, the k-nearest kernel at
// every D): the norms enter the accumulator through one more K = 16 MMA step
// per tile, A = a constant tile of ones, B = the tile's -||c||^2 / 2 split
// into three bf16 parts.  Single-block shared memory: the ones tile, then kFoldStages
// slots of NT rows x 32 bytes (plain K-major layout: 8-row groups of 256
// bytes, each two 128-byte core matrices along K) that a norm warp fills.
constexpr int kFoldStages = 3;
constexpr uint32_t kOnesBytes = 4096;                 // 128 rows x 16 columns of bf16 1.0
constexpr uint32_t kFoldLbo = 128;                    // between the two core matrices along K
constexpr uint32_t kFoldSbo = 256;                    // between 8-row groups
// The CTA pair's fold operand comes from global memory by TMA, one block of
// 128 centroids (4 KiB) per CTA and tile, laid out [K half][128 rows][16 B]:
// the same unswizzled K-major core matrices with other offsets.  It has one
// slot per group of C stages (the stages of one tile), loaded and freed with
// the group.
constexpr uint32_t kFoldBlockBytes = 4096;
constexpr uint32_t kFoldPairLbo = 2048;               // between the two K halves
constexpr uint32_t kFoldPairSbo = 128;                // between 8-row groups
constexpr uint32_t kConsumerBarrier = 1;              // named barrier id
constexpr uint32_t kSplitBarrier = 2;                 // + sub-tile: a split row group's barrier
// Bound on the teardown waits after an abort (copies and MMAs in flight
// always finish; this only guards against a hardware failure).
constexpr uint64_t kDrainLimitNs = 2000000000ull;

__device__ __forceinline__ void record_timeout()
{
    atomicCAS(&g_status_word, 0, static_cast<int>(KMASSIGN_ERR_TIMEOUT));
}

// Debug build (compiled with KMASSIGN_DEBUG): device-side consistency checks
// of what the host planned against what the kernels index -- the shared
// memory layout against the launch's dynamic size, ring and buffer counts,
// decoded work units against N and K, split-key indices against the split
// rows.  A failed check records KMASSIGN_ERR_DEBUG_CHECK in the status word
// (the first failure wins) and the access it guards is skipped or clamped;
// nothing traps.  In the normal build every check is the constant true.
#ifdef KMASSIGN_DEBUG
constexpr bool kDebugChecks = true;
#else
constexpr bool kDebugChecks = false;
#endif

__device__ __forceinline__ bool debug_ok(bool cond)
{
    if (kDebugChecks && !cond)
        atomicCAS(&g_status_word, 0, static_cast<int>(KMASSIGN_ERR_DEBUG_CHECK));
    return !kDebugChecks || cond;
}

__device__ __forceinline__ uint32_t dynamic_smem_bytes()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%dynamic_smem_size;" : "=r"(r));
    return r;
}

// The block's shared-memory layout ends at layout_end (bytes from the start
// of dynamic shared memory, alignment padding included) and its rings are
// within the compiled bounds.  Uniform across the block (and across a CTA
// pair, which computes the same): a block that fails returns before it sets
// anything up.
__device__ __forceinline__ bool debug_layout_ok(const AssignParams &p, uint32_t layout_end)
{
    if (!kDebugChecks)
        return true;
    const bool ok = layout_end <= dynamic_smem_bytes() && p.stages >= 2 &&
                    p.stages <= kMaxStages && p.xbufs >= 1 && p.xbufs <= kMaxXBufs && p.ksplit >= 1 &&
                    p.chunk_tiles >= 1 && p.ntiles >= 1;
    if (!ok && threadIdx.x == 0)
        debug_ok(false);
    return ok;
}

// Slow path of a bounded wait (the phase was not complete on first try).
__device__ __noinline__ bool wait_slow(uint32_t bar, uint32_t parity, volatile uint32_t *abort_flag,
                                       uint64_t limit_ns, bool honour_abort)
{
    const uint64_t t0 = globaltimer_ns();
    while (true) {
        if (mbar_try_wait(bar, parity))
            return true;
        if (honour_abort && *abort_flag)
            return false;
        if (globaltimer_ns() - t0 > limit_ns) {
            *abort_flag = 1u;
            record_timeout();
            return false;
        }
    }
}

// Single-thread bounded wait.  Returns false on timeout or block abort.
__device__ __forceinline__ bool wait1(uint32_t bar, uint32_t parity, volatile uint32_t *abort_flag,
                                      uint64_t limit_ns, bool honour_abort = true)
{
    if (mbar_try_wait(bar, parity))
        return true;
    return wait_slow(bar, parity, abort_flag, limit_ns, honour_abort);
}

// Whole-warp bounded wait; the decision is uniform across the warp.
__device__ __forceinline__ bool wait_warp(uint32_t bar, uint32_t parity,
                                          volatile uint32_t *abort_flag, uint64_t limit_ns,
                                          bool honour_abort = true)
{
    if (__all_sync(0xffffffffu, mbar_try_wait(bar, parity)))
        return true;
    const uint64_t t0 = globaltimer_ns();
    while (true) {
        if (__all_sync(0xffffffffu, mbar_try_wait(bar, parity)))
            return true;
        int give_up = 0;
        if ((threadIdx.x & 31) == 0) {
            if (honour_abort && *abort_flag) {
                give_up = 1;
            } else if (globaltimer_ns() - t0 > limit_ns) {
                *abort_flag = 1u;
                record_timeout();
                give_up = 1;
            }
        }
        if (__shfl_sync(0xffffffffu, give_up, 0))
            return false;
    }
}

struct Unit {
    int32_t row0;      // first point of the row tile
    int32_t nsub;      // 128-point sub-tiles holding at least one point
    int32_t t_begin;   // first centroid tile
    int32_t t_end;     // one past the last centroid tile
    bool split;        // part of a split centroid range: merged after the kernel
};

// Units [0, full_units) cover one row tile and every centroid tile; the
// remaining units split the row tiles from split_row0 on into ksplit
// centroid ranges (all of them when full_units == 0, only the last, partial
// wave of row tiles when the plan balances the wave tail).
template <int SUB>
__device__ __forceinline__ Unit decode_unit(const AssignParams &p, int u)
{
    Unit w;
    int rt;
    if (u < p.full_units) {
        rt = u;
        w.t_begin = 0;
        w.t_end = p.ntiles;
        w.split = false;
    } else {
        const int v = u - p.full_units;
        const int r = v / p.ksplit;
        const int kc = v - r * p.ksplit;
        rt = p.split_row0 + r;
        w.t_begin = kc * p.chunk_tiles;
        w.t_end = min(p.ntiles, w.t_begin + p.chunk_tiles);
        w.split = true;
    }
    w.row0 = rt * SUB * kTileM;
    const int left = p.N - w.row0;
    w.nsub = min(SUB, (left + kTileM - 1) / kTileM);
    if (kDebugChecks &&
        !debug_ok(rt >= 0 && rt < p.rowtiles && left > 0 && w.t_begin >= 0 &&
                  w.t_begin < w.t_end && w.t_end <= p.ntiles)) {
        // clamped: an empty centroid range, every role alike
        w.t_end = w.t_begin = 0;
        w.nsub = max(w.nsub, 0);
    }
    return w;
}

// Minimum of 32 scores by a tree of 3-input mins (a NaN is ignored unless
// every score is NaN).
__device__ __forceinline__ float chunk_min(const float (&s)[32])
{
    float a[11];
#pragma unroll
    for (int i = 0; i < 10; ++i)
        a[i] = min3(s[3 * i], s[3 * i + 1], s[3 * i + 2]);
    a[10] = min2(s[30], s[31]);
    const float b0 = min3(a[0], a[1], a[2]);
    const float b1 = min3(a[3], a[4], a[5]);
    const float b2 = min3(a[6], a[7], a[8]);
    const float b3 = min2(a[9], a[10]);
    return min3(b0, b1, min2(b2, b3));
}

// s[i] = fmaf(-2, acc[i], cnorm[j0 + i]) in place, norms from shared memory.
__device__ __forceinline__ void apply_norms(float (&v)[32], uint32_t cn_addr)
{
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const float4 c = ld_shared_v4(cn_addr + 16u * i);
        fma2(v[4 * i + 0], v[4 * i + 1], -2.0f, -2.0f, v[4 * i + 0], v[4 * i + 1], c.x, c.y);
        fma2(v[4 * i + 2], v[4 * i + 3], -2.0f, -2.0f, v[4 * i + 2], v[4 * i + 3], c.z, c.w);
    }
}

// Barriers of a single-block kernel with kConsumerWarps consumer warps
// (thread 0 only).  With FOLD the norm slots are freed by the MMA warp's
// commit instead of by the consumers.
template <int kConsumerWarps, bool FOLD = false>
__device__ __forceinline__ void init_barriers(uint32_t bar_base, volatile uint32_t *abort_flag)
{
    auto bar = [&](int i) -> uint32_t { return bar_base + 8u * static_cast<uint32_t>(i); };
    for (int b = 0; b < kMaxXBufs; ++b) {
        mbar_init(bar(kBarXFull + b), 1);
        mbar_init(bar(kBarXEmpty + b), 1);
    }
    for (int a = 0; a < 2; ++a) {
        mbar_init(bar(kBarAccFull + a), 1);
        mbar_init(bar(kBarAccEmpty + a), kConsumerWarps);
    }
    mbar_init(bar(kBarDrain), 1);
    for (int s = 0; s < kMaxStages; ++s) {
        mbar_init(bar(kBarCFull + s), 1);
        mbar_init(bar(kBarCEmpty + s), 1);
    }
    for (int s = 0; s < kCnStages; ++s) {
        mbar_init(bar(kBarCnFull + s), 32);
        mbar_init(bar(kBarCnEmpty + s), FOLD ? 1 : kConsumerWarps);
    }
    *abort_flag = 0u;
    fence_mbar_init();
}

// Producer warp: streams C k-blocks (NT rows x 64 columns each) through the
// ring of shared-memory stages, straight across unit boundaries.
template <int SUB, int NT, int KB>
__device__ __forceinline__ void producer_role(const AssignParams &p, const CUtensorMap *xmap,
                                              const CUtensorMap *cmap, uint32_t c_base,
                                              uint32_t bar_base, volatile uint32_t *abort_flag)
{
    constexpr uint32_t kCStageBytes = NT * 128;
    auto bar = [&](int i) -> uint32_t { return bar_base + 8u * static_cast<uint32_t>(i); };
    if ((threadIdx.x & 31) == 0) {
        tma_prefetch_desc(xmap);
        tma_prefetch_desc(cmap);
        const uint64_t pol_c = policy_evict_last();
        uint32_t stage = 0, phase = 0;
        uint32_t c_issued = 0;
        bool ok = true;
        for (int u = blockIdx.x; ok && u < p.num_units; u += gridDim.x) {
            const Unit w = decode_unit<SUB>(p, u);
            for (int tile = w.t_begin; ok && tile < w.t_end; ++tile) {
#pragma unroll
                for (int kb = 0; kb < KB; ++kb) {
                    if (!(ok = wait1(bar(kBarCEmpty + stage), phase ^ 1u, abort_flag,
                                     p.timeout_ns)))
                        break;
                    mbar_arrive_expect_tx(bar(kBarCFull + stage), kCStageBytes);
                    tma_load_2d(c_base + stage * kCStageBytes, cmap, bar(kBarCFull + stage),
                                kb * kKBlock, tile * NT, pol_c);
                    ++c_issued;
                    if (++stage == static_cast<uint32_t>(p.stages)) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
        }
        if (!ok) {
            // Let every copy still in flight land before the block exits.
            const uint32_t S = p.stages;
            for (uint32_t n = (c_issued > S ? c_issued - S : 0); n < c_issued; ++n)
                wait1(bar(kBarCFull + n % S), (n / S) & 1u, abort_flag, kDrainLimitNs, false);
        }
    }
    __syncwarp();
}

// X warp: TMA-loads the block's X tile once per work unit; it stays resident
// while the unit's centroids stream past it.
template <int SUB, int KB>
__device__ __forceinline__ void x_role(const AssignParams &p, const CUtensorMap *xmap,
                                       uint32_t x_base, uint32_t bar_base,
                                       volatile uint32_t *abort_flag)
{
    constexpr uint32_t kXBufBytes = SUB * KB * kXTileBytes;
    auto bar = [&](int i) -> uint32_t { return bar_base + 8u * static_cast<uint32_t>(i); };
    if ((threadIdx.x & 31) == 0) {
        const uint64_t pol_x = policy_evict_first();
        uint32_t x_issued = 0;
        bool ok = true;
        for (int u = blockIdx.x; ok && u < p.num_units; u += gridDim.x) {
            const Unit w = decode_unit<SUB>(p, u);
            const uint32_t xb = x_issued % p.xbufs;
            const uint32_t xph = (x_issued / p.xbufs) & 1u;
            if (!(ok = wait1(bar(kBarXEmpty + xb), xph ^ 1u, abort_flag, p.timeout_ns)))
                break;
            mbar_arrive_expect_tx(bar(kBarXFull + xb), w.nsub * KB * kXTileBytes);
            const uint32_t xdst = x_base + xb * kXBufBytes;
            for (int t = 0; t < w.nsub; ++t)
#pragma unroll
                for (int kb = 0; kb < KB; ++kb)
                    tma_load_2d(xdst + (t * KB + kb) * kXTileBytes, xmap, bar(kBarXFull + xb),
                                kb * kKBlock, w.row0 + t * kTileM, pol_x);
            ++x_issued;
        }
        if (!ok) {
            const uint32_t B = p.xbufs;
            for (uint32_t n = (x_issued > B ? x_issued - B : 0); n < x_issued; ++n)
                wait1(bar(kBarXFull + n % B), (n / B) & 1u, abort_flag, kDrainLimitNs, false);
        }
    }
    __syncwarp();
}

// MMA warp: the whole warp walks the schedule and waits; one elected lane
// issues tcgen05.mma into one of two accumulator stages.  The k-loop is
// unrolled at compile time with the operand descriptors computed once per
// unit: the tensor pipe's issue queue is shallow and any extra work between
// MMAs shows up as pipe bubbles.
// With FOLD, each tile gets one more K = 16 step that adds -||c||^2 / 2
// (ones x the norm slot the norm warp filled), and its commit frees the slot.
template <int SUB, int NT, int KB, bool FOLD = false>
__device__ __forceinline__ void mma_role(const AssignParams &p, uint32_t x_base, uint32_t c_base,
                                         uint32_t bar_base, uint32_t tmem_base,
                                         volatile uint32_t *abort_flag, uint32_t fold_base = 0)
{
    constexpr uint32_t kCStageBytes = NT * 128;
    constexpr uint32_t kXBufBytes = SUB * KB * kXTileBytes;
    constexpr uint32_t kAccCols = SUB * NT;
    constexpr uint32_t kIdesc = idesc_bf16_f32(kTileM, NT);
    constexpr bool kPreWait = FOLD && KB <= 2;
    auto bar = [&](int i) -> uint32_t { return bar_base + 8u * static_cast<uint32_t>(i); };
    uint32_t stage = 0, phase = 0, x_used = 0, acc_used = 0, fold_used = 0;
    bool ok = true, issued = false;
    const uint64_t ones_desc = FOLD ? plain_kmajor_desc(fold_base, kFoldLbo, kFoldSbo) : 0;
    for (int u = blockIdx.x; ok && u < p.num_units; u += gridDim.x) {
        const Unit w = decode_unit<SUB>(p, u);
        const uint32_t xb = x_used % p.xbufs;
        const uint32_t xph = (x_used / p.xbufs) & 1u;
        // Operands landed by TMA are ordered by the mbarrier itself; no
        // tcgen05 fence is needed before MMAs read them.
        if (!(ok = wait_warp(bar(kBarXFull + xb), xph, abort_flag, p.timeout_ns)))
            break;
        uint64_t adesc[SUB][KB];
#pragma unroll
        for (int t = 0; t < SUB; ++t)
#pragma unroll
            for (int kb = 0; kb < KB; ++kb)
                adesc[t][kb] =
                    sw128_kmajor_desc(x_base + xb * kXBufBytes + (t * KB + kb) * kXTileBytes);
        for (int tile = w.t_begin; ok && tile < w.t_end; ++tile) {
            const uint32_t as = acc_used & 1u;
            const uint32_t aph = (acc_used >> 1) & 1u;
            const uint32_t fb = fold_used % kFoldStages;
            const uint32_t fph = (fold_used / kFoldStages) & 1u;
            if (kPreWait) {
                // Short folded tiles: the operands (copied tiles ahead) are
                // waited for before the accumulator stage, so the MMAs issue
                // as soon as the consumers hand the stage back.  Only at
                // KB <= 2: the ring always holds that many stages.
                uint32_t s2 = stage, ph2 = phase;
#pragma unroll
                for (int kb = 0; kb < KB; ++kb) {
                    if (ok)
                        ok = wait_warp(bar(kBarCFull + s2), ph2, abort_flag, p.timeout_ns);
                    if (++s2 == static_cast<uint32_t>(p.stages)) {
                        s2 = 0;
                        ph2 ^= 1u;
                    }
                }
                if (ok)
                    ok = wait_warp(bar(kBarCnFull + fb), fph, abort_flag, p.timeout_ns);
                if (!ok)
                    break;
            }
            if (!(ok = wait_warp(bar(kBarAccEmpty + as), aph ^ 1u, abort_flag, p.timeout_ns)))
                break;
            tc_fence_after();
            const uint32_t d_tmem = tmem_base + as * kAccCols;
#pragma unroll
            for (int kb = 0; kb < KB; ++kb) {
                if (!kPreWait &&
                    !(ok = wait_warp(bar(kBarCFull + stage), phase, abort_flag, p.timeout_ns)))
                    break;
                const uint64_t cdesc = sw128_kmajor_desc(c_base + stage * kCStageBytes);
                if (elect_one()) {
                    // Sub-tiles past the last point compute on stale
                    // operands; their rows are never stored.
#pragma unroll
                    for (int k = 0; k < 4; ++k)
#pragma unroll
                        for (int t = 0; t < SUB; ++t)
                            mma_bf16(d_tmem + t * NT, adesc[t][kb] + 2u * k, cdesc + 2u * k,
                                     kIdesc, (kb | k) != 0);
                    mma_commit(bar(kBarCEmpty + stage));
                }
                __syncwarp();
                issued = true;
                if (++stage == static_cast<uint32_t>(p.stages)) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            if (!ok)
                break;
            if (FOLD) {
                if (!kPreWait &&
                    !(ok = wait_warp(bar(kBarCnFull + fb), fph, abort_flag, p.timeout_ns)))
                    break;
                const uint64_t bdesc =
                    plain_kmajor_desc(fold_base + kOnesBytes + fb * NT * 32u, kFoldLbo, kFoldSbo);
                if (elect_one()) {
#pragma unroll
                    for (int t = 0; t < SUB; ++t)
                        mma_bf16(d_tmem + t * NT, ones_desc, bdesc, kIdesc, 1u);
                    mma_commit(bar(kBarCnEmpty + fb));
                }
                __syncwarp();
                ++fold_used;
            }
            if (elect_one())
                mma_commit(bar(kBarAccFull + as));
            __syncwarp();
            ++acc_used;
        }
        if (!ok)
            break;
        if (elect_one())
            mma_commit(bar(kBarXEmpty + xb));
        __syncwarp();
        ++x_used;
    }
    if (issued) {
        // All MMAs (and the arrivals they signal) finish before teardown.
        if (elect_one())
            mma_commit(bar(kBarDrain));
        __syncwarp();
        wait_warp(bar(kBarDrain), 0u, abort_flag, kDrainLimitNs, false);
    }
}

// Norm warp: copies each tile's NT centroid norms (NaN past K) into one slot
// of a small ring in shared memory, up to kCnStages tiles ahead of the
// consumers, so the reduction reads them with broadcast shared loads.
template <int SUB, int NT>
__device__ __forceinline__ void norm_role(const AssignParams &p, float *cn_smem, uint32_t bar_base,
                                          volatile uint32_t *abort_flag)
{
    auto bar = [&](int i) -> uint32_t { return bar_base + 8u * static_cast<uint32_t>(i); };
    const int lane = threadIdx.x & 31;
    const float kNaN = __int_as_float(0x7fc00000);
    uint32_t n = 0;
    bool ok = true;
    for (int u = blockIdx.x; ok && u < p.num_units; u += gridDim.x) {
        const Unit w = decode_unit<SUB>(p, u);
        for (int tile = w.t_begin; tile < w.t_end; ++tile, ++n) {
            const uint32_t b = n % kCnStages;
            const uint32_t ph = (n / kCnStages) & 1u;
            if (!(ok = wait_warp(bar(kBarCnEmpty + b), ph ^ 1u, abort_flag, p.timeout_ns)))
                break;
            const int j = tile * NT;
#pragma unroll
            for (int e = 0; e < NT / 32; ++e) {
                const int i = e * 32 + lane;
                cn_smem[b * NT + i] = (j + i < p.K) ? __ldg(p.cnorm + j + i) : kNaN;
            }
            mbar_arrive(bar(kBarCnFull + b));   // release: this lane's stores
        }
    }
}

// Fill the ones tile and zero the norm slots (all threads of the block, before
// the block-wide barrier that follows the set-up).  The second core matrix of
// every slot row stays zero, so only the first 16 bytes change per tile.
template <int NT>
__device__ __forceinline__ void fold_init(uint32_t fold_base)
{
    constexpr uint32_t kBytes = kOnesBytes + kFoldStages * NT * 32u;
    const uint32_t one2 = 0x3F803F80u;   // two bf16 1.0
    for (uint32_t off = threadIdx.x * 16u; off < kBytes; off += blockDim.x * 16u) {
        const uint32_t w = off < kOnesBytes ? one2 : 0u;
        st_shared_v4_u32(fold_base + off, w, w, w, w);
    }
    fence_proxy_async_smem();
}

// Norm warp with FOLD: per tile, -||c_j||^2 / 2 for its NT centroids (NaN
// past K) split into three bf16 parts h + m + l (each the rounding of what
// the previous parts leave, so the sum carries the fp32 value's 24 bits), at
// K positions 0, 1, 2 of the tile's slot.  A non-finite value goes whole
// into h.  The MMA warp waits on these slots, so the next tile's norms are
// loaded before this tile's are split and stored (their latency overlaps).
template <int SUB, int NT>
__device__ __forceinline__ void fold_norm_role(const AssignParams &p, uint32_t fold_base,
                                               uint32_t bar_base, volatile uint32_t *abort_flag)
{
    constexpr int kPer = NT / 32;   // centroids per lane per tile
    auto bar = [&](int i) -> uint32_t { return bar_base + 8u * static_cast<uint32_t>(i); };
    const int lane = threadIdx.x & 31;
    const float kNaN = __int_as_float(0x7fc00000);
    auto load = [&](int tile, float (&cn)[kPer]) {
        const int j = tile * NT;
#pragma unroll
        for (int e = 0; e < kPer; ++e) {
            const int i = e * 32 + lane;
            cn[e] = (j + i < p.K) ? __ldg(p.cnorm + j + i) : kNaN;
        }
    };
    // The block's tiles in schedule order: (unit u, tile) pairs.
    int u = blockIdx.x;
    Unit w{};
    int tile = 0;
    bool have = u < p.num_units;
    if (have) {
        w = decode_unit<SUB>(p, u);
        tile = w.t_begin;
    }
    float cur[kPer];
    if (have)
        load(tile, cur);
    uint32_t n = 0;
    while (have) {
        // next tile of the schedule, and its norms in flight
        int u2 = u, tile2 = tile + 1;
        Unit w2 = w;
        if (tile2 >= w.t_end) {
            u2 = u + gridDim.x;
            if (u2 < p.num_units) {
                w2 = decode_unit<SUB>(p, u2);
                tile2 = w2.t_begin;
            }
        }
        const bool have2 = u2 < p.num_units;
        float nxt[kPer];
        if (have2)
            load(tile2, nxt);
        // split this tile's norms
        uint32_t w0[kPer], w1[kPer];
#pragma unroll
        for (int e = 0; e < kPer; ++e)
            fold_split(cur[e], w0[e], w1[e]);
        const uint32_t b = n % kFoldStages;
        const uint32_t ph = (n / kFoldStages) & 1u;
        if (!wait_warp(bar(kBarCnEmpty + b), ph ^ 1u, abort_flag, p.timeout_ns))
            break;
        const uint32_t slot = fold_base + kOnesBytes + b * NT * 32u;
#pragma unroll
        for (int e = 0; e < kPer; ++e) {
            const int i = e * 32 + lane;
            st_shared_v4_u32(slot + static_cast<uint32_t>(i >> 3) * kFoldSbo +
                                 static_cast<uint32_t>(i & 7) * 16u,
                             w0[e], w1[e], 0u, 0u);
        }
        fence_proxy_async_smem();
        mbar_arrive(bar(kBarCnFull + b));   // release: this lane's stores
        ++n;
        u = u2;
        w = w2;
        tile = tile2;
        have = have2;
#pragma unroll
        for (int e = 0; e < kPer; ++e)
            cur[e] = nxt[e];
    }
}

}  // namespace
}  // namespace kma
