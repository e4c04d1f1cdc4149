// assign.cu -- the warp-specialised k-means assignment kernel for sm_103a.
//
// What it computes (flashlib PR #22 "Optimize Blackwell k-means assignment
// reduction", Summary and Key ideas): for each point, the score tile
// X . C^T is produced by the tensor cores into tensor memory, the centroid
// norms are applied (s = ||c||^2 - 2 x.c) and the winning centroid is
// selected with lowest-index tie breaking.
//
// Roles inside one thread block (one block per SM, persistent; the first four
// are shared with the k-nearest kernel and live in pipeline.cuh):
//   * X warp         - TMA-loads the block's X tile once per work unit (the
//                      tile stays resident while centroids stream past it);
//   * producer warp  - streams C k-blocks through a ring of shared-memory
//                      stages guarded by full/empty mbarriers, straight across
//                      unit boundaries;
//   * MMA warp       - converged, one elected lane issues tcgen05.mma (bf16
//                      in, fp32 out) into one of two tensor-memory accumulator
//                      stages; the k-loop is unrolled at compile time with the
//                      operand descriptors computed once per unit, because the
//                      tensor pipe's issue queue is shallow and any extra work
//                      between MMAs shows up as pipe bubbles;
//   * consumer warps - 4 per 128-point sub-tile and column slice, one point
//                      per thread: load the scores with tcgen05.ld, wait for
//                      the loads, hand the accumulator stage back (the
//                      fenced-load pattern of the Key ideas table), then apply
//                      the norms and reduce.
//
// Centroid norms reach the consumers through shared memory: a norm warp runs
// up to kCnStages tiles ahead, copying each tile's norms (NaN past K) into a
// small ring guarded by full/empty mbarriers, so the reduction reads them
// with broadcast shared loads (the L1 cache is mostly carved out for the
// operand ring and would miss) and the consumer warps never wait on one
// another within a unit.
//
// The reduction works on 32-column chunks: s = fmaf(-2, acc, cnorm) for the
// chunk (two lanes per packed fma), the chunk minimum by a 3-input min tree
// (NaN ignored) -- four chunks at a time so their dependency chains overlap --
// and only when a chunk minimum beats the running best is the first column
// holding it located.  The whole warp pays for that step whenever any of its
// lanes improves, which early in a scan is nearly every chunk, so for D <= 128
// (where the reduction, not the tensor pipe, bounds the kernel) an improving
// lane only stores its chunk's 32 scores to its own shared-memory slot and
// the position is found once, when the unit ends; for larger D the lane
// searches at once.  Chunks are visited in increasing centroid order, so a
// warp keeps the lowest index on ties; column slices and split centroid
// ranges merge by (score, index).  A NaN score never wins.
//
// A work unit is (row tile, centroid range).  When the centroid axis of a
// row tile is split (for every row tile when there are too few of them to
// fill the GPU, or only for the last, partial wave of row tiles -- the
// wave-tail balancing of the GEMM page, applied along K), partial winners
// meet in a 64-bit atomicMin on keys holding the order-preserving score bits
// above the centroid index, which keeps the result deterministic and the
// lowest index on ties.
//
// Every mbarrier wait is bounded by p.timeout_ns of %globaltimer.  A wait that
// runs out records KMASSIGN_ERR_TIMEOUT in the status word and raises a
// block-wide abort flag; after that every wait returns at once, consumer
// warps skip their work but keep meeting their named barrier, the producer
// waits (again bounded) for its copies in flight, the MMA warp waits for its
// MMAs, and the tensor memory is freed before the block returns.
#include "pipeline.cuh"

#include <algorithm>

namespace kma {
namespace {

// Ordered key: fp32 score bits mapped so unsigned order == numeric order,
// -0 folded onto +0, index in the low word.
__device__ __forceinline__ unsigned long long pack_key(float s, int j)
{
    uint32_t u = __float_as_uint(s);
    if (u == 0x80000000u)
        u = 0u;
    const uint32_t o = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
    return (static_cast<unsigned long long>(o) << 32) | static_cast<uint32_t>(j);
}

// Key of a unit that saw no number (every score NaN): above every real key
// (whose high word is at most that of +inf), below the initial all-ones.
constexpr unsigned long long kKeyNoNumber = ~1ull;

// The (index, score) a packed key stands for; a key with an all-ones high
// word (the initial value, or kKeyNoNumber: no number seen, every score NaN)
// gives index 0 and NaN.
__device__ __forceinline__ void unpack_key(unsigned long long key, int &ix, float &ms)
{
    if ((key >> 32) == 0xffffffffull) {
        ix = 0;
        ms = __int_as_float(0x7fc00000);
        return;
    }
    ix = static_cast<int>(key & 0xffffffffull);
    const uint32_t o = static_cast<uint32_t>(key >> 32);
    ms = __uint_as_float((o & 0x80000000u) ? (o & 0x7fffffffu) : ~o);
}

// The row's answer from its merged key: idx, the histogram count, minscore.
__device__ __forceinline__ void store_split_row(const AssignParams &p, int row,
                                                unsigned long long key)
{
    int ix;
    float ms;
    unpack_key(key, ix, ms);
    p.idx[row] = ix;
    if (p.counts != nullptr)
        atomicAdd(p.counts + ix, 1);
    if (p.minscore != nullptr)
        p.minscore[row] = ms;
}

// Split rows, at the end of a unit, by all 128 consumer threads of one group
// of 128 rows (bar_id: a named barrier of theirs; flag: a shared word of
// theirs).  Every key starts at all-ones.
// - Two units per row (p.ksplit == 2, the usual tail split): each thread
//   merges its winner (kKeyNoNumber when it saw no number) with one atomicMin
//   and gets the key it replaced.  Anything but all-ones there is the other
//   unit's winner, already merged, so this thread holds both and stores the
//   row; the atomic's own order on the one key is the whole protocol.
// - More units per row: merge this unit's winners into the packed keys, then
//   count the unit in at the group's counter.  The counter starts at
//   all-ones, so the unit that reads ksplit - 2 is the last; it turns the
//   group's keys into idx and minscore.  Each thread fences its atomic before
//   the count, and the last unit fences before it reads the keys from L2.
__device__ __forceinline__ void merge_split_group(const AssignParams &p, int rows_per_unit,
                                                  int row, bool store, float best, int bi,
                                                  uint32_t bar_id, volatile uint32_t *flag,
                                                  bool counts)
{
    const int64_t rel = row - static_cast<int64_t>(p.split_row0) * rows_per_unit;
    if (kDebugChecks) {
        // the keys and counters cover exactly the split rows
        const int64_t n_split = p.N - static_cast<int64_t>(p.split_row0) * rows_per_unit;
        store = store && debug_ok(rel >= 0 && rel < n_split);
        counts = counts && debug_ok(rel >= 0 && (rel >> 7) < (n_split + 127) / 128);
    }
    if (p.ksplit == 2) {
        if (store) {
            const unsigned long long mine = bi == kNone ? kKeyNoNumber : pack_key(best, bi);
            const unsigned long long old = atomicMin(p.keys + rel, mine);
            if (old != ~0ull)
                store_split_row(p, row, old < mine ? old : mine);
        }
        return;
    }
    if (store && bi != kNone)
        atomicMin(p.keys + rel, pack_key(best, bi));
    __threadfence();
    named_bar_sync(bar_id, 128);
    if (counts) {
        const uint32_t old = atomicAdd(p.counters + (rel >> 7), 1u);
        *flag = old == static_cast<uint32_t>(p.ksplit - 2) ? 1u : 0u;
    }
    named_bar_sync(bar_id, 128);
    if (*flag != 0u) {
        __threadfence();
        if (store)
            store_split_row(p, row, __ldcg(p.keys + rel));
    }
}

// First position of m in s (m is the minimum of s, so one exists).
__device__ __forceinline__ int first_of(const float (&s)[32], float m)
{
    int pos = 31;
#pragma unroll
    for (int i = 30; i >= 0; --i)
        pos = (s[i] == m) ? i : pos;
    return pos;
}

// Fold chunk scores s (columns j0 .. j0+31, chunk minimum m) into (best, bi).
// SNAP: keep the chunk's scores in this thread's shared slot (float4 i of
// thread t at slot + 512*i, conflict-free across the warp) and let bi hold the
// chunk's first column until resolve_snapshot.  MAX: the values are
// t = -s / 2 (norm-folded accumulators), so the best is the largest, and m is
// the chunk maximum.
template <bool SNAP, bool MAX = false>
__device__ __forceinline__ void fold_chunk(const float (&s)[32], float m, int j0, float &best,
                                           int &bi, uint32_t slot)
{
    if ((MAX ? m > best : m < best) || (m == best && bi == kNone)) {
        best = m;
        if (SNAP) {
#pragma unroll
            for (int i = 0; i < 8; ++i)
                st_shared_v4(slot + 512u * i, s[4 * i], s[4 * i + 1], s[4 * i + 2], s[4 * i + 3]);
            bi = j0;
        } else {
            bi = j0 + first_of(s, m);
        }
    }
}

// Turn a 16-value snapshot's start column into the winning column.
__device__ __forceinline__ void resolve_snapshot16(float best, int &bi, uint32_t slot)
{
    if (bi == kNone)
        return;
    float s[16];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float4 q = ld_shared_v4(slot + 512u * i);
        s[4 * i] = q.x;
        s[4 * i + 1] = q.y;
        s[4 * i + 2] = q.z;
        s[4 * i + 3] = q.w;
    }
    int pos = 15;
#pragma unroll
    for (int i = 14; i >= 0; --i)
        pos = (s[i] == best) ? i : pos;
    bi += pos;
}

// Turn a snapshot's chunk start into the winning column.
__device__ __forceinline__ void resolve_snapshot(float best, int &bi, uint32_t slot)
{
    if (bi == kNone)
        return;
    float s[32];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const float4 q = ld_shared_v4(slot + 512u * i);
        s[4 * i] = q.x;
        s[4 * i + 1] = q.y;
        s[4 * i + 2] = q.z;
        s[4 * i + 3] = q.w;
    }
    bi += first_of(s, best);
}

template <int SUB, int NT, int CH, int KB>
__global__ void __launch_bounds__(32 * (4 * SUB * CH + 4), 1)
    assign_kernel(const __grid_constant__ CUtensorMap xmap, const __grid_constant__ CUtensorMap cmap,
                  const AssignParams p)
{
    constexpr int kConsumerWarps = 4 * SUB * CH;
    constexpr int kConsumerThreads = 32 * kConsumerWarps;
    constexpr int kProducerWarp = kConsumerWarps;
    constexpr int kMmaWarp = kConsumerWarps + 1;
    constexpr int kNormWarp = kConsumerWarps + 2;
    constexpr int kXWarp = kConsumerWarps + 3;
    constexpr bool kSnap = KB <= 2;                    // D <= 128: epilogue-bound
    // D <= 128: the norms enter the accumulator through one more MMA step
    // (25% more tensor work at D = 64, 12.5% at D = 128); the accumulator then
    // holds t = x.c - ||c||^2 / 2 = -s / 2, the reduction takes the largest t,
    // and the tensor-memory loads reduce each chunk's maximum themselves.
    // Every kernel folds at exactly these D, so a point's answer does not
    // depend on the plan, the batch or the other points of the call.
    constexpr bool kFold = KB <= 2;
    constexpr uint32_t kNormBytes =
        kFold ? kOnesBytes + kFoldStages * NT * 32u : kCnStages * NT * 4u;
    constexpr int kCW = NT / CH;                       // columns per consumer warp per tile
    constexpr int kChunks = kCW / 32;
    constexpr int kGroup = kChunks < 4 ? kChunks : 4;  // chunks loaded per tcgen05.wait::ld
    constexpr int kGroups = kChunks / kGroup;
    constexpr uint32_t kCStageBytes = NT * 128;
    constexpr uint32_t kXBufBytes = SUB * KB * kXTileBytes;
    constexpr uint32_t kAccCols = SUB * NT;            // columns of one accumulator stage
    constexpr uint32_t kTmemCols = 2 * kAccCols;       // two stages: 256 or 512
    static_assert(kTmemCols <= 512, "accumulators exceed tensor memory");
    static_assert(kCW % 32 == 0 && kChunks % kGroup == 0, "column slice must be whole chunks");

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    const uint32_t x_base = base;
    const uint32_t c_base = x_base + p.xbufs * kXBufBytes;
    const uint32_t cn_base = c_base + p.stages * kCStageBytes;   // norm ring, or fold region
    const uint32_t red_base = cn_base + kNormBytes;               // {float,int}[CH-1][SUB*128]
    const uint32_t snap_base = red_base + (CH - 1) * SUB * kTileM * 8;   // [warp][8][32] float4
    const uint32_t bar_base = snap_base + (kSnap ? kConsumerWarps * 4096u : 0u);
    uint8_t *const sbase = smem_raw + (base - raw);
    uint8_t *misc_ptr = smem_raw + (bar_base - raw) + kNumBars * 8;
    volatile uint32_t *tmem_slot = reinterpret_cast<volatile uint32_t *>(misc_ptr);
    volatile uint32_t *abort_flag = reinterpret_cast<volatile uint32_t *>(misc_ptr + 4);
    // last-unit flags of the split row groups (one per 128-row sub-tile)
    volatile uint32_t *split_flag = reinterpret_cast<volatile uint32_t *>(misc_ptr + 8);
    auto bar = [&](int i) -> uint32_t { return bar_base + 8u * static_cast<uint32_t>(i); };
    if (!debug_layout_ok(p, bar_base - raw + kMiscBytes))
        return;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0)
        init_barriers<kConsumerWarps, kFold>(bar_base, abort_flag);
    if (kFold)
        fold_init<NT>(cn_base);
    if (warp == kMmaWarp) {
        tmem_alloc(smem_addr(const_cast<uint32_t *>(tmem_slot)), kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    if (warp == kProducerWarp) {
        producer_role<SUB, NT, KB>(p, &xmap, &cmap, c_base, bar_base, abort_flag);
    } else if (warp == kXWarp) {
        x_role<SUB, KB>(p, &xmap, x_base, bar_base, abort_flag);
    } else if (warp == kMmaWarp) {
        mma_role<SUB, NT, KB, kFold>(p, x_base, c_base, bar_base, tmem_base, abort_flag, cn_base);
    } else if (warp == kNormWarp) {
        grid_dep_wait();   // the norms may come from the preparation launch
        if (kFold)
            fold_norm_role<SUB, NT>(p, cn_base, bar_base, abort_flag);
        else
            norm_role<SUB, NT>(p, reinterpret_cast<float *>(sbase + (cn_base - base)), bar_base,
                               abort_flag);
    } else {
        grid_dep_wait();   // split rows' keys and counters come from the preparation launch
        // Consumer warp w reads TMEM lanes 32*(w%4) .. +31 of sub-tile
        // (w/4)%SUB, columns [col0, col0 + kCW) of every tile.
        const int q = warp & 3;
        const int t = (warp >> 2) % SUB;
        const int h = warp / (4 * SUB);
        const int col0 = h * kCW;
        const uint32_t cn_col = cn_base + 4u * static_cast<uint32_t>(col0);
        const uint32_t slot = snap_base + 4096u * warp + 16u * lane;
        const float kNaN = __int_as_float(0x7fc00000);
        uint32_t acc_used = 0;
        bool ok = true;

        for (int u = blockIdx.x; u < p.num_units; u += gridDim.x) {
            const Unit w = decode_unit<SUB>(p, u);
            // +inf for scores, -inf for folded t
            float best = __int_as_float(kFold ? 0xff800000 : 0x7f800000);
            int bi = kNone;
            for (int tile = w.t_begin; tile < w.t_end; ++tile, ++acc_used) {
                const uint32_t as = acc_used & 1u;
                const uint32_t aph = (acc_used >> 1) & 1u;
                const uint32_t nb = acc_used % kCnStages;
                const uint32_t nph = (acc_used / kCnStages) & 1u;
                if (ok)
                    ok = wait_warp(bar(kBarAccFull + as), aph, abort_flag, p.timeout_ns);
                if (ok && !kFold)
                    ok = wait_warp(bar(kBarCnFull + nb), nph, abort_flag, p.timeout_ns);
                if (ok) {
                    tc_fence_after();
                    const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                                           as * kAccCols + t * NT + col0;
                    const uint32_t cn_tile = cn_col + 4u * NT * nb;
#pragma unroll
                    for (int g = 0; g < kGroups; ++g) {
                        __syncwarp();   // tcgen05.ld is .sync.aligned
                        float v[kGroup][32];
                        float m[kGroup];
#pragma unroll
                        for (int c = 0; c < kGroup; ++c) {
                            // folded: the load also reduces the chunk's maximum
                            if (kFold)
                                tmem_ld_red_max_32x32b_x32(taddr + (g * kGroup + c) * 32, v[c],
                                                           m[c]);
                            else
                                tmem_ld_32x32b_x32(taddr + (g * kGroup + c) * 32, v[c]);
                        }
                        tmem_wait_ld();
                        if (g == kGroups - 1) {
                            // Scores are in registers: hand the stage back.
                            tc_fence_before();
                            __syncwarp();
                            if (lane == 0)
                                mbar_arrive(bar(kBarAccEmpty + as));
                        }
#pragma unroll
                        for (int c = 0; c < kGroup; ++c) {
                            if (!kFold) {
                                apply_norms(v[c], cn_tile + 128u * (g * kGroup + c));
                                m[c] = chunk_min(v[c]);
                            }
                        }
                        const int jg = tile * NT + col0 + g * kGroup * 32;
#pragma unroll
                        for (int c = 0; c < kGroup; ++c)
                            fold_chunk<kSnap, kFold>(v[c], m[c], jg + 32 * c, best, bi, slot);
                    }
                    if (!kFold) {
                        // This warp is done with the tile's norms.
                        __syncwarp();
                        if (lane == 0)
                            mbar_arrive(bar(kBarCnEmpty + nb));
                    }
                }
            }

            if (kSnap)
                resolve_snapshot(best, bi, slot);
            if (kFold)
                best = -2.0f * best;   // t back to the score s (exact)
            // Merge the column slices of each point: (score, index) order.
            const int lrow = t * kTileM + q * 32 + lane;
            if (CH > 1) {
                float *red_s = reinterpret_cast<float *>(sbase + (red_base - base));
                int *red_i = reinterpret_cast<int *>(red_s + (CH - 1) * SUB * kTileM);
                if (h > 0) {
                    red_s[(h - 1) * SUB * kTileM + lrow] = best;
                    red_i[(h - 1) * SUB * kTileM + lrow] = bi;
                }
                named_bar_sync(kConsumerBarrier, kConsumerThreads);
                if (h == 0) {
#pragma unroll
                    for (int o = 0; o < CH - 1; ++o) {
                        const float b2 = red_s[o * SUB * kTileM + lrow];
                        const int i2 = red_i[o * SUB * kTileM + lrow];
                        if (b2 < best || (b2 == best && i2 < bi)) {
                            best = b2;
                            bi = i2;
                        }
                    }
                }
                // The next unit's winners may not overwrite these before
                // they are read.
                named_bar_sync(kConsumerBarrier, kConsumerThreads);
            }
            const int row = w.row0 + lrow;
            if (h == 0 && t < w.nsub) {
                if (!w.split) {
                    if (ok && row < p.N) {
                        float ms;
                        int ix;
                        if (bi == kNone) {
                            ix = 0;
                            ms = kNaN;
                        } else {
                            ix = bi;
                            ms = (__float_as_uint(best) == 0x80000000u) ? 0.0f : best;
                        }
                        p.idx[row] = ix;
                        if (p.counts != nullptr)
                            atomicAdd(p.counts + ix, 1);
                        if (p.minscore != nullptr)
                            p.minscore[row] = ms;
                    }
                } else {
                    merge_split_group(p, SUB * kTileM, row, ok && row < p.N, best, bi,
                                      kSplitBarrier + t, split_flag + t, q == 0 && lane == 0);
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tmem_base, kTmemCols);
    }
}

// ---------------------------------------------------------------------------
// CTA-pair variant (cta_group::2): a cluster of two CTAs on two SMs computes
// 256x256 tiles.  Each CTA keeps its own 128 X rows resident and loads only
// its 128-row half of every C k-block (16 KiB instead of 32), so L2 traffic
// per flop halves and the ring of stages reaches twice as far ahead for the
// same shared memory.  The leader CTA (rank 0) issues the pair MMAs; their
// completion is multicast to both CTAs' barriers; the peer's copies count on
// the leader's full barriers and its consumers hand accumulator stages back
// by arriving on the leader's empty barriers.  At D <= 128 the pair folds the
// norms into the MMA (one more step per tile, its B operand TMA-loaded from a
// precomputed fold operand like a C k-block); above, a norm ring serves the
// epilogue as in the single-CTA kernel.  The stores are per CTA and identical
// to the single-CTA kernel's.  Folded, the reduction differs in three ways,
// all measured faster and bit-identical:
//   * each 32-column chunk is read as two 16-column reducing loads, and a
//     lane that improves keeps only the 16-value half holding the group's
//     first maximum (4 shared-memory stores instead of 8);
//   * a warp tests its whole column slice of the tile at once: the largest t
//     of the slice against the running best, one vote, and only when some
//     lane improves the search for the first half holding that maximum
//     (the best after the slice is its maximum at its first position);
//   * the column slices of a row publish their running best per tile in
//     shared memory and skip chunks strictly below another slice's best (a
//     stale value only skips less; equal values are still kept, and the
//     slices' merge by (score, index) keeps the lowest index).
template <int CH, int KB>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(32 * (4 * CH + 4), 1)
    assign_pair_kernel(const __grid_constant__ CUtensorMap xmap,
                       const __grid_constant__ CUtensorMap cmap,
                       const __grid_constant__ CUtensorMap fmap, const AssignParams p)
{
    constexpr int NT = 256;                            // centroids per pair tile
    constexpr int kHalf = 128;                         // C rows each CTA loads
    constexpr int kConsumerWarps = 4 * CH;
    constexpr int kProducerWarp = kConsumerWarps;
    constexpr int kMmaWarp = kConsumerWarps + 1;
    constexpr int kNormWarp = kConsumerWarps + 2;
    constexpr int kXWarp = kConsumerWarps + 3;
    // The pair's half-size C stages leave room for the deferred first-index
    // search up to D = 192, where its consumers, not the tensor pipe, set the
    // pace (measured 5-8% faster there; at D = 256 the stages it costs matter
    // more).
    constexpr bool kSnap = KB <= 3;
    // D <= 128: the norms enter the accumulator through one more pair MMA
    // step, A = each CTA's tile of ones, B = each CTA's half of the tile's
    // fold operand (the split -||c||^2 / 2, precomputed in global memory and
    // brought in by TMA like a C k-block, so the copy engine, not a thread's
    // stores, signals the leader).  The consumers then take the largest
    // t = -s / 2.  Here the pair's N = 256 MMAs leave the tensor pipe room
    // for the extra step, and the lighter reduction is what sets the pace.
    constexpr bool kFold = KB <= 2;
    // Folded, one full/empty barrier pair covers a whole tile: its KB C
    // k-block halves and its fold rows.  A tcgen05.commit that completes a
    // barrier phase costs the tensor pipe ~30-45 clocks on GB300 (measured
    // with commits to barriers that do and do not complete a phase), and so
    // does each wait of the issuing thread; per-tile grouping leaves one
    // commit and one wait for the ring where per-k-block barriers and a
    // separate fold ring took KB + 1 of each, against a tile of only 5 or 9
    // MMA steps.  Above D = 128 a tile has 12 or 16 MMA steps and its
    // k-blocks keep a barrier pair each, so that the ring can refill at
    // k-block granularity (pairs of k-blocks per barrier at D = 256 measured
    // 6-17% slower on the long shapes, the ring then holding 4 stages
    // instead of 5).
    constexpr int kGroupKB = kFold ? KB : 1;   // C k-blocks per barrier pair
    constexpr int kCW = NT / CH;
    constexpr int kChunks = kCW / 32;
    constexpr int kGroup = kChunks < 4 ? kChunks : 4;
    constexpr int kGroups = kChunks / kGroup;
    constexpr uint32_t kCStageBytes = kHalf * 128;
    constexpr uint32_t kXBufBytes = KB * kXTileBytes;
    constexpr uint32_t kAccCols = NT;
    constexpr uint32_t kTmemCols = 2 * kAccCols;
    constexpr uint32_t kIdesc = idesc_bf16_f32(2 * kTileM, NT);
    constexpr uint16_t kBoth = 0x3;
    static_assert(kCW % 32 == 0 && kChunks % kGroup == 0, "column slice must be whole chunks");

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    const uint32_t x_base = base;
    const uint32_t c_base = x_base + p.xbufs * kXBufBytes;
    const uint32_t cn_base = c_base + p.stages * kCStageBytes;
    // C stage groups (p.stages is a multiple of kGroupKB)
    const uint32_t ngroups = static_cast<uint32_t>(p.stages / kGroupKB);
    // fold: the ones tile, then one fold slot per stage group; else the norm
    // ring
    const uint32_t norm_bytes =
        kFold ? kOnesBytes + ngroups * kFoldBlockBytes : kCnStages * NT * 4u;
    const uint32_t red_base = cn_base + norm_bytes;
    const uint32_t snap_base = red_base + (CH - 1) * kTileM * 8;
    const uint32_t thr_base = snap_base + (kSnap ? kConsumerWarps * 4096u : 0u);
    const uint32_t bar_base = thr_base + CH * kTileM * 4u;
    uint8_t *const sbase = smem_raw + (base - raw);
    uint8_t *misc_ptr = smem_raw + (bar_base - raw) + kNumBars * 8;
    volatile uint32_t *tmem_slot = reinterpret_cast<volatile uint32_t *>(misc_ptr);
    volatile uint32_t *abort_flag = reinterpret_cast<volatile uint32_t *>(misc_ptr + 4);
    // last-unit flags of the split row groups (one per 128-row sub-tile)
    volatile uint32_t *split_flag = reinterpret_cast<volatile uint32_t *>(misc_ptr + 8);
    auto bar = [&](int i) -> uint32_t { return bar_base + 8u * static_cast<uint32_t>(i); };

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const bool leader = rank == 0;
    // The leader's copy of barrier i, as a cluster address.
    auto lead_bar = [&](int i) -> uint32_t { return map_to_rank(bar(i), 0); };
    if (!debug_layout_ok(p, bar_base - raw + kMiscBytes) ||
        !debug_ok(p.stage_group == kGroupKB && p.stages % kGroupKB == 0))
        return;   // both CTAs of the pair decide alike

    if (threadIdx.x == 0) {
        for (int b = 0; b < kMaxXBufs; ++b) {
            mbar_init(bar(kBarXFull + b), 1);
            mbar_init(bar(kBarXEmpty + b), 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(bar(kBarAccFull + a), 1);
            mbar_init(bar(kBarAccEmpty + a), 2 * kConsumerWarps);
        }
        mbar_init(bar(kBarDrain), 1);
        for (int s = 0; s < kMaxStages; ++s) {
            mbar_init(bar(kBarCFull + s), 1);
            mbar_init(bar(kBarCEmpty + s), 1);
        }
        for (int s = 0; s < kCnStages; ++s) {
            mbar_init(bar(kBarCnFull + s), 32);
            mbar_init(bar(kBarCnEmpty + s), kConsumerWarps);
        }
        *abort_flag = 0u;
        fence_mbar_init();
    }
    if (kFold)
        fold_init<kHalf>(cn_base);   // the ones tile (the slots are overwritten by copies)
    for (int i = threadIdx.x; i < CH * kTileM; i += blockDim.x)
        reinterpret_cast<float *>(sbase + (thr_base - base))[i] = __int_as_float(0xff800000);
    if (warp == kMmaWarp) {
        tmem_alloc_pair(smem_addr(const_cast<uint32_t *>(tmem_slot)), kTmemCols);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync();   // both CTAs' barriers exist before any cross-CTA signal
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    const int cluster = static_cast<int>(blockIdx.x >> 1);
    const int nclusters = static_cast<int>(gridDim.x >> 1);

    if (warp == kProducerWarp) {
        if (kFold)
            grid_dep_wait();   // the fold operand comes from the preparation launch
        if (lane == 0) {
            tma_prefetch_desc(&cmap);
            if (kFold)
                tma_prefetch_desc(&fmap);
            const uint64_t pol_c = policy_evict_last();
            // folded: stage = the stage group, else the stage
            uint32_t stage = 0, phase = 0;
            bool ok = true;
            for (int u = cluster; ok && u < p.num_units; u += nclusters) {
                const Unit w = decode_unit<2>(p, u);
                for (int tile = w.t_begin; ok && tile < w.t_end; ++tile) {
                    if constexpr (kFold) {
                        // The tile's group: its KB k-block halves of C and
                        // this CTA's 128 centroids of the fold operand
                        // (block 2 * tile + rank, 256 rows of 16 bytes), all
                        // counted on one full barrier of the leader.
                        if (!(ok = wait1(bar(kBarCEmpty + stage), phase ^ 1u, abort_flag,
                                         p.timeout_ns)))
                            break;
                        if (leader)
                            mbar_arrive_expect_tx(bar(kBarCFull + stage),
                                                  2 * (KB * kCStageBytes + kFoldBlockBytes));
#pragma unroll
                        for (int kb = 0; kb < KB; ++kb)
                            tma_load_2d_pair(c_base + (stage * KB + kb) * kCStageBytes, &cmap,
                                             lead_bar(kBarCFull + stage), kb * kKBlock,
                                             tile * NT + static_cast<int>(rank) * kHalf, pol_c);
                        tma_load_2d_pair(cn_base + kOnesBytes + stage * kFoldBlockBytes, &fmap,
                                         lead_bar(kBarCFull + stage), 0,
                                         (2 * tile + static_cast<int>(rank)) * 256, pol_c);
                        if (++stage == ngroups) {
                            stage = 0;
                            phase ^= 1u;
                        }
                    } else {
#pragma unroll
                        for (int kb = 0; kb < KB; ++kb) {
                            if (!(ok = wait1(bar(kBarCEmpty + stage), phase ^ 1u, abort_flag,
                                             p.timeout_ns)))
                                break;
                            if (leader)
                                mbar_arrive_expect_tx(bar(kBarCFull + stage), 2 * kCStageBytes);
                            tma_load_2d_pair(c_base + stage * kCStageBytes, &cmap,
                                             lead_bar(kBarCFull + stage), kb * kKBlock,
                                             tile * NT + static_cast<int>(rank) * kHalf, pol_c);
                            if (++stage == static_cast<uint32_t>(p.stages)) {
                                stage = 0;
                                phase ^= 1u;
                            }
                        }
                    }
                }
            }
            if (!ok) {
                // Copies in flight complete on the leader's barriers, out of
                // this CTA's sight: give them time to land (they take
                // microseconds) before the block can exit.
                const uint64_t t0 = globaltimer_ns();
                while (globaltimer_ns() - t0 < 1000000ull) {
                }
            }
        }
        __syncwarp();
    } else if (warp == kXWarp) {
        if (lane == 0) {
            tma_prefetch_desc(&xmap);
            const uint64_t pol_x = policy_evict_first();
            uint32_t x_issued = 0;
            bool ok = true;
            for (int u = cluster; ok && u < p.num_units; u += nclusters) {
                const Unit w = decode_unit<2>(p, u);
                const uint32_t xb = x_issued % p.xbufs;
                const uint32_t xph = (x_issued / p.xbufs) & 1u;
                if (!(ok = wait1(bar(kBarXEmpty + xb), xph ^ 1u, abort_flag, p.timeout_ns)))
                    break;
                // The leader's barrier counts both CTAs' rows (the peer's only
                // when its 128 rows hold points).
                if (leader)
                    mbar_arrive_expect_tx(bar(kBarXFull + xb), w.nsub * KB * kXTileBytes);
                if (static_cast<int>(rank) < w.nsub) {
                    const uint32_t xdst = x_base + xb * kXBufBytes;
#pragma unroll
                    for (int kb = 0; kb < KB; ++kb)
                        tma_load_2d_pair(xdst + kb * kXTileBytes, &xmap, lead_bar(kBarXFull + xb),
                                         kb * kKBlock, w.row0 + static_cast<int>(rank) * kTileM,
                                         pol_x);
                }
                ++x_issued;
            }
            if (!ok) {
                const uint64_t t0 = globaltimer_ns();
                while (globaltimer_ns() - t0 < 1000000ull) {
                }
            }
        }
        __syncwarp();
    } else if (warp == kMmaWarp) {
        if (leader) {
            // folded: stage = the stage group, else the stage
            uint32_t stage = 0, phase = 0, x_used = 0, acc_used = 0;
            bool ok = true, issued = false;
            const uint64_t ones_desc = kFold ? plain_kmajor_desc(cn_base, kFoldLbo, kFoldSbo) : 0;
            for (int u = cluster; ok && u < p.num_units; u += nclusters) {
                const Unit w = decode_unit<2>(p, u);
                const uint32_t xb = x_used % p.xbufs;
                const uint32_t xph = (x_used / p.xbufs) & 1u;
                if (!(ok = wait_warp(bar(kBarXFull + xb), xph, abort_flag, p.timeout_ns)))
                    break;
                uint64_t adesc[KB];
#pragma unroll
                for (int kb = 0; kb < KB; ++kb)
                    adesc[kb] = sw128_kmajor_desc(x_base + xb * kXBufBytes + kb * kXTileBytes);
                for (int tile = w.t_begin; ok && tile < w.t_end; ++tile) {
                    const uint32_t as = acc_used & 1u;
                    const uint32_t aph = (acc_used >> 1) & 1u;
                    if constexpr (kFold) {
                        // Folded tiles are short (5 or 9 MMA steps), so the
                        // accumulator hand-off is on the critical path: wait
                        // for the tile's group first (the copies run tiles
                        // ahead), then for the stage, and issue at once: the
                        // k-steps, the fold step (ones x the group's fold
                        // rows), one commit that frees the group in both
                        // CTAs and one that hands the stage to the consumers.
                        if (!(ok = wait_warp(bar(kBarCFull + stage), phase, abort_flag,
                                             p.timeout_ns)))
                            break;
                        if (!(ok = wait_warp(bar(kBarAccEmpty + as), aph ^ 1u, abort_flag,
                                             p.timeout_ns)))
                            break;
                        tc_fence_after();
                        const uint32_t d_tmem = tmem_base + as * kAccCols;
                        const uint64_t bdesc =
                            plain_kmajor_desc(cn_base + kOnesBytes + stage * kFoldBlockBytes,
                                              kFoldPairLbo, kFoldPairSbo);
                        if (elect_one()) {
#pragma unroll
                            for (int kb = 0; kb < KB; ++kb) {
                                const uint64_t cdesc =
                                    sw128_kmajor_desc(c_base + (stage * KB + kb) * kCStageBytes);
#pragma unroll
                                for (int k = 0; k < 4; ++k)
                                    mma_bf16_pair(d_tmem, adesc[kb] + 2u * k, cdesc + 2u * k,
                                                  kIdesc, (kb | k) != 0);
                            }
                            mma_bf16_pair(d_tmem, ones_desc, bdesc, kIdesc, 1u);
                            mma_commit_pair(bar(kBarCEmpty + stage), kBoth);
                            mma_commit_pair(bar(kBarAccFull + as), kBoth);
                        }
                        __syncwarp();
                        issued = true;
                        if (++stage == ngroups) {
                            stage = 0;
                            phase ^= 1u;
                        }
                        ++acc_used;
                        continue;
                    }
                    if (!(ok = wait_warp(bar(kBarAccEmpty + as), aph ^ 1u, abort_flag,
                                         p.timeout_ns)))
                        break;
                    tc_fence_after();
                    const uint32_t d_tmem = tmem_base + as * kAccCols;
#pragma unroll
                    for (int kb = 0; kb < KB; ++kb) {
                        if (!kFold && !(ok = wait_warp(bar(kBarCFull + stage), phase, abort_flag,
                                                       p.timeout_ns)))
                            break;
                        const uint64_t cdesc = sw128_kmajor_desc(c_base + stage * kCStageBytes);
                        if (elect_one()) {
#pragma unroll
                            for (int k = 0; k < 4; ++k)
                                mma_bf16_pair(d_tmem, adesc[kb] + 2u * k, cdesc + 2u * k, kIdesc,
                                              (kb | k) != 0);
                            mma_commit_pair(bar(kBarCEmpty + stage), kBoth);
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
                    if (elect_one())
                        mma_commit_pair(bar(kBarAccFull + as), kBoth);
                    __syncwarp();
                    ++acc_used;
                }
                if (!ok)
                    break;
                if (elect_one())
                    mma_commit_pair(bar(kBarXEmpty + xb), kBoth);
                __syncwarp();
                ++x_used;
            }
            if (issued) {
                if (elect_one())
                    mma_commit_pair(bar(kBarDrain), 0x1);
                __syncwarp();
                wait_warp(bar(kBarDrain), 0u, abort_flag, kDrainLimitNs, false);
            }
        }
    } else if (warp == kNormWarp) {
        // Folded, the norms come in with the fold operand: nothing to stage.
        if (!kFold)
            grid_dep_wait();   // the norms may come from the preparation launch
        float *const cn_smem = reinterpret_cast<float *>(sbase + (cn_base - base));
        const float kNaN = __int_as_float(0x7fc00000);
        uint32_t n = 0;
        bool ok = true;
        for (int u = cluster; !kFold && ok && u < p.num_units; u += nclusters) {
            const Unit w = decode_unit<2>(p, u);
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
                mbar_arrive(bar(kBarCnFull + b));
            }
        }
    } else {
        grid_dep_wait();   // split rows' keys and counters come from the preparation launch
        // Consumer warp w: TMEM lanes 32*(w%4) .. +31 of this CTA's 128 rows,
        // columns [col0, col0 + kCW) of every 256-column tile.
        const int q = warp & 3;
        const int h = warp >> 2;
        const int col0 = h * kCW;
        const uint32_t cn_col = cn_base + 4u * static_cast<uint32_t>(col0);
        const uint32_t slot = snap_base + 4096u * warp + 16u * lane;
        const float kNaN = __int_as_float(0x7fc00000);
        uint32_t acc_used = 0;
        bool ok = true;
        for (int u = cluster; u < p.num_units; u += nclusters) {
            const Unit w = decode_unit<2>(p, u);
            // +inf for scores, -inf for folded t
            float best = __int_as_float(kFold ? 0xff800000 : 0x7f800000);
            int bi = kNone;
            volatile float *thr = reinterpret_cast<volatile float *>(sbase + (thr_base - base));
            const int trow = q * 32 + lane;
            for (int tile = w.t_begin; tile < w.t_end; ++tile, ++acc_used) {
                const uint32_t as = acc_used & 1u;
                const uint32_t aph = (acc_used >> 1) & 1u;
                const uint32_t nb = acc_used % kCnStages;
                const uint32_t nph = (acc_used / kCnStages) & 1u;
                // the best t the other column slices of these rows have seen
                float other = __int_as_float(0xff800000);
                if (kFold && CH > 1) {
#pragma unroll
                    for (int o = 0; o < CH; ++o)
                        if (o != h)
                            other = fmaxf(other, thr[o * kTileM + trow]);
                }
                if (ok)
                    ok = wait_warp(bar(kBarAccFull + as), aph, abort_flag, p.timeout_ns);
                if (ok && !kFold)
                    ok = wait_warp(bar(kBarCnFull + nb), nph, abort_flag, p.timeout_ns);
                if (ok) {
                    tc_fence_after();
                    const uint32_t taddr =
                        tmem_base + (static_cast<uint32_t>(q * 32) << 16) + as * kAccCols + col0;
                    const uint32_t cn_tile = cn_col + 4u * NT * nb;
#pragma unroll
                    for (int g = 0; g < kGroups; ++g) {
                        __syncwarp();
                        float v[kGroup][32];
                        float m[kGroup];
                        float mh[kGroup];   // folded: maximum of each chunk's second half
#pragma unroll
                        for (int c = 0; c < kGroup; ++c) {
                            if (kFold) {
                                tmem_ld_red_max_32x32b_x16(taddr + (g * kGroup + c) * 32, v[c],
                                                           m[c]);
                                tmem_ld_red_max_32x32b_x16(taddr + (g * kGroup + c) * 32 + 16,
                                                           v[c] + 16, mh[c]);
                            } else {
                                tmem_ld_32x32b_x32(taddr + (g * kGroup + c) * 32, v[c]);
                            }
                        }
                        tmem_wait_ld();
                        if (g == kGroups - 1) {
                            tc_fence_before();
                            __syncwarp();
                            if (lane == 0) {
                                if (leader)
                                    mbar_arrive(bar(kBarAccEmpty + as));
                                else
                                    mbar_arrive_cluster(lead_bar(kBarAccEmpty + as));
                            }
                        }
#pragma unroll
                        for (int c = 0; c < kGroup; ++c) {
                            if (!kFold) {
                                apply_norms(v[c], cn_tile + 128u * (g * kGroup + c));
                                m[c] = chunk_min(v[c]);
                            }
                        }
                        const int jg = tile * NT + col0 + g * kGroup * 32;
                        if (kFold) {
                            // One test for the whole group: its largest t
                            // (NaN only when every value is NaN, which never
                            // improves).  The best after the group is that
                            // maximum at its first position, so only when some
                            // lane improves does the warp look for the first
                            // 16-column half holding it and snapshot that half.
                            float M = max2(m[0], mh[0]);
#pragma unroll
                            for (int c = 1; c < kGroup; ++c)
                                M = max3(M, m[c], mh[c]);
                            const bool imp = ((M > best) || (M == best && bi == kNone)) &&
                                             !(M < other);
                            if (__any_sync(0xffffffffu, imp)) {
                                bool found = !imp;
#pragma unroll
                                for (int c = 0; c < kGroup; ++c) {
#pragma unroll
                                    for (int hf = 0; hf < 2; ++hf) {
                                        const bool st = !found && ((hf ? mh[c] : m[c]) == M);
                                        found = found || st;
#pragma unroll
                                        for (int i = 0; i < 4; ++i)
                                            st_shared_v4_if(st, slot + 512u * i,
                                                            v[c][16 * hf + 4 * i],
                                                            v[c][16 * hf + 4 * i + 1],
                                                            v[c][16 * hf + 4 * i + 2],
                                                            v[c][16 * hf + 4 * i + 3]);
                                        bi = st ? jg + 32 * c + 16 * hf : bi;
                                    }
                                }
                                best = imp ? M : best;
                            }
                        } else {
#pragma unroll
                            for (int c = 0; c < kGroup; ++c)
                                fold_chunk<kSnap, kFold>(v[c], m[c], jg + 32 * c, best, bi, slot);
                        }
                    }
                    if (!kFold) {
                        __syncwarp();
                        if (lane == 0)
                            mbar_arrive(bar(kBarCnEmpty + nb));
                    }
                    if (kFold && CH > 1)
                        thr[h * kTileM + trow] = best;
                }
            }
            if (kFold)
                resolve_snapshot16(best, bi, slot);
            else if (kSnap)
                resolve_snapshot(best, bi, slot);
            if (kFold)
                best = -2.0f * best;   // t back to the score s (exact)
            const int lrow = q * 32 + lane;
            if (CH > 1) {
                float *red_s = reinterpret_cast<float *>(sbase + (red_base - base));
                int *red_i = reinterpret_cast<int *>(red_s + (CH - 1) * kTileM);
                if (h > 0) {
                    red_s[(h - 1) * kTileM + lrow] = best;
                    red_i[(h - 1) * kTileM + lrow] = bi;
                }
                named_bar_sync(kConsumerBarrier, 32 * kConsumerWarps);
                // every slice is done with this unit's thresholds
                reinterpret_cast<volatile float *>(sbase + (thr_base - base))[h * kTileM + lrow] =
                    __int_as_float(0xff800000);
                if (h == 0) {
#pragma unroll
                    for (int o = 0; o < CH - 1; ++o) {
                        const float b2 = red_s[o * kTileM + lrow];
                        const int i2 = red_i[o * kTileM + lrow];
                        if (b2 < best || (b2 == best && i2 < bi)) {
                            best = b2;
                            bi = i2;
                        }
                    }
                }
                named_bar_sync(kConsumerBarrier, 32 * kConsumerWarps);
            }
            const int row = w.row0 + static_cast<int>(rank) * kTileM + lrow;
            if (h == 0 && static_cast<int>(rank) < w.nsub) {
                if (!w.split) {
                    if (ok && row < p.N) {
                        float ms;
                        int ix;
                        if (bi == kNone) {
                            ix = 0;
                            ms = kNaN;
                        } else {
                            ix = bi;
                            ms = (__float_as_uint(best) == 0x80000000u) ? 0.0f : best;
                        }
                        p.idx[row] = ix;
                        if (p.counts != nullptr)
                            atomicAdd(p.counts + ix, 1);
                        if (p.minscore != nullptr)
                            p.minscore[row] = ms;
                    }
                } else {
                    merge_split_group(p, 2 * kTileM, row, ok && row < p.N, best, bi,
                                      kSplitBarrier, split_flag, q == 0 && lane == 0);
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    cluster_sync();   // no CTA leaves while its pair can still touch its memory
    if (warp == kMmaWarp) {
        tc_fence_after();
        tmem_dealloc_pair(tmem_base, kTmemCols);
    }
}

template <int CH, int KB>
cudaError_t prepare_pair(size_t smem)
{
    return cudaFuncSetAttribute(assign_pair_kernel<CH, KB>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
}

// Launch configuration; after_prep makes the launch the programmatic
// dependent of the preparation kernel just before it in the stream.
struct LaunchCfg {
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    LaunchCfg(int grid, int threads, size_t smem, cudaStream_t stream, bool after_prep)
    {
        cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
        cfg.blockDim = dim3(static_cast<unsigned>(threads), 1, 1);
        cfg.dynamicSmemBytes = smem;
        cfg.stream = stream;
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = after_prep ? 1 : 0;
    }
};

template <int CH, int KB>
cudaError_t launch_pair(const AssignParams &p, const CUtensorMap &xmap, const CUtensorMap &cmap,
                        const CUtensorMap &fmap, int grid, size_t smem, cudaStream_t stream,
                        bool after_prep)
{
    LaunchCfg lc(grid, 32 * (4 * CH + 4), smem, stream, after_prep);
    return cudaLaunchKernelEx(&lc.cfg, assign_pair_kernel<CH, KB>, xmap, cmap, fmap, p);
}

template <int CH>
cudaError_t dispatch_pair_kb(bool prepare, int kb, const AssignParams *p, const CUtensorMap *xmap,
                             const CUtensorMap *cmap, const CUtensorMap *fmap, int grid,
                             size_t smem, cudaStream_t stream, bool after_prep)
{
    switch (kb) {
    case 1:
        return prepare ? prepare_pair<CH, 1>(smem)
                       : launch_pair<CH, 1>(*p, *xmap, *cmap, *fmap, grid, smem, stream,
                                                after_prep);
    case 2:
        return prepare ? prepare_pair<CH, 2>(smem)
                       : launch_pair<CH, 2>(*p, *xmap, *cmap, *fmap, grid, smem, stream,
                                                after_prep);
    case 3:
        return prepare ? prepare_pair<CH, 3>(smem)
                       : launch_pair<CH, 3>(*p, *xmap, *cmap, *fmap, grid, smem, stream,
                                                after_prep);
    case 4:
        return prepare ? prepare_pair<CH, 4>(smem)
                       : launch_pair<CH, 4>(*p, *xmap, *cmap, *fmap, grid, smem, stream,
                                                after_prep);
    default:
        return cudaErrorInvalidValue;
    }
}

template <int SUB, int NT, int CH, int KB>
cudaError_t prepare_one(size_t smem)
{
    return cudaFuncSetAttribute(assign_kernel<SUB, NT, CH, KB>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
}

template <int SUB, int NT, int CH, int KB>
cudaError_t launch_one(const AssignParams &p, const CUtensorMap &xmap, const CUtensorMap &cmap,
                       int grid, size_t smem, cudaStream_t stream, bool after_prep)
{
    LaunchCfg lc(grid, 32 * (4 * SUB * CH + 4), smem, stream, after_prep);
    return cudaLaunchKernelEx(&lc.cfg, assign_kernel<SUB, NT, CH, KB>, xmap, cmap, p);
}

template <int SUB, int NT, int CH>
cudaError_t dispatch_kb(bool prepare, int kb, const AssignParams *p, const CUtensorMap *xmap,
                        const CUtensorMap *cmap, int grid, size_t smem, cudaStream_t stream,
                        bool after_prep)
{
    switch (kb) {
    case 1:
        return prepare ? prepare_one<SUB, NT, CH, 1>(smem)
                       : launch_one<SUB, NT, CH, 1>(*p, *xmap, *cmap, grid, smem, stream,
                                                       after_prep);
    case 2:
        return prepare ? prepare_one<SUB, NT, CH, 2>(smem)
                       : launch_one<SUB, NT, CH, 2>(*p, *xmap, *cmap, grid, smem, stream,
                                                       after_prep);
    case 3:
        return prepare ? prepare_one<SUB, NT, CH, 3>(smem)
                       : launch_one<SUB, NT, CH, 3>(*p, *xmap, *cmap, grid, smem, stream,
                                                       after_prep);
    case 4:
        return prepare ? prepare_one<SUB, NT, CH, 4>(smem)
                       : launch_one<SUB, NT, CH, 4>(*p, *xmap, *cmap, grid, smem, stream,
                                                       after_prep);
    default:
        return cudaErrorInvalidValue;
    }
}

cudaError_t dispatch(bool prepare, const Variant &v, int kb, const AssignParams *p,
                     const CUtensorMap *xmap, const CUtensorMap *cmap, const CUtensorMap *fmap,
                     int grid, size_t smem, cudaStream_t stream, bool after_prep)
{
    if (v.pair) {
        if (v.ch == 2)
            return dispatch_pair_kb<2>(prepare, kb, p, xmap, cmap, fmap, grid, smem, stream,
                                       after_prep);
        if (v.ch == 4)
            return dispatch_pair_kb<4>(prepare, kb, p, xmap, cmap, fmap, grid, smem, stream,
                                       after_prep);
        return cudaErrorInvalidValue;
    }
    if (v.sub == 1 && v.nt == 128 && v.ch == 1)
        return dispatch_kb<1, 128, 1>(prepare, kb, p, xmap, cmap, grid, smem, stream,
                                          after_prep);
    if (v.sub == 1 && v.nt == 256 && v.ch == 2)
        return dispatch_kb<1, 256, 2>(prepare, kb, p, xmap, cmap, grid, smem, stream,
                                          after_prep);
    if (v.sub == 2 && v.nt == 128 && v.ch == 1)
        return dispatch_kb<2, 128, 1>(prepare, kb, p, xmap, cmap, grid, smem, stream,
                                          after_prep);
    if (v.sub == 2 && v.nt == 128 && v.ch == 2)
        return dispatch_kb<2, 128, 2>(prepare, kb, p, xmap, cmap, grid, smem, stream,
                                          after_prep);
    if (v.sub == 1 && v.nt == 256 && v.ch == 4)
        return dispatch_kb<1, 256, 4>(prepare, kb, p, xmap, cmap, grid, smem, stream,
                                          after_prep);
    return cudaErrorInvalidValue;
}

}  // namespace

const Variant kVariants[kNumVariants] = {{2, 128, 1, false}, {1, 256, 2, false},
                                         {1, 128, 1, false}, {2, 128, 2, false},
                                         {1, 256, 4, false}, {1, 256, 2, true},
                                         {1, 256, 4, true}};

int assign_stage_group(const Variant &v, int kblocks)
{
    return v.pair && assign_folds(v, kblocks) ? kblocks : 1;
}

size_t assign_smem_bytes(const Variant &v, int kblocks, int stages, int xbufs)
{
    const size_t stage_rows = v.pair ? v.nt / 2 : v.nt;
    const bool fold = assign_folds(v, kblocks);   // the kernels' kFold
    // a folding pair: one fold slot per stage group (one tile's stages)
    const size_t fold_slots =
        v.pair ? static_cast<size_t>(stages / assign_stage_group(v, kblocks)) : kFoldStages;
    const size_t fold_slot = v.pair ? kFoldBlockBytes : static_cast<size_t>(v.nt) * 32;
    const size_t norm_bytes =
        fold ? kOnesBytes + fold_slots * fold_slot : kCnStages * v.nt * 4;
    return 1024 + static_cast<size_t>(xbufs) * v.sub * kblocks * kXTileBytes +
           static_cast<size_t>(stages) * stage_rows * 128 + norm_bytes +
           static_cast<size_t>(v.ch - 1) * v.sub * kTileM * 8 +
           (kblocks <= 2 || (v.pair && kblocks <= 3) ? static_cast<size_t>(4 * v.sub * v.ch) * 4096
                                                      : 0) +
           (v.pair ? static_cast<size_t>(v.ch) * kTileM * 4 : 0) + kMiscBytes;
}

cudaError_t assign_prepare(const Variant &v, int kblocks, size_t smem)
{
    return dispatch(true, v, kblocks, nullptr, nullptr, nullptr, nullptr, 0, smem, nullptr, false);
}

cudaError_t launch_assign(const Variant &v, int kblocks, const AssignParams &p,
                          const CUtensorMap &xmap, const CUtensorMap &cmap,
                          const CUtensorMap &fmap, int grid, size_t smem, cudaStream_t stream,
                          bool after_prep)
{
    return dispatch(false, v, kblocks, &p, &xmap, &cmap, &fmap, grid, smem, stream, after_prep);
}

cudaError_t assign_max_clusters(const Variant &v, int kblocks, size_t smem, int *clusters)
{
    if (kblocks < 1 || kblocks > 4)
        return cudaErrorInvalidValue;
    const void *fn = nullptr;
    if (v.ch == 2) {
        const void *t[4] = {(const void *)assign_pair_kernel<2, 1>,
                            (const void *)assign_pair_kernel<2, 2>,
                            (const void *)assign_pair_kernel<2, 3>,
                            (const void *)assign_pair_kernel<2, 4>};
        fn = t[kblocks - 1];
    } else {
        const void *t[4] = {(const void *)assign_pair_kernel<4, 1>,
                            (const void *)assign_pair_kernel<4, 2>,
                            (const void *)assign_pair_kernel<4, 3>,
                            (const void *)assign_pair_kernel<4, 4>};
        fn = t[kblocks - 1];
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2, 1, 1);
    cfg.blockDim = dim3(32 * (4 * v.ch + 4), 1, 1);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = 2;
    attr.val.clusterDim.y = 1;
    attr.val.clusterDim.z = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    return cudaOccupancyMaxActiveClusters(clusters, fn, &cfg);
}

bool assign_folds(const Variant &, int kblocks)
{
    return kblocks <= 2;
}

int64_t fold_operand_blocks(int64_t K)
{
    return (K + 255) / 256 * 2;
}

size_t split_counter_offset(int64_t n_split)
{
    return static_cast<size_t>(n_split) * 8;
}

size_t split_scratch_bytes(int64_t n_split)
{
    const size_t groups = static_cast<size_t>((n_split + kTileM - 1) / kTileM);
    return (split_counter_offset(n_split) + groups * 4 + 15) / 16 * 16;
}

size_t fold_operand_bytes(int64_t K)
{
    return static_cast<size_t>(fold_operand_blocks(K)) * kFoldBlockBytes;
}

cudaError_t status_read_and_clear(int *code)
{
    int zero = 0;
    cudaError_t e = cudaMemcpyFromSymbol(code, g_status_word, sizeof(int));
    if (e != cudaSuccess)
        return e;
    return cudaMemcpyToSymbol(g_status_word, &zero, sizeof(int));
}

}  // namespace kma
