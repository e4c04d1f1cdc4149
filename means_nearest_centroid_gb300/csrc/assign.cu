// assign.cu -- the warp-specialised k-means assignment kernel for sm_103a.
//
// What it computes (flashlib PR #22 "Optimize Blackwell k-means assignment
// reduction", Summary and Key ideas): for each point, the score tile
// X . C^T is produced by the tensor cores into tensor memory, the centroid
// norms are applied (s = ||c||^2 - 2 x.c) and the winning centroid is
// selected with lowest-index tie breaking.
//
// Roles inside one thread block (one block per SM, persistent):
//   * producer warp  - TMA-loads the block's X tile once per work unit (the
//                      tile stays resident while centroids stream past it)
//                      and streams C k-blocks through a ring of shared-memory
//                      stages guarded by full/empty mbarriers;
//   * MMA warp       - one thread issues tcgen05.mma (bf16 in, fp32 out) into
//                      one of two tensor-memory accumulator stages and
//                      commits completion to mbarriers;
//   * consumer warps - 4 per 128-point sub-tile, one point per thread: load
//                      the scores with tcgen05.ld, wait for the loads, hand
//                      the accumulator stage back (the fenced-load pattern of
//                      the Key ideas table), then apply the norms and reduce.
//
// The reduction works on 32-column chunks: s = fmaf(-2, acc, cnorm) for the
// chunk (two lanes per packed fma), the chunk minimum by a 3-input min tree
// (NaN ignored), and only when that minimum beats the running best the first
// column holding it is searched.  Scanning chunks in increasing centroid
// order keeps the lowest index on ties; a NaN score never wins.
//
// A work unit is (row tile, centroid range).  When the centroid axis is
// split, partial winners meet in a 64-bit atomicMin on keys holding the
// order-preserving score bits above the centroid index, which keeps the
// result deterministic and the lowest index on ties.
//
// Every mbarrier wait is bounded by p.timeout_ns of %globaltimer.  A wait that
// runs out records KMASSIGN_ERR_TIMEOUT in the status word and raises a
// block-wide abort flag; all roles then leave their loops, the producer waits
// (again bounded) for its copies in flight, the MMA thread waits for its MMAs,
// and the tensor memory is freed before the block returns.
#include "internal.h"
#include "ptx.cuh"

#include "../../include/kmassign.h"

namespace kma {

__device__ int g_status_word = 0;

namespace {

// Barrier slots (8 bytes each) after the operand buffers.
constexpr int kBarXFull = 0;                       // [kMaxXBufs]
constexpr int kBarXEmpty = kBarXFull + kMaxXBufs;  // [kMaxXBufs]
constexpr int kBarAccFull = kBarXEmpty + kMaxXBufs;   // [2]
constexpr int kBarAccEmpty = kBarAccFull + 2;         // [2]
constexpr int kBarDrain = kBarAccEmpty + 2;           // [1]
constexpr int kBarCFull = kBarDrain + 1;              // [kMaxStages]
constexpr int kBarCEmpty = kBarCFull + kMaxStages;    // [kMaxStages]
constexpr int kNumBars = kBarCEmpty + kMaxStages;
constexpr uint32_t kMiscBytes = kNumBars * 8 + 16;   // + tmem slot + abort flag

__device__ __forceinline__ void record_timeout()
{
    atomicCAS(&g_status_word, 0, static_cast<int>(KMASSIGN_ERR_TIMEOUT));
}

// Single-thread bounded wait.  Returns false on timeout or block abort.
__device__ __noinline__ bool wait1(uint32_t bar, uint32_t parity, volatile uint32_t *abort_flag,
                                   uint64_t limit_ns, bool honour_abort)
{
    if (mbar_try_wait(bar, parity))
        return true;
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

// Whole-warp bounded wait; the decision is uniform across the warp.
__device__ __forceinline__ bool wait_warp(uint32_t bar, uint32_t parity,
                                          volatile uint32_t *abort_flag, uint64_t limit_ns,
                                          int lane)
{
    uint64_t t0 = 0;
    bool started = false;
    while (true) {
        const bool done = mbar_try_wait(bar, parity);
        if (__all_sync(0xffffffffu, done))
            return true;
        int give_up = 0;
        if (lane == 0) {
            const uint64_t now = globaltimer_ns();
            if (!started) {
                t0 = now;
                started = true;
            }
            if (*abort_flag) {
                give_up = 1;
            } else if (now - t0 > limit_ns) {
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
};

template <int SUB>
__device__ __forceinline__ Unit decode_unit(const AssignParams &p, int u)
{
    Unit w;
    const int rt = u / p.ksplit;
    const int kc = u - rt * p.ksplit;
    w.row0 = rt * SUB * kTileM;
    const int left = p.N - w.row0;
    w.nsub = min(SUB, (left + kTileM - 1) / kTileM);
    w.t_begin = kc * p.chunk_tiles;
    w.t_end = min(p.ntiles, w.t_begin + p.chunk_tiles);
    return w;
}

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

// One 32-column chunk of one point's scores: fold into (best, bi).
__device__ __forceinline__ void reduce_chunk(const float (&acc)[32], const AssignParams &p, int j0,
                                             float &best, int &bi)
{
    float cn[32];
    if (j0 + 32 <= p.K) {
        const float4 *src = reinterpret_cast<const float4 *>(p.cnorm + j0);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float4 q = __ldg(src + i);
            cn[4 * i + 0] = q.x;
            cn[4 * i + 1] = q.y;
            cn[4 * i + 2] = q.z;
            cn[4 * i + 3] = q.w;
        }
    } else {
        // columns past K: a NaN norm makes a NaN score, which never wins
#pragma unroll
        for (int i = 0; i < 32; ++i)
            cn[i] = (j0 + i < p.K) ? __ldg(p.cnorm + j0 + i) : __int_as_float(0x7fc00000);
    }
    float s[32];
#pragma unroll
    for (int i = 0; i < 32; i += 2)
        fma2(s[i], s[i + 1], -2.0f, -2.0f, acc[i], acc[i + 1], cn[i], cn[i + 1]);
    float a[11];
#pragma unroll
    for (int i = 0; i < 10; ++i)
        a[i] = min3(s[3 * i], s[3 * i + 1], s[3 * i + 2]);
    a[10] = min2(s[30], s[31]);
    const float b0 = min3(a[0], a[1], a[2]);
    const float b1 = min3(a[3], a[4], a[5]);
    const float b2 = min3(a[6], a[7], a[8]);
    const float b3 = min2(a[9], a[10]);
    const float m = min3(b0, b1, min2(b2, b3));
    if (m < best || (m == best && bi == kNone)) {
        int pos = 31;
#pragma unroll
        for (int i = 30; i >= 0; --i)
            pos = (s[i] == m) ? i : pos;
        best = m;
        bi = j0 + pos;
    }
}

template <int SUB, int NT>
__global__ void __launch_bounds__(32 * (4 * SUB + 2), 1)
    assign_kernel(const __grid_constant__ CUtensorMap xmap, const __grid_constant__ CUtensorMap cmap,
                  const AssignParams p)
{
    constexpr int kConsumerWarps = 4 * SUB;
    constexpr int kProducerWarp = kConsumerWarps;
    constexpr int kMmaWarp = kConsumerWarps + 1;
    constexpr uint32_t kCStageBytes = NT * 128;
    constexpr uint32_t kAccCols = SUB * NT;        // columns of one accumulator stage
    constexpr uint32_t kTmemCols = 2 * kAccCols;   // two stages: 256 or 512
    constexpr uint32_t kIdesc = idesc_bf16_f32(kTileM, NT);
    static_assert(kTmemCols <= 512, "accumulators exceed tensor memory");
    static_assert(NT % 128 == 0, "consumer groups read 128 columns at a time");

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    const uint32_t x_buf_bytes = SUB * p.kblocks * kXTileBytes;
    const uint32_t x_base = base;
    const uint32_t c_base = x_base + p.xbufs * x_buf_bytes;
    const uint32_t bar_base = c_base + p.stages * kCStageBytes;
    uint8_t *misc_ptr = smem_raw + (bar_base - raw) + kNumBars * 8;
    volatile uint32_t *tmem_slot = reinterpret_cast<volatile uint32_t *>(misc_ptr);
    volatile uint32_t *abort_flag = reinterpret_cast<volatile uint32_t *>(misc_ptr + 4);
    auto bar = [&](int i) -> uint32_t { return bar_base + 8u * static_cast<uint32_t>(i); };

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
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
        *abort_flag = 0u;
        fence_mbar_init();
    }
    if (warp == kMmaWarp) {
        tmem_alloc(smem_addr(const_cast<uint32_t *>(tmem_slot)), kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    if (warp == kProducerWarp) {
        if (lane == 0) {
            tma_prefetch_desc(&xmap);
            tma_prefetch_desc(&cmap);
            const uint64_t pol_x = policy_evict_first();
            const uint64_t pol_c = policy_evict_last();
            uint32_t stage = 0, phase = 0;
            uint32_t c_issued = 0, x_issued = 0;
            bool ok = true;
            for (int u = blockIdx.x; ok && u < p.num_units; u += gridDim.x) {
                const Unit w = decode_unit<SUB>(p, u);
                const uint32_t xb = x_issued % p.xbufs;
                const uint32_t xph = (x_issued / p.xbufs) & 1u;
                if (!(ok = wait1(bar(kBarXEmpty + xb), xph ^ 1u, abort_flag, p.timeout_ns, true)))
                    break;
                mbar_arrive_expect_tx(bar(kBarXFull + xb), w.nsub * p.kblocks * kXTileBytes);
                const uint32_t xdst = x_base + xb * x_buf_bytes;
                for (int t = 0; t < w.nsub; ++t)
                    for (int kb = 0; kb < p.kblocks; ++kb)
                        tma_load_2d(xdst + (t * p.kblocks + kb) * kXTileBytes, &xmap,
                                    bar(kBarXFull + xb), kb * kKBlock, w.row0 + t * kTileM, pol_x);
                ++x_issued;
                for (int tile = w.t_begin; ok && tile < w.t_end; ++tile) {
                    for (int kb = 0; kb < p.kblocks; ++kb) {
                        if (!(ok = wait1(bar(kBarCEmpty + stage), phase ^ 1u, abort_flag,
                                         p.timeout_ns, true)))
                            break;
                        mbar_arrive_expect_tx(bar(kBarCFull + stage), kCStageBytes);
                        tma_load_2d(c_base + stage * kCStageBytes, &cmap, bar(kBarCFull + stage),
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
                    wait1(bar(kBarCFull + n % S), (n / S) & 1u, abort_flag, p.timeout_ns, false);
                const uint32_t B = p.xbufs;
                for (uint32_t n = (x_issued > B ? x_issued - B : 0); n < x_issued; ++n)
                    wait1(bar(kBarXFull + n % B), (n / B) & 1u, abort_flag, p.timeout_ns, false);
            }
        }
        __syncwarp();
    } else if (warp == kMmaWarp) {
        if (lane == 0) {
            uint32_t stage = 0, phase = 0, x_used = 0, acc_used = 0;
            bool ok = true, issued = false;
            for (int u = blockIdx.x; ok && u < p.num_units; u += gridDim.x) {
                const Unit w = decode_unit<SUB>(p, u);
                const uint32_t xb = x_used % p.xbufs;
                const uint32_t xph = (x_used / p.xbufs) & 1u;
                if (!(ok = wait1(bar(kBarXFull + xb), xph, abort_flag, p.timeout_ns, true)))
                    break;
                tc_fence_after();
                const uint32_t xsrc = x_base + xb * x_buf_bytes;
                for (int tile = w.t_begin; ok && tile < w.t_end; ++tile) {
                    const uint32_t as = acc_used & 1u;
                    const uint32_t aph = (acc_used >> 1) & 1u;
                    if (!(ok = wait1(bar(kBarAccEmpty + as), aph ^ 1u, abort_flag, p.timeout_ns, true)))
                        break;
                    tc_fence_after();
                    const uint32_t d_tmem = tmem_base + as * kAccCols;
                    for (int kb = 0; kb < p.kblocks; ++kb) {
                        if (!(ok = wait1(bar(kBarCFull + stage), phase, abort_flag, p.timeout_ns,
                                         true)))
                            break;
                        tc_fence_after();
                        const uint64_t cdesc = sw128_kmajor_desc(c_base + stage * kCStageBytes);
                        const int kk = min(4, p.ksteps - kb * 4);
                        for (int k = 0; k < kk; ++k) {
                            for (int t = 0; t < w.nsub; ++t) {
                                const uint64_t adesc =
                                    sw128_kmajor_desc(xsrc + (t * p.kblocks + kb) * kXTileBytes);
                                mma_bf16(d_tmem + t * NT, adesc + 2u * k, cdesc + 2u * k, kIdesc,
                                         (kb | k) != 0);
                            }
                        }
                        issued = true;
                        mma_commit(bar(kBarCEmpty + stage));
                        if (++stage == static_cast<uint32_t>(p.stages)) {
                            stage = 0;
                            phase ^= 1u;
                        }
                    }
                    if (!ok)
                        break;
                    mma_commit(bar(kBarAccFull + as));
                    ++acc_used;
                }
                if (!ok)
                    break;
                mma_commit(bar(kBarXEmpty + xb));
                ++x_used;
            }
            if (issued) {
                // All MMAs (and the arrivals they signal) finish before teardown.
                mma_commit(bar(kBarDrain));
                wait1(bar(kBarDrain), 0u, abort_flag, p.timeout_ns, false);
            }
        }
        __syncwarp();
    } else {
        // Consumer warps: warp w reads TMEM lanes 32*(w%4) .. +31 of sub-tile w/4.
        const int t = warp >> 2;
        const int q = warp & 3;
        uint32_t acc_used = 0;
        for (int u = blockIdx.x; u < p.num_units; u += gridDim.x) {
            const Unit w = decode_unit<SUB>(p, u);
            float best = __int_as_float(0x7f800000);   // +inf
            int bi = kNone;
            bool ok = true;
            for (int tile = w.t_begin; tile < w.t_end; ++tile) {
                const uint32_t as = acc_used & 1u;
                const uint32_t aph = (acc_used >> 1) & 1u;
                if (!(ok = wait_warp(bar(kBarAccFull + as), aph, abort_flag, p.timeout_ns, lane)))
                    break;
                tc_fence_after();
                const uint32_t taddr =
                    tmem_base + (static_cast<uint32_t>(q * 32) << 16) + as * kAccCols + t * NT;
#pragma unroll
                for (int g = 0; g < NT / 128; ++g) {
                    __syncwarp();   // tcgen05.ld is .sync.aligned: the warp must be converged
                    float v0[32], v1[32], v2[32], v3[32];
                    tmem_ld_32x32b_x32(taddr + g * 128 + 0, v0);
                    tmem_ld_32x32b_x32(taddr + g * 128 + 32, v1);
                    tmem_ld_32x32b_x32(taddr + g * 128 + 64, v2);
                    tmem_ld_32x32b_x32(taddr + g * 128 + 96, v3);
                    tmem_wait_ld();
                    if (g == NT / 128 - 1) {
                        // Scores are in registers: hand the stage back to the MMA warp.
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0)
                            mbar_arrive(bar(kBarAccEmpty + as));
                    }
                    const int j0 = tile * NT + g * 128;
                    reduce_chunk(v0, p, j0 + 0, best, bi);
                    reduce_chunk(v1, p, j0 + 32, best, bi);
                    reduce_chunk(v2, p, j0 + 64, best, bi);
                    reduce_chunk(v3, p, j0 + 96, best, bi);
                }
                ++acc_used;
            }
            if (!ok)
                break;
            const int row = w.row0 + t * kTileM + q * 32 + lane;
            if (t < w.nsub && row < p.N) {
                if (p.keys == nullptr) {
                    float ms;
                    int ix;
                    if (bi == kNone) {
                        ix = 0;
                        ms = __int_as_float(0x7fc00000);
                    } else {
                        ix = bi;
                        ms = (__float_as_uint(best) == 0x80000000u) ? 0.0f : best;
                    }
                    p.idx[row] = ix;
                    if (p.minscore != nullptr)
                        p.minscore[row] = ms;
                } else if (bi != kNone) {
                    atomicMin(p.keys + row, pack_key(best, bi));
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

template <int SUB, int NT>
cudaError_t prepare_one(size_t smem)
{
    return cudaFuncSetAttribute(assign_kernel<SUB, NT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                static_cast<int>(smem));
}

template <int SUB, int NT>
cudaError_t launch_one(const AssignParams &p, const CUtensorMap &xmap, const CUtensorMap &cmap,
                       int grid, size_t smem, cudaStream_t stream)
{
    assign_kernel<SUB, NT><<<grid, 32 * (4 * SUB + 2), smem, stream>>>(xmap, cmap, p);
    return cudaGetLastError();
}

}  // namespace

size_t assign_smem_bytes(int sub, int nt, int kblocks, int stages, int xbufs)
{
    return 1024 + static_cast<size_t>(xbufs) * sub * kblocks * kXTileBytes +
           static_cast<size_t>(stages) * nt * 128 + kMiscBytes;
}

cudaError_t assign_prepare(int sub, int nt, size_t smem)
{
    if (sub == 1 && nt == 128)
        return prepare_one<1, 128>(smem);
    if (sub == 1 && nt == 256)
        return prepare_one<1, 256>(smem);
    if (sub == 2 && nt == 128)
        return prepare_one<2, 128>(smem);
    return cudaErrorInvalidValue;
}

cudaError_t launch_assign(int sub, int nt, const AssignParams &p, const CUtensorMap &xmap,
                          const CUtensorMap &cmap, int grid, size_t smem, cudaStream_t stream)
{
    if (sub == 1 && nt == 128)
        return launch_one<1, 128>(p, xmap, cmap, grid, smem, stream);
    if (sub == 1 && nt == 256)
        return launch_one<1, 256>(p, xmap, cmap, grid, smem, stream);
    if (sub == 2 && nt == 128)
        return launch_one<2, 128>(p, xmap, cmap, grid, smem, stream);
    return cudaErrorInvalidValue;
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
