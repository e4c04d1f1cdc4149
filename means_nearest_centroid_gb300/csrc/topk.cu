// topk.cu -- the k nearest centroids of every point, and optionally the true
// squared distances to them.
//
// Not part of flashlib PR #22 "Optimize Blackwell k-means assignment
// reduction", which selects one winner per point; this widens its Summary's
// selection step to the k best (score, index) pairs under the same order:
// s_ij = ||c_j||^2 - 2 x_i.c_j ascending, NaN above every number, -0 equal to
// +0, the lower index first among equal scores.  k = 1 gives the assignment.
// The squared distance is ||x_i||^2 + s_ij (fp32, negative rounding results
// clamped to 0), with ||x_i||^2 from the norm kernel.
//
// The score tiles come from the same pipeline as the assignment (pipeline.cuh:
// X warp, C producer, MMA warp, norm warp), in the 256-point x 128-centroid
// shape with one column slice, so each consumer thread owns one point and
// sees every centroid in increasing order.  The consumer keeps that point's
// best L >= k candidates in registers as a sorted list of (ordered score bits,
// index) pairs:
//   * a 32-column chunk whose minimum does not beat the list's last entry is
//     dropped after the same few instructions the assignment spends on it;
//   * otherwise a bit mask marks the chunk's columns below that bound, and
//     each marked column goes through an insertion network (L compare-selects,
//     no memory traffic); since a thread's columns arrive in increasing index
//     order, a new column only displaces entries with strictly larger scores.
// The expected number of insertions for scores in random order is about
// L (1 + ln(K / L)), so for large K nearly all chunks take the cheap path.
//
// Split centroid ranges (few row tiles, or the last partial wave) write each
// unit's sorted list to a buffer of packed 64-bit keys (ordered score << 32 |
// index); a merge kernel then takes, per point, the k smallest keys over the
// ranges with one warp per point.
#include "pipeline.cuh"

namespace kma {
namespace {

constexpr int kTopSub = 2;                       // 256 points per block
constexpr int kTopNt = 128;                      // centroids per tile
constexpr int kTopConsumerWarps = 4 * kTopSub;   // one point per thread
constexpr uint32_t kEmpty = 0xffffffffu;         // ordered value of an unused slot
constexpr uint32_t kNaNOrd = 0xfffffffeu;        // ordered value of every NaN score

// fp32 score -> unsigned value with the same order (NaN above every number,
// -0 folded onto +0).
__device__ __forceinline__ uint32_t ord_of(float s)
{
    if (s != s)
        return kNaNOrd;
    uint32_t u = __float_as_uint(s);
    if (u == 0x80000000u)
        u = 0u;
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float of_ord(uint32_t o)
{
    if (o >= kNaNOrd)
        return __int_as_float(0x7fc00000);
    return __uint_as_float((o & 0x80000000u) ? (o & 0x7fffffffu) : ~o);
}

// The value written for one result: the score, or the squared distance
// ||x||^2 + s with a negative rounding result clamped to 0 (NaN stays NaN).
__device__ __forceinline__ float finish_score(uint32_t o, float xn, bool distances)
{
    const float s = of_ord(o);
    if (!distances)
        return s;
    const float d = xn + s;
    return d < 0.0f ? 0.0f : d;
}

// One 32-bit shared-memory load.
__device__ __forceinline__ float lds_f32(uint32_t addr)
{
    float v;
    asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
    return v;
}

// A sorted list (ascending by ordered score, then index) of the best L
// candidates seen, in registers.
template <int L>
struct TopList {
    uint32_t o[L];
    int32_t j[L];

    __device__ __forceinline__ void clear()
    {
#pragma unroll
        for (int i = 0; i < L; ++i) {
            o[i] = kEmpty;
            j[i] = kNone;
        }
    }

    // Insert (u, jj) where jj is larger than every index in the list: it goes
    // after every entry whose score is not larger.
    __device__ __forceinline__ void push_later(uint32_t u, int32_t jj)
    {
#pragma unroll
        for (int i = L - 1; i > 0; --i) {
            const bool above = u < o[i - 1];
            const bool here = u < o[i];
            j[i] = above ? j[i - 1] : (here ? jj : j[i]);
            o[i] = above ? o[i - 1] : (here ? u : o[i]);
        }
        if (u < o[0]) {
            o[0] = u;
            j[0] = jj;
        }
    }

    // Insert (u, jj) under the full (score, index) order.
    __device__ __forceinline__ void push(uint32_t u, int32_t jj)
    {
        bool below_prev = u < o[L - 1] || (u == o[L - 1] && jj < j[L - 1]);
#pragma unroll
        for (int i = L - 1; i > 0; --i) {
            const bool here = below_prev;
            const bool above = u < o[i - 1] || (u == o[i - 1] && jj < j[i - 1]);
            j[i] = above ? j[i - 1] : (here ? jj : j[i]);
            o[i] = above ? o[i - 1] : (here ? u : o[i]);
            below_prev = above;
        }
        if (below_prev) {
            o[0] = u;
            j[0] = jj;
        }
    }

    __device__ __forceinline__ void pop_front()
    {
#pragma unroll
        for (int i = 0; i < L - 1; ++i) {
            o[i] = o[i + 1];
            j[i] = j[i + 1];
        }
        o[L - 1] = kEmpty;
        j[L - 1] = kNone;
    }
};

// Offer a chunk's 32 scores (columns j0 .. j0 + 31, minimum m ignoring NaN)
// to the list.  thr is the list's last score as a float: NaN while a slot is
// unused or when the last entry is NaN, so !(s >= thr) lets every column
// through to the exact test.  Behind a NaN last entry only numbers can still
// enter (a NaN column's index is larger than every NaN held), so a chunk with
// no number (m is NaN) returns at once: a point whose scores are all NaN
// costs two comparisons per chunk.
// The chunk is first copied to this thread's shared slot (float4 i at
// slot + 512 i, conflict-free across the warp), so each marked column is one
// shared load instead of a 31-select tree.
//
// The accumulators hold the folded t = x.c - ||c||^2 / 2 = -s / 2 (the norms
// enter through one more MMA step), so the tests run on t: s < thr exactly
// when t > tthr = -thr / 2, and a candidate's score is s = -2 t (both exact).
// mt is the chunk's largest t (NaN only if every t is NaN).
template <int L>
__device__ __forceinline__ void admit_chunk(TopList<L> &lst, const float (&t)[32], float mt,
                                            int j0, float &tthr, uint32_t slot)
{
    if (mt != mt && lst.o[L - 1] == kNaNOrd)
        return;
    uint32_t mask = 0;
#pragma unroll
    for (int e = 0; e < 32; ++e)
        mask |= (t[e] <= tthr) ? 0u : (1u << e);
#pragma unroll
    for (int i = 0; i < 8; ++i)
        st_shared_v4(slot + 512u * i, t[4 * i], t[4 * i + 1], t[4 * i + 2], t[4 * i + 3]);
    while (mask != 0u) {
        const int e = __ffs(mask) - 1;
        mask &= mask - 1u;
        const uint32_t u = ord_of(
            -2.0f * lds_f32(slot + 512u * static_cast<uint32_t>(e >> 2) + 4u * (e & 3)));
        if (u < lst.o[L - 1])
            lst.push_later(u, j0 + e);
    }
    tthr = -0.5f * of_ord(lst.o[L - 1]);
}

template <int KB, int L>
__global__ void __launch_bounds__(32 * (kTopConsumerWarps + 4), 1)
    topk_kernel(const __grid_constant__ CUtensorMap xmap, const __grid_constant__ CUtensorMap cmap,
                const AssignParams p)
{
    constexpr int SUB = kTopSub;
    constexpr int NT = kTopNt;
    constexpr int kConsumerWarps = kTopConsumerWarps;
    constexpr int kProducerWarp = kConsumerWarps;
    constexpr int kMmaWarp = kConsumerWarps + 1;
    constexpr int kNormWarp = kConsumerWarps + 2;
    constexpr int kXWarp = kConsumerWarps + 3;
    constexpr int kChunks = NT / 32;
    // Chunks loaded per tcgen05.wait::ld: fewer for long lists, whose
    // registers would otherwise spill.
    constexpr int kGroup = L >= 32 ? 1 : L >= 8 ? 2 : 4;
    constexpr int kGroups = kChunks / kGroup;
    constexpr uint32_t kCStageBytes = NT * 128;
    constexpr uint32_t kXBufBytes = SUB * KB * kXTileBytes;
    constexpr uint32_t kAccCols = SUB * NT;
    constexpr uint32_t kTmemCols = 2 * kAccCols;
    static_assert(kTmemCols <= 512, "accumulators exceed tensor memory");
    static_assert(L >= 1 && L <= 32, "list longer than a chunk");

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    const uint32_t x_base = base;
    const uint32_t c_base = x_base + p.xbufs * kXBufBytes;
    const uint32_t cn_base = c_base + p.stages * kCStageBytes;   // float[kCnStages][NT]
    // folded norms: the ones tile, then the fold slots the norm warp fills
    const uint32_t snap_base = cn_base + kOnesBytes + kFoldStages * NT * 32u;   // [warp][8][32] float4
    const uint32_t bar_base = snap_base + kConsumerWarps * 4096u;
    uint8_t *misc_ptr = smem_raw + (bar_base - raw) + kNumBars * 8;
    volatile uint32_t *tmem_slot = reinterpret_cast<volatile uint32_t *>(misc_ptr);
    volatile uint32_t *abort_flag = reinterpret_cast<volatile uint32_t *>(misc_ptr + 4);
    auto bar = [&](int i) -> uint32_t { return bar_base + 8u * static_cast<uint32_t>(i); };

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0)
        init_barriers<kConsumerWarps, true>(bar_base, abort_flag);
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
        mma_role<SUB, NT, KB, true>(p, x_base, c_base, bar_base, tmem_base, abort_flag, cn_base);
    } else if (warp == kNormWarp) {
        fold_norm_role<SUB, NT>(p, cn_base, bar_base, abort_flag);
    } else {
        // Consumer warp w reads TMEM lanes 32*(w%4) .. +31 of sub-tile w/4,
        // every column of every tile.
        const int q = warp & 3;
        const int t = warp >> 2;
        const bool distances = p.xnorm != nullptr;
        const uint32_t slot = snap_base + 4096u * warp + 16u * lane;
        uint32_t acc_used = 0;
        bool ok = true;

        for (int u = blockIdx.x; u < p.num_units; u += gridDim.x) {
            const Unit w = decode_unit<SUB>(p, u);
            TopList<L> lst;
            lst.clear();
            float tthr = __int_as_float(0x7fc00000);   // -(the list's last score) / 2
            for (int tile = w.t_begin; tile < w.t_end; ++tile, ++acc_used) {
                const uint32_t as = acc_used & 1u;
                const uint32_t aph = (acc_used >> 1) & 1u;
                if (ok)
                    ok = wait_warp(bar(kBarAccFull + as), aph, abort_flag, p.timeout_ns);
                if (ok) {
                    tc_fence_after();
                    const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                                           as * kAccCols + t * NT;
#pragma unroll
                    for (int g = 0; g < kGroups; ++g) {
                        __syncwarp();   // tcgen05.ld is .sync.aligned
                        float v[kGroup][32];
                        float m[kGroup];   // chunk maxima, reduced by the loads
#pragma unroll
                        for (int c = 0; c < kGroup; ++c)
                            tmem_ld_red_max_32x32b_x32(taddr + (g * kGroup + c) * 32, v[c], m[c]);
                        tmem_wait_ld();
                        if (g == kGroups - 1) {
                            // Scores are in registers: hand the stage back.
                            tc_fence_before();
                            __syncwarp();
                            if (lane == 0)
                                mbar_arrive(bar(kBarAccEmpty + as));
                        }
                        const int jg = tile * NT + g * kGroup * 32;
#pragma unroll
                        for (int c = 0; c < kGroup; ++c)
                            if (!(m[c] <= tthr))
                                admit_chunk<L>(lst, v[c], m[c], jg + 32 * c, tthr, slot);
                    }
                }
            }

            const int row = w.row0 + t * kTileM + q * 32 + lane;
            if (ok && t < w.nsub && row < p.N) {
                if (!w.split) {
                    const float xn = distances ? p.xnorm[row] : 0.0f;
                    int32_t *oi = p.idx + static_cast<int64_t>(row) * p.topk;
                    float *os = p.minscore == nullptr
                                    ? nullptr
                                    : p.minscore + static_cast<int64_t>(row) * p.topk;
#pragma unroll
                    for (int e = 0; e < L; ++e) {
                        if (e < p.topk) {
                            oi[e] = lst.j[e];
                            if (os != nullptr)
                                os[e] = finish_score(lst.o[e], xn, distances);
                        }
                    }
                } else {
                    const int kc = w.t_begin / p.chunk_tiles;
                    const int64_t r = static_cast<int64_t>(row) -
                                      static_cast<int64_t>(p.split_row0) * SUB * kTileM;
                    ulonglong2 *dst =
                        reinterpret_cast<ulonglong2 *>(p.keys + (r * p.ksplit + kc) * L);
#pragma unroll
                    for (int e = 0; e < L; e += 2) {
                        ulonglong2 pr;
                        pr.x = (static_cast<unsigned long long>(lst.o[e]) << 32) |
                               static_cast<uint32_t>(lst.j[e]);
                        pr.y = (static_cast<unsigned long long>(lst.o[e + 1]) << 32) |
                               static_cast<uint32_t>(lst.j[e + 1]);
                        dst[e / 2] = pr;
                    }
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

// One warp per split point: lane l merges the sorted lists of ranges l,
// l + 32, ...; then k rounds each take the smallest head across the lanes.
template <int L>
__global__ void __launch_bounds__(256)
    topk_merge_kernel(const unsigned long long *__restrict__ part, int64_t rows, int ksplit, int k,
                      const float *__restrict__ xnorm, int32_t *__restrict__ idx,
                      float *__restrict__ score)
{
    const int lane = threadIdx.x & 31;
    const int64_t r = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    if (r >= rows)
        return;   // uniform per warp
    TopList<L> lst;
    lst.clear();
    const unsigned long long *src = part + r * ksplit * L;
    if (lane < ksplit) {
        // The first list is already sorted.
#pragma unroll
        for (int e = 0; e < L; ++e) {
            const unsigned long long key = src[lane * L + e];
            lst.o[e] = static_cast<uint32_t>(key >> 32);
            lst.j[e] = static_cast<int32_t>(key & 0xffffffffull);
        }
    }
    for (int s = lane + 32; s < ksplit; s += 32) {
#pragma unroll
        for (int e = 0; e < L; ++e) {
            const unsigned long long key = src[s * L + e];
            const uint32_t u = static_cast<uint32_t>(key >> 32);
            const int32_t jj = static_cast<int32_t>(key & 0xffffffffull);
            if (u < lst.o[L - 1] || (u == lst.o[L - 1] && jj < lst.j[L - 1]))
                lst.push(u, jj);
        }
    }
    const bool distances = xnorm != nullptr;
    const float xn = distances ? xnorm[r] : 0.0f;
    for (int e = 0; e < k; ++e) {
        uint32_t bo = lst.o[0];
        int32_t bj = lst.j[0];
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            const uint32_t oo = __shfl_xor_sync(0xffffffffu, bo, off);
            const int32_t oj = __shfl_xor_sync(0xffffffffu, bj, off);
            if (oo < bo || (oo == bo && oj < bj)) {
                bo = oo;
                bj = oj;
            }
        }
        if (lst.o[0] == bo && lst.j[0] == bj)
            lst.pop_front();
        if (lane == 0) {
            idx[r * k + e] = bj;
            if (score != nullptr)
                score[r * k + e] = finish_score(bo, xn, distances);
        }
    }
}

template <int KB, int L>
cudaError_t prepare_topk_one(size_t smem)
{
    return cudaFuncSetAttribute(topk_kernel<KB, L>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                static_cast<int>(smem));
}

template <int KB, int L>
cudaError_t launch_topk_one(const AssignParams &p, const CUtensorMap &xmap, const CUtensorMap &cmap,
                            int grid, size_t smem, cudaStream_t stream)
{
    topk_kernel<KB, L><<<grid, 32 * (kTopConsumerWarps + 4), smem, stream>>>(xmap, cmap, p);
    return cudaGetLastError();
}

template <int L>
cudaError_t dispatch_topk_kb(bool prepare, int kb, const AssignParams *p, const CUtensorMap *xmap,
                             const CUtensorMap *cmap, int grid, size_t smem, cudaStream_t stream)
{
    switch (kb) {
    case 1:
        return prepare ? prepare_topk_one<1, L>(smem)
                       : launch_topk_one<1, L>(*p, *xmap, *cmap, grid, smem, stream);
    case 2:
        return prepare ? prepare_topk_one<2, L>(smem)
                       : launch_topk_one<2, L>(*p, *xmap, *cmap, grid, smem, stream);
    case 3:
        return prepare ? prepare_topk_one<3, L>(smem)
                       : launch_topk_one<3, L>(*p, *xmap, *cmap, grid, smem, stream);
    case 4:
        return prepare ? prepare_topk_one<4, L>(smem)
                       : launch_topk_one<4, L>(*p, *xmap, *cmap, grid, smem, stream);
    default:
        return cudaErrorInvalidValue;
    }
}

cudaError_t dispatch_topk(bool prepare, int kb, int L, const AssignParams *p,
                          const CUtensorMap *xmap, const CUtensorMap *cmap, int grid, size_t smem,
                          cudaStream_t stream)
{
    switch (L) {
    case 4:
        return dispatch_topk_kb<4>(prepare, kb, p, xmap, cmap, grid, smem, stream);
    case 8:
        return dispatch_topk_kb<8>(prepare, kb, p, xmap, cmap, grid, smem, stream);
    case 16:
        return dispatch_topk_kb<16>(prepare, kb, p, xmap, cmap, grid, smem, stream);
    case 32:
        return dispatch_topk_kb<32>(prepare, kb, p, xmap, cmap, grid, smem, stream);
    default:
        return cudaErrorInvalidValue;
    }
}

}  // namespace

const Variant kTopkVariant = {kTopSub, kTopNt, 1, false};

int topk_list_size(int k)
{
    return k <= 4 ? 4 : k <= 8 ? 8 : k <= 16 ? 16 : 32;
}

size_t topk_smem_bytes(int kblocks, int stages, int xbufs)
{
    return 1024 + static_cast<size_t>(xbufs) * kTopSub * kblocks * kXTileBytes +
           static_cast<size_t>(stages) * kTopNt * 128 + kOnesBytes + kFoldStages * kTopNt * 32 +
           static_cast<size_t>(kTopConsumerWarps) * 4096 + kMiscBytes;
}

cudaError_t topk_prepare(int kblocks, int list, size_t smem)
{
    return dispatch_topk(true, kblocks, list, nullptr, nullptr, nullptr, 0, smem, nullptr);
}

cudaError_t launch_topk(int kblocks, int list, const AssignParams &p, const CUtensorMap &xmap,
                        const CUtensorMap &cmap, int grid, size_t smem, cudaStream_t stream)
{
    return dispatch_topk(false, kblocks, list, &p, &xmap, &cmap, grid, smem, stream);
}

cudaError_t launch_topk_merge(int list, const unsigned long long *part, int64_t rows, int ksplit,
                              int k, const float *xnorm, int32_t *idx, float *score,
                              cudaStream_t stream)
{
    const int threads = 256;
    const int64_t blocks = (rows * 32 + threads - 1) / threads;
    switch (list) {
    case 4:
        topk_merge_kernel<4><<<static_cast<unsigned>(blocks), threads, 0, stream>>>(
            part, rows, ksplit, k, xnorm, idx, score);
        break;
    case 8:
        topk_merge_kernel<8><<<static_cast<unsigned>(blocks), threads, 0, stream>>>(
            part, rows, ksplit, k, xnorm, idx, score);
        break;
    case 16:
        topk_merge_kernel<16><<<static_cast<unsigned>(blocks), threads, 0, stream>>>(
            part, rows, ksplit, k, xnorm, idx, score);
        break;
    case 32:
        topk_merge_kernel<32><<<static_cast<unsigned>(blocks), threads, 0, stream>>>(
            part, rows, ksplit, k, xnorm, idx, score);
        break;
    default:
        return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

cudaError_t topk_status_read_and_clear(int *code)
{
    int zero = 0;
    cudaError_t e = cudaMemcpyFromSymbol(code, g_status_word, sizeof(int));
    if (e != cudaSuccess)
        return e;
    return cudaMemcpyToSymbol(g_status_word, &zero, sizeof(int));
}

}  // namespace kma
