// api.cu -- the C ABI of libkmassign: argument checks, planning, temporaries,
// TMA descriptors and launches.  No arithmetic of the method lives here.
#include "kmassign.h"
#include "internal.h"

#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <cstdint>
#include <mutex>

namespace {

using kma::AssignParams;

constexpr uint64_t kDefaultTimeoutNs = 2000000000ull;   // 2 s per pipeline wait
constexpr int kMaxDevices = 64;
std::atomic<uint64_t> g_wait_timeout_ns{kDefaultTimeoutNs};

struct DeviceInfo {
    bool ready = false;
    int sms = 0;
    int smem_optin = 0;
    // Library-owned stream-ordered pool for the temporaries.  It keeps up to
    // kPoolKeepBytes reserved across synchronisations; the default pool would
    // hand its memory back at every synchronisation and re-map it per call.
    cudaMemPool_t pool = nullptr;
    int pair_clusters = 0;   // co-resident clusters of the pair kernel (0: none)
};
constexpr uint64_t kPoolKeepBytes = uint64_t(1) << 30;

std::mutex g_mutex;
DeviceInfo g_dev[kMaxDevices];
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
bool g_encode_tried = false;

int current_device_info(DeviceInfo *out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return KMASSIGN_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mutex);
    DeviceInfo &d = g_dev[dev];
    if (!d.ready) {
        if (cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&d.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) !=
                cudaSuccess)
            return KMASSIGN_ERR_CUDA;
        for (const auto &v : kma::kVariants)
            for (int kb = 1; kb <= 4; ++kb)
                if (kma::assign_prepare(v, kb, static_cast<size_t>(d.smem_optin)) != cudaSuccess)
                    return KMASSIGN_ERR_CUDA;
        for (int list = 4; list <= 32; list *= 2)
            for (int kb = 1; kb <= 4; ++kb)
                if (kma::topk_prepare(kb, list, static_cast<size_t>(d.smem_optin)) != cudaSuccess)
                    return KMASSIGN_ERR_CUDA;
        cudaMemPoolProps props = {};
        props.allocType = cudaMemAllocationTypePinned;
        props.location.type = cudaMemLocationTypeDevice;
        props.location.id = dev;
        int clusters = 0;
        const kma::Variant pv{1, 256, 2, true};
        if (kma::assign_max_clusters(pv, 4, static_cast<size_t>(d.smem_optin), &clusters) !=
            cudaSuccess) {
            cudaGetLastError();
            clusters = 0;
        }
        d.pair_clusters = std::min(clusters, d.sms / 2);
        uint64_t keep = kPoolKeepBytes;
        if (cudaMemPoolCreate(&d.pool, &props) != cudaSuccess ||
            cudaMemPoolSetAttribute(d.pool, cudaMemPoolAttrReleaseThreshold, &keep) != cudaSuccess)
            return KMASSIGN_ERR_CUDA;
        d.ready = true;
    }
    *out = d;
    return KMASSIGN_OK;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn()
{
    std::lock_guard<std::mutex> lock(g_mutex);
    if (!g_encode_tried) {
        g_encode_tried = true;
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    return g_encode;
}

// Row-major bf16 [rows, D], boxes of 64 columns x box_rows rows, 128-byte
// swizzle (the K-major layout the tensor-core descriptors expect).  Boxes
// reaching past the tensor are zero-filled by the copy engine.
bool encode_map(CUtensorMap *m, const void *ptr, uint64_t rows, uint64_t D, uint32_t box_rows)
{
    auto fn = encode_fn();
    if (fn == nullptr)
        return false;
    cuuint64_t dims[2] = {D, rows};
    cuuint64_t strides[1] = {D * 2};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(kma::kKBlock), box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(ptr), dims, strides,
                    box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// The CTA pair's fold operand (fold_operand_blocks(K) blocks of 4 KiB) as
// rows of 8 bf16 (16 bytes), boxes of 256 rows = one block, no swizzle.
bool encode_fold_map(CUtensorMap *m, const void *ptr, int64_t K)
{
    auto fn = encode_fn();
    if (fn == nullptr)
        return false;
    cuuint64_t dims[2] = {8, static_cast<cuuint64_t>(kma::fold_operand_blocks(K)) * 256};
    cuuint64_t strides[1] = {16};
    cuuint32_t box[2] = {8, 256};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(ptr), dims, strides,
                    box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

bool aligned(const void *p, uintptr_t a)
{
    return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0;
}

// Host or foreign pointers would make the copy engine fault: reject them.
// Every non-NULL pointer must be device (or managed) memory of one device;
// that device is made current for this library's runtime before launching
// (the caller's framework may track its current device separately), and the
// entry point's DeviceRestore puts the caller's current device back.
int check_device_ptrs(const void *const *ptrs, int n)
{
    int owner = -1;
    for (int i = 0; i < n; ++i) {
        if (ptrs[i] == nullptr)
            continue;
        cudaPointerAttributes a;
        if (cudaPointerGetAttributes(&a, ptrs[i]) != cudaSuccess) {
            cudaGetLastError();
            return KMASSIGN_ERR_NOT_DEVICE;
        }
        if (a.type != cudaMemoryTypeDevice && a.type != cudaMemoryTypeManaged)
            return KMASSIGN_ERR_NOT_DEVICE;
        if (a.type == cudaMemoryTypeDevice) {
            if (owner >= 0 && a.device != owner)
                return KMASSIGN_ERR_NOT_DEVICE;
            owner = a.device;
        }
    }
    if (owner >= 0) {
        int cur = -1;
        if (cudaGetDevice(&cur) != cudaSuccess)
            return KMASSIGN_ERR_CUDA;
        if (cur != owner && cudaSetDevice(owner) != cudaSuccess)
            return KMASSIGN_ERR_CUDA;
    }
    return KMASSIGN_OK;
}

// Puts back the calling thread's current device when an entry point returns
// (check_device_ptrs makes the pointers' device current for the launches;
// the caller's own notion of its current device must not change).
class DeviceRestore {
public:
    DeviceRestore()
    {
        if (cudaGetDevice(&dev_) != cudaSuccess) {
            cudaGetLastError();
            dev_ = -1;
        }
    }
    ~DeviceRestore()
    {
        int cur = -1;
        if (dev_ >= 0 && cudaGetDevice(&cur) == cudaSuccess && cur != dev_)
            cudaSetDevice(dev_);
    }
    DeviceRestore(const DeviceRestore &) = delete;
    DeviceRestore &operator=(const DeviceRestore &) = delete;

private:
    int dev_ = -1;
};

int check_shape(int64_t N, int64_t K, int64_t D)
{
    const int64_t lim = int64_t(1) << 31;
    if (N < 0 || N >= lim || K < 1 || K >= lim)
        return KMASSIGN_ERR_SHAPE;
    if (D < 16 || D > 256 || (D % 16) != 0)
        return KMASSIGN_ERR_UNSUPPORTED_D;
    return KMASSIGN_OK;
}

struct Plan {
    kma::Variant v;
    int ksplit, grid, stages, xbufs;
    int rowtiles, ntiles, chunk_tiles, units;
    int full_units, split_row0;   // see AssignParams
    size_t smem;
};

int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Units u < X with u % P == b under the static round-robin schedule.
int64_t units_of_block(int64_t X, int64_t P, int64_t b) { return X > b ? (X - b - 1) / P + 1 : 0; }

// Pick the kernel shape and the centroid split from a cost model in SM
// clocks per centroid tile, fitted to measurements of the kernel on GB300
// (the five benchmark workloads, every shape forced in turn):
//   * tensor pipe: a 128x256x16 bf16 MMA takes 128 clocks back to back, a
//     128x128x16 one ~80 with two accumulators and ~92 with one, plus ~500
//     clocks of hand-over per tile (with folded norms one more MMA step);
//   * epilogue floor per tile (latency-bound reduction): ~2150 clocks for a
//     128x256 tile with 8 or 16 warps, ~1700 / ~1550 for a 256x128 tile with
//     8 / 16 warps (~1500 / ~1600 with folded norms), ~1400 for a 128x128
//     tile with 4 warps;
//   * a CTA pair costs its measured tile time: above D = 128 the larger of
//     its MMA time and floor, scaled by 0.94; at D <= 128, where it folds,
//     ~1050 (D = 64) / ~1380 (D = 128) clocks with 8 warps, plus ~4000
//     clocks per call for the fold operand (written by the preparation
//     launch, which computes the norms too when the caller gives none);
//   * a unit pays ~5000 clocks to load its X tile and fill the pipe;
//   * any split pays ~5000 clocks: the keys' initial values (the same
//     preparation launch) and the merge at the end of each split unit (one
//     atomic per row for two ranges; with more, an arrival count whose last
//     unit turns the keys into the answers).  The variant is chosen with
//     that flat cost; within the chosen variant a split into two ranges is
//     then re-weighed at ~3000 clocks (kTwoRangeSplitCost, below), since
//     its merge is one atomic per row.  Re-weighing before the variant
//     choice tipped some shapes from a CTA pair to single blocks, which
//     measured slower.
// Splits considered: every row tile into ks centroid ranges (ks >= 1), or
// only the row tiles of the last partial wave (the rest stay whole), which
// evens out the last wave when there are a few waves of whole row tiles.
// force_ksplit > 0 forces a uniform split, < -1 a tail split into
// -force_ksplit ranges.  topk plans the k-nearest kernel: its one shape (256
// x 128 tiles) and shared-memory layout; its epilogue cost per tile depends on
// the data and is taken as the assignment's, which only matters for choosing
// the split.
// A two-range split's cost in the re-weighing below: on the shapes whose plan
// it changes (a whole plan becoming a tail split in 2, N 65,536-524,288) the
// new plans measured level to 5.5% faster.
constexpr double kTwoRangeSplitCost = 3000.0;

int make_plan(int64_t N, int64_t K, int64_t D, const DeviceInfo &dev, int force_ksplit,
              int force_rows, int force_nt, int force_cw, bool topk, Plan *out,
              bool no_pair = false)
{
    auto smem_of = [&](const kma::Variant &v, int kblocks, int stages, int xbufs) {
        return topk ? kma::topk_smem_bytes(kblocks, stages, xbufs)
                    : kma::assign_smem_bytes(v, kblocks, stages, xbufs);
    };
    const int kblocks = static_cast<int>(cdiv(D, kma::kKBlock));
    bool found = false;
    double best_cost = 0.0;
    Plan best{};
    // The re-weighed cost of the plan chosen so far, its variant, and each
    // variant's two-range split candidates (at most two: every row tile, or
    // the last wave's) with their re-weighed costs.
    double best_cost2 = 0.0;
    int best_vi = 0;
    struct TwoRange {
        double cost2;
        Plan plan;
    };
    TwoRange two_range[kma::kNumVariants][2];
    int n_two_range[kma::kNumVariants] = {};
    const kma::Variant *variants = topk ? &kma::kTopkVariant : kma::kVariants;
    const int nvariants = topk ? 1 : kma::kNumVariants;
    for (int vi = 0; vi < nvariants; ++vi) {
        const kma::Variant &v = variants[vi];
        const int rows = (v.pair ? 2 : v.sub) * kma::kTileM;   // points per unit
        if (force_rows != 0 && force_rows != rows)
            continue;
        if (force_nt != 0 && force_nt != v.nt)
            continue;
        if (force_cw != 0 && force_cw != 4 * v.sub * v.ch)
            continue;
        if (v.pair && (dev.pair_clusters < 1 || no_pair))
            continue;
        const int64_t P = v.pair ? dev.pair_clusters : dev.sms;   // units run in parallel
        // Shared memory: at least 2 ring stages and one X buffer; two X
        // buffers when 4 stages still fit; then as many stages as fit.
        // A folding CTA pair's ring holds whole tiles (groups of kblocks
        // stages, at least two groups).
        const size_t budget = static_cast<size_t>(dev.smem_optin);
        auto fits = [&](int st, int xb) { return smem_of(v, kblocks, st, xb) <= budget; };
        const int group = topk ? 1 : kma::assign_stage_group(v, kblocks);
        if (!fits(2 * group, 1))
            continue;
        const int xbufs = fits(std::max(4, 2 * group), 2) ? 2 : 1;
        int stages = 2 * group;
        while (stages + group <= kma::kMaxStages && fits(stages + group, xbufs))
            stages += group;
        const int64_t ntiles = cdiv(K, v.nt);
        const int64_t R = cdiv(N, static_cast<int64_t>(rows));
        const double mma_clk = v.nt == 256 ? 128.0 : (v.sub == 2 ? 80.0 : 92.0);
        // Kernels that fold the norms into one more MMA step (every shape at
        // D <= 128) have a lighter reduction (256x128 single-block tiles at
        // D = 64: ~1,500 clocks with 8 warps, ~1,600 with 16; a CTA pair's
        // 128x256 per SM: ~1,050 at D = 64 and ~1,380 at D = 128, against
        // ~1,780 for the 256x128 single block at D = 128).
        const bool fold = !topk && kma::assign_folds(v, kblocks);
        const double tile_mma = double(v.sub) * (kblocks * 4 + (fold ? 1 : 0)) * mma_clk + 500.0;
        const double tile_epi =
            (v.pair && fold)
                ? (v.ch == 2 ? 1450.0 : 1600.0)
                : fold ? (v.nt == 256 ? 2150.0 : v.sub == 2 ? (v.ch == 2 ? 1600.0 : 1500.0) : 1400.0)
                       : (v.nt == 256 ? 2150.0 : v.sub == 2 ? (v.ch == 2 ? 1550.0 : 1700.0)
                                                            : 1400.0);
        // The pair kernel halves each SM's C traffic but couples both SMs'
        // consumers on every tile.  Measured against the single-block shapes
        // (iid inputs): 5-8% faster at D = 192 and at D = 256 with at most 16
        // tiles per unit; at D = 256 with 64 tiles per unit level in short
        // bursts at full clock and 5-7% faster in long runs under the power
        // cap (less L2 traffic per flop).  At D <= 128 it folds, modelled
        // by its reduction floor above.
        const double pair_factor = kblocks >= 3 ? 0.94 : 1.0;
        // A folding pair's tile is its fitted time (8 warps: ~1,050 clocks
        // at D = 64, ~1,380 at D = 128, since its tiles take one ring wait
        // and two commits), below its modelled MMA time; its fold operand
        // costs one small kernel per call.  Fitted so that the pair is chosen
        // from ~2,048 centroids up at D = 64, where it measured 7-12% faster
        // than the single block, and single blocks below.
        const bool pair_fold = v.pair && fold;
        const double tile = pair_fold ? (v.ch == 2 ? (kblocks == 1 ? 1050.0 : 1380.0) : 1600.0)
                                      : std::max(tile_mma, tile_epi) * (v.pair ? pair_factor : 1.0);
        const double call_over = pair_fold ? 4000.0 : 0.0;
        const double unit_over = 5000.0;

        // Candidate (F whole row tiles, split the rest into ks ranges).
        auto consider = [&](int64_t F, int64_t ks) {
            const int64_t chunk = cdiv(ntiles, ks);
            const int64_t ks_eff = cdiv(ntiles, chunk);
            const int64_t split_rows = R - F;
            const int64_t units = F + split_rows * ks_eff;
            if (units >= (int64_t(1) << 31) || units <= 0)
                return;
            const bool any_split = split_rows > 0 && ks_eff > 1;
            const int64_t full_units = any_split ? F : R;   // ks 1: nothing is split
            const int64_t split_row0 = any_split ? F : R;
            const int64_t nunits = full_units + (R - split_row0) * (any_split ? ks_eff : 1);
            // A block's load is piecewise constant in its index, changing
            // only where the whole and the split ranges end.
            double worst = 0.0;
            const int64_t probes[4] = {0, full_units % P, nunits % P, P - 1};
            for (int64_t b : probes) {
                if (b >= std::min<int64_t>(P, nunits))
                    continue;
                const int64_t nf = units_of_block(full_units, P, b);
                const int64_t ns = units_of_block(nunits, P, b) - nf;
                const double c = double(nf) * (double(ntiles) * tile + unit_over) +
                                 double(ns) * (double(chunk) * tile + unit_over);
                worst = std::max(worst, c);
            }
            const double cost = worst + (any_split ? 5000.0 : 0.0) + call_over;
            const bool two = any_split && ks_eff == 2;
            const double cost2 = two ? worst + kTwoRangeSplitCost + call_over : cost;
            const bool take = !found || cost < best_cost * 0.995;
            if (!take && !(two && !topk))
                return;
            Plan c{};
            c.v = v;
            c.ksplit = any_split ? static_cast<int>(ks_eff) : 1;
            c.rowtiles = static_cast<int>(R);
            c.ntiles = static_cast<int>(ntiles);
            c.chunk_tiles = any_split ? static_cast<int>(chunk) : static_cast<int>(ntiles);
            c.full_units = static_cast<int>(full_units);
            c.split_row0 = static_cast<int>(split_row0);
            c.units = static_cast<int>(nunits);
            c.grid = static_cast<int>(std::min<int64_t>(nunits, P) * (v.pair ? 2 : 1));
            c.stages = stages;
            c.xbufs = xbufs;
            c.smem = smem_of(v, kblocks, stages, xbufs);
            if (take) {
                found = true;
                best_cost = cost;
                best_cost2 = cost2;
                best_vi = vi;
                best = c;
            }
            if (two && !topk && n_two_range[vi] < 2)
                two_range[vi][n_two_range[vi]++] = TwoRange{cost2, c};
        };
        if (force_ksplit > 0) {
            const int64_t ks = std::min<int64_t>(force_ksplit, ntiles);
            consider(ks > 1 ? 0 : R, ks);
        } else if (force_ksplit < -1) {
            const int64_t ks = std::min<int64_t>(-force_ksplit, ntiles);
            const int64_t F = (R > P && R % P != 0) ? (R / P) * P : 0;
            consider(F, ks);
        } else {
            for (int64_t ks = 1; ks <= std::min<int64_t>(ntiles, 64); ++ks) {
                const int64_t chunk = cdiv(ntiles, ks);
                if (cdiv(ntiles, chunk) != ks)
                    continue;
                consider(ks > 1 ? 0 : R, ks);
                if (ks > 1 && R > P && R % P != 0 && ks <= 16)
                    consider((R / P) * P, ks);
            }
        }
    }
    if (!found)
        return KMASSIGN_ERR_ARG;
    // The variant stays the one chosen above; within it, a two-range split
    // replaces the plan when its re-weighed cost is lower by the same margin.
    if (force_ksplit == 0) {
        for (int i = 0; i < n_two_range[best_vi]; ++i) {
            const TwoRange &t = two_range[best_vi][i];
            if (t.cost2 < best_cost2 * 0.995) {
                best_cost2 = t.cost2;
                best = t.plan;
            }
        }
    }
    *out = best;
    return KMASSIGN_OK;
}

// Plans are pure functions of (shape, forced fields, device): remember them.
struct PlanKey {
    int64_t N, K, D;
    int ksplit, rows, nt, cw, dev;
    bool topk, no_pair;
    bool operator==(const PlanKey &o) const
    {
        return N == o.N && K == o.K && D == o.D && ksplit == o.ksplit && rows == o.rows &&
               nt == o.nt && cw == o.cw && dev == o.dev && topk == o.topk &&
               no_pair == o.no_pair;
    }
};
constexpr int kPlanCacheSize = 64;
PlanKey g_plan_keys[kPlanCacheSize];
Plan g_plans[kPlanCacheSize];
int g_plan_count = 0, g_plan_next = 0;

int cached_plan(int64_t N, int64_t K, int64_t D, const DeviceInfo &dev, int dev_id, int ksplit,
                int rows, int nt, int cw, Plan *out, bool topk = false, bool no_pair = false)
{
    const PlanKey key{N, K, D, ksplit, rows, nt, cw, dev_id, topk, no_pair};
    {
        std::lock_guard<std::mutex> lock(g_mutex);
        for (int i = 0; i < g_plan_count; ++i)
            if (g_plan_keys[i] == key) {
                *out = g_plans[i];
                return KMASSIGN_OK;
            }
    }
    const int rc = make_plan(N, K, D, dev, ksplit, rows, nt, cw, topk, out, no_pair);
    if (rc != KMASSIGN_OK)
        return rc;
    std::lock_guard<std::mutex> lock(g_mutex);
    g_plan_keys[g_plan_next] = key;
    g_plans[g_plan_next] = *out;
    g_plan_next = (g_plan_next + 1) % kPlanCacheSize;
    g_plan_count = std::min(g_plan_count + 1, kPlanCacheSize);
    return KMASSIGN_OK;
}

// Fill the kernel parameters of a plan.
AssignParams make_params(const Plan &plan, const float *cnorm, int32_t *idx, float *minscore,
                         unsigned long long *keys, int64_t N, int64_t K, int64_t D)
{
    AssignParams p{};
    p.cnorm = cnorm;
    p.idx = idx;
    p.minscore = minscore;
    p.keys = keys;
    p.N = static_cast<int32_t>(N);
    p.K = static_cast<int32_t>(K);
    p.D = static_cast<int32_t>(D);
    p.ksteps = static_cast<int32_t>(D / 16);
    p.kblocks = static_cast<int32_t>(cdiv(D, kma::kKBlock));
    p.rowtiles = plan.rowtiles;
    p.full_units = plan.full_units;
    p.split_row0 = plan.split_row0;
    p.ksplit = plan.ksplit;
    p.chunk_tiles = plan.chunk_tiles;
    p.ntiles = plan.ntiles;
    p.num_units = plan.units;
    p.stages = plan.stages;
    p.stage_group = kma::assign_stage_group(plan.v, p.kblocks);
    p.xbufs = plan.xbufs;
    p.timeout_ns = g_wait_timeout_ns.load();
    return p;
}

// Rows of C in one TMA box: the whole tile, or each CTA's half of it when a
// CTA pair shares the tile (each loads 128 of its 256 centroids).
uint32_t c_box_rows(const Plan &plan)
{
    return static_cast<uint32_t>(plan.v.pair ? plan.v.nt / 2 : plan.v.nt);
}

// First point whose answer goes through the packed keys.
int64_t split_first_row(const Plan &plan)
{
    return int64_t(plan.split_row0) * (plan.v.pair ? 2 : plan.v.sub) * kma::kTileM;
}

int run_assign(const void *X, const void *C, const float *cnorm, int64_t N, int64_t K, int64_t D,
               int32_t *idx, float *minscore, int force_ksplit, int force_rows, int force_nt,
               int force_cw, cudaStream_t stream, int32_t *counts = nullptr)
{
    int rc = check_shape(N, K, D);
    if (rc != KMASSIGN_OK)
        return rc;
    if (force_ksplit == -1 || (force_rows != 0 && force_rows != 128 && force_rows != 256) ||
        (force_nt != 0 && force_nt != 128 && force_nt != 256) ||
        (force_cw != 0 && force_cw != 4 && force_cw != 8 && force_cw != 16))
        return KMASSIGN_ERR_ARG;
    if (N == 0)
        return KMASSIGN_OK;
    if (X == nullptr || C == nullptr || idx == nullptr)
        return KMASSIGN_ERR_NULL;
    if (!aligned(X, 16) || !aligned(C, 16) || (cnorm && !aligned(cnorm, 16)) || !aligned(idx, 4) ||
        (minscore && !aligned(minscore, 4)))
        return KMASSIGN_ERR_ALIGN;
    const void *ptrs[5] = {X, C, cnorm, idx, minscore};
    if ((rc = check_device_ptrs(ptrs, 5)) != KMASSIGN_OK)
        return rc;

    DeviceInfo dev;
    if ((rc = current_device_info(&dev)) != KMASSIGN_OK)
        return rc;
    int dev_id = 0;
    cudaGetDevice(&dev_id);
    Plan plan;
    if ((rc = cached_plan(N, K, D, dev, dev_id, force_ksplit, force_rows, force_nt, force_cw,
                          &plan)) != KMASSIGN_OK)
        return rc;

    CUtensorMap xmap, cmap;
    if (!encode_map(&xmap, X, static_cast<uint64_t>(N), static_cast<uint64_t>(D), kma::kTileM) ||
        !encode_map(&cmap, C, static_cast<uint64_t>(K), static_cast<uint64_t>(D),
                    c_box_rows(plan)))
        return KMASSIGN_ERR_CUDA;

    // Temporaries from the pool, all filled by one preparation launch: the
    // norms (when not given), the fold operand of a CTA pair that folds the
    // norms, and the split rows' packed keys and arrival counters.
    float *tmp_norm = nullptr;
    void *fold = nullptr;
    unsigned char *split = nullptr;
    const int kblocks = static_cast<int>(cdiv(D, kma::kKBlock));
    const bool need_fold = plan.v.pair && kma::assign_folds(plan.v, kblocks);
    const int64_t row_split = split_first_row(plan);
    const int64_t n_split = plan.ksplit > 1 ? N - row_split : 0;
    const size_t split_bytes = n_split > 0 ? kma::split_scratch_bytes(n_split) : 0;
    auto take = [&](void **ptr, size_t bytes) {
        return cudaMallocFromPoolAsync(ptr, bytes, dev.pool, stream) == cudaSuccess;
    };
    rc = KMASSIGN_OK;
    if ((cnorm == nullptr &&
         !take(reinterpret_cast<void **>(&tmp_norm), static_cast<size_t>(K) * 4)) ||
        (need_fold && !take(&fold, kma::fold_operand_bytes(K))) ||
        (split_bytes > 0 && !take(reinterpret_cast<void **>(&split), split_bytes)))
        rc = KMASSIGN_ERR_CUDA;
    CUtensorMap fmap{};
    bool prepped = false;
    if (rc == KMASSIGN_OK && (tmp_norm != nullptr || fold != nullptr || split != nullptr)) {
        if (kma::launch_prep(C, K, D, cnorm, tmp_norm, fold, split, split_bytes, stream,
                             &prepped) != cudaSuccess ||
            (fold != nullptr && !encode_fold_map(&fmap, fold, K)))
            rc = KMASSIGN_ERR_CUDA;
    }
    if (rc == KMASSIGN_OK) {
        AssignParams p = make_params(plan, cnorm != nullptr ? cnorm : tmp_norm, idx, minscore,
                                     reinterpret_cast<unsigned long long *>(split), N, K, D);
        p.counts = counts;
        if (split != nullptr)
            p.counters =
                reinterpret_cast<uint32_t *>(split + kma::split_counter_offset(n_split));
        if (kma::launch_assign(plan.v, p.kblocks, p, xmap, cmap, fmap, plan.grid, plan.smem,
                               stream, prepped) != cudaSuccess)
            rc = KMASSIGN_ERR_CUDA;
    }
    for (void *t : {static_cast<void *>(split), fold, static_cast<void *>(tmp_norm)})
        if (t != nullptr && cudaFreeAsync(t, stream) != cudaSuccess)
            rc = KMASSIGN_ERR_CUDA;
    return rc;
}

}  // namespace

namespace kma {

int library_pool(cudaMemPool_t *pool)
{
    DeviceInfo dev;
    const int rc = current_device_info(&dev);
    if (rc == KMASSIGN_OK)
        *pool = dev.pool;
    return rc;
}

int assign_wave_rows(int64_t N, int64_t K, int64_t D, int64_t *rows)
{
    int rc = check_shape(N, K, D);
    if (rc != KMASSIGN_OK)
        return rc;
    DeviceInfo dev;
    if ((rc = current_device_info(&dev)) != KMASSIGN_OK)
        return rc;
    int dev_id = 0;
    cudaGetDevice(&dev_id);
    Plan plan;
    if ((rc = cached_plan(std::max<int64_t>(N, 1), K, D, dev, dev_id, 0, 0, 0, 0, &plan)) !=
        KMASSIGN_OK)
        return rc;
    const int64_t blocks = plan.v.pair ? plan.grid / 2 : plan.grid;
    *rows = std::max<int64_t>(1, blocks * (plan.v.pair ? 2 : plan.v.sub) * kma::kTileM);
    return KMASSIGN_OK;
}

}  // namespace kma

namespace {

// The k nearest centroids of every point: idx and score hold [N, k] row-major;
// distances selects ||x||^2 + s over s for score.
int run_topk(const void *X, const void *C, const float *cnorm, int64_t N, int64_t K, int64_t D,
             int k, int32_t *idx, float *score, int distances, int force_ksplit,
             cudaStream_t stream)
{
    int rc = check_shape(N, K, D);
    if (rc != KMASSIGN_OK)
        return rc;
    if (k < 1 || k > KMASSIGN_TOPK_MAX || k > K || (distances != 0 && distances != 1) ||
        force_ksplit == -1)
        return KMASSIGN_ERR_ARG;
    if (N * k >= (int64_t(1) << 31))
        return KMASSIGN_ERR_SHAPE;
    if (N == 0)
        return KMASSIGN_OK;
    if (X == nullptr || C == nullptr || idx == nullptr || (distances && score == nullptr))
        return KMASSIGN_ERR_NULL;
    if (!aligned(X, 16) || !aligned(C, 16) || (cnorm && !aligned(cnorm, 16)) || !aligned(idx, 4) ||
        (score && !aligned(score, 4)))
        return KMASSIGN_ERR_ALIGN;
    const void *ptrs[5] = {X, C, cnorm, idx, score};
    if ((rc = check_device_ptrs(ptrs, 5)) != KMASSIGN_OK)
        return rc;

    DeviceInfo dev;
    if ((rc = current_device_info(&dev)) != KMASSIGN_OK)
        return rc;
    if (k == 1) {
        // The single nearest centroid is the assignment itself.
        if ((rc = run_assign(X, C, cnorm, N, K, D, idx, score, force_ksplit, 0, 0, 0, stream)) !=
                KMASSIGN_OK ||
            !distances)
            return rc;
        float *xnorm = nullptr;
        if (cudaMallocFromPoolAsync(reinterpret_cast<void **>(&xnorm), static_cast<size_t>(N) * 4,
                                    dev.pool, stream) != cudaSuccess)
            return KMASSIGN_ERR_CUDA;
        if (kma::launch_norms(X, N, D, xnorm, stream) != cudaSuccess ||
            kma::launch_add_norms(score, xnorm, N, stream) != cudaSuccess)
            rc = KMASSIGN_ERR_CUDA;
        if (cudaFreeAsync(xnorm, stream) != cudaSuccess)
            rc = KMASSIGN_ERR_CUDA;
        return rc;
    }
    int dev_id = 0;
    cudaGetDevice(&dev_id);
    const int list = kma::topk_list_size(k);
    Plan plan;
    if ((rc = cached_plan(N, K, D, dev, dev_id, force_ksplit, 0, 0, 0, &plan, true)) !=
        KMASSIGN_OK)
        return rc;

    CUtensorMap xmap, cmap;
    if (!encode_map(&xmap, X, static_cast<uint64_t>(N), static_cast<uint64_t>(D), kma::kTileM) ||
        !encode_map(&cmap, C, static_cast<uint64_t>(K), static_cast<uint64_t>(D),
                    c_box_rows(plan)))
        return KMASSIGN_ERR_CUDA;

    float *tmp_norm = nullptr, *xnorm = nullptr;
    unsigned long long *part = nullptr;
    auto take = [&](void **ptr, size_t bytes) {
        return cudaMallocFromPoolAsync(ptr, bytes, dev.pool, stream) == cudaSuccess;
    };
    if (cnorm == nullptr) {
        if (!take(reinterpret_cast<void **>(&tmp_norm), static_cast<size_t>(K) * 4))
            return KMASSIGN_ERR_CUDA;
        if (kma::launch_norms(C, K, D, tmp_norm, stream) != cudaSuccess)
            rc = KMASSIGN_ERR_CUDA;
        cnorm = tmp_norm;
    }
    if (rc == KMASSIGN_OK && distances) {
        if (!take(reinterpret_cast<void **>(&xnorm), static_cast<size_t>(N) * 4) ||
            kma::launch_norms(X, N, D, xnorm, stream) != cudaSuccess)
            rc = KMASSIGN_ERR_CUDA;
    }
    const int64_t row_split = split_first_row(plan);
    const int64_t n_split = plan.ksplit > 1 ? N - row_split : 0;
    if (rc == KMASSIGN_OK && n_split > 0 &&
        !take(reinterpret_cast<void **>(&part),
              static_cast<size_t>(n_split) * plan.ksplit * list * 8))
        rc = KMASSIGN_ERR_CUDA;
    if (rc == KMASSIGN_OK) {
        AssignParams p = make_params(plan, cnorm, idx, score, part, N, K, D);
        p.topk = k;
        p.xnorm = xnorm;
        if (kma::launch_topk(p.kblocks, list, p, xmap, cmap, plan.grid, plan.smem, stream) !=
            cudaSuccess)
            rc = KMASSIGN_ERR_CUDA;
        else if (part != nullptr &&
                 kma::launch_topk_merge(list, part, n_split, plan.ksplit, k,
                                        xnorm ? xnorm + row_split : nullptr, idx + row_split * k,
                                        score ? score + row_split * k : nullptr,
                                        stream) != cudaSuccess)
            rc = KMASSIGN_ERR_CUDA;
    }
    for (void *t : {static_cast<void *>(part), static_cast<void *>(xnorm),
                    static_cast<void *>(tmp_norm)})
        if (t != nullptr && cudaFreeAsync(t, stream) != cudaSuccess)
            rc = KMASSIGN_ERR_CUDA;
    return rc;
}

}  // namespace

// ---------------------------------------------------------------------------
// The update step and the Lloyd loop.

namespace {

int check_update_args(const void *X, const int32_t *idx, int64_t N, int64_t K, int64_t D,
                      const float *sums, const int32_t *counts)
{
    int rc = check_shape(N, K, D);
    if (rc != KMASSIGN_OK)
        return rc;
    if (N > 0 && (X == nullptr || idx == nullptr))
        return KMASSIGN_ERR_NULL;
    if (sums == nullptr || counts == nullptr)
        return KMASSIGN_ERR_NULL;
    if ((X && !aligned(X, 16)) || (idx && !aligned(idx, 4)) || !aligned(sums, 16) ||
        !aligned(counts, 4))
        return KMASSIGN_ERR_ALIGN;
    return KMASSIGN_OK;
}

// Below this many X elements the single atomic launch beats the sort's five
// (measured on GB300: at N * D = 2^23, 19 us atomic against 31 us sorted).
constexpr int64_t kSortedUpdateMinElems = int64_t(1) << 24;

int run_update(const void *X, const int32_t *idx, int64_t N, int64_t K, int64_t D, float *sums,
               int32_t *counts, int method, cudaStream_t stream)
{
    int rc = check_update_args(X, idx, N, K, D, sums, counts);
    if (rc != KMASSIGN_OK)
        return rc;
    if (method < 0 || method > 2)
        return KMASSIGN_ERR_ARG;
    if (N == 0)
        return KMASSIGN_OK;
    const void *ptrs[4] = {X, idx, sums, counts};
    if ((rc = check_device_ptrs(ptrs, 4)) != KMASSIGN_OK)
        return rc;
    DeviceInfo dev;
    if ((rc = current_device_info(&dev)) != KMASSIGN_OK)
        return rc;
    if (method == 0)
        method = N * D >= kSortedUpdateMinElems ? 2 : 1;
    if (method == 1) {
        if (kma::launch_update(X, idx, N, K, D, sums, counts, dev.sms, stream) != cudaSuccess)
            return KMASSIGN_ERR_CUDA;
        return KMASSIGN_OK;
    }
    void *scratch = nullptr;
    if (cudaMallocFromPoolAsync(&scratch, kma::update_sorted_scratch_bytes(N, K), dev.pool,
                                stream) != cudaSuccess)
        return KMASSIGN_ERR_CUDA;
    if (kma::launch_update_sorted(X, idx, N, K, D, sums, counts, scratch, dev.sms, stream) !=
        cudaSuccess)
        rc = KMASSIGN_ERR_CUDA;
    if (cudaFreeAsync(scratch, stream) != cudaSuccess)
        rc = KMASSIGN_ERR_CUDA;
    return rc;
}

int run_centroids(const float *sums, const int32_t *counts, const void *C_old, int64_t K,
                  int64_t D, void *C_new, float *means, cudaStream_t stream)
{
    int rc = check_shape(0, K, D);
    if (rc != KMASSIGN_OK)
        return rc;
    if (sums == nullptr || counts == nullptr || C_old == nullptr || C_new == nullptr)
        return KMASSIGN_ERR_NULL;
    if (!aligned(sums, 16) || !aligned(counts, 4) || !aligned(C_old, 16) || !aligned(C_new, 16) ||
        (means && !aligned(means, 16)))
        return KMASSIGN_ERR_ALIGN;
    const void *ptrs[5] = {sums, counts, C_old, C_new, means};
    if ((rc = check_device_ptrs(ptrs, 5)) != KMASSIGN_OK)
        return rc;
    if (kma::launch_centroids(sums, counts, C_old, K, D, C_new, means, stream) != cudaSuccess)
        return KMASSIGN_ERR_CUDA;
    return KMASSIGN_OK;
}

}  // namespace

extern "C" {

int kmassign_update(const void *X, const int32_t *idx, int64_t N, int64_t K, int64_t D,
                    float *sums, int32_t *counts, void *stream)
{
    DeviceRestore restore;
    return run_update(X, idx, N, K, D, sums, counts, 0, static_cast<cudaStream_t>(stream));
}

int kmassign_update_ex(const void *X, const int32_t *idx, int64_t N, int64_t K, int64_t D,
                       float *sums, int32_t *counts, int method, void *stream)
{
    DeviceRestore restore;
    return run_update(X, idx, N, K, D, sums, counts, method, static_cast<cudaStream_t>(stream));
}

int kmassign_centroids(const float *sums, const int32_t *counts, const void *C_old, int64_t K,
                       int64_t D, void *C_new, float *means, void *stream)
{
    DeviceRestore restore;
    return run_centroids(sums, counts, C_old, K, D, C_new, means,
                         static_cast<cudaStream_t>(stream));
}

int kmassign_lloyd(const void *X, void *C, int64_t N, int64_t K, int64_t D, int iters,
                   int32_t *idx, void *stream)
{
    DeviceRestore restore;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int rc = check_shape(N, K, D);
    if (rc != KMASSIGN_OK)
        return rc;
    if (iters < 0)
        return KMASSIGN_ERR_ARG;
    if (N == 0 || iters == 0)
        return KMASSIGN_OK;
    if (X == nullptr || C == nullptr || idx == nullptr)
        return KMASSIGN_ERR_NULL;
    if (!aligned(X, 16) || !aligned(C, 16) || !aligned(idx, 4))
        return KMASSIGN_ERR_ALIGN;
    const void *ptrs[3] = {X, C, idx};
    if ((rc = check_device_ptrs(ptrs, 3)) != KMASSIGN_OK)
        return rc;
    DeviceInfo dev;
    if ((rc = current_device_info(&dev)) != KMASSIGN_OK)
        return rc;
    float *sums = nullptr;
    int32_t *counts = nullptr;
    const size_t sum_bytes = static_cast<size_t>(K) * D * 4;
    // padded to whole 16-byte groups: the sorted update scans it with 16-byte loads
    const size_t count_bytes = static_cast<size_t>(kma::update_padded_bins(K)) * 4;
    if (cudaMallocFromPoolAsync(reinterpret_cast<void **>(&sums), sum_bytes, dev.pool, s) !=
            cudaSuccess ||
        cudaMallocFromPoolAsync(reinterpret_cast<void **>(&counts), count_bytes, dev.pool, s) !=
            cudaSuccess) {
        if (sums != nullptr)
            cudaFreeAsync(sums, s);
        return KMASSIGN_ERR_CUDA;
    }
    void *scratch = nullptr;   // the sorted update's temporaries, when it is used
    if (N * D >= kSortedUpdateMinElems &&
        cudaMallocFromPoolAsync(&scratch, kma::update_sorted_scratch_bytes(N, K), dev.pool, s) !=
            cudaSuccess)
        rc = KMASSIGN_ERR_CUDA;
    for (int it = 0; rc == KMASSIGN_OK && it < iters; ++it) {
        if (cudaMemsetAsync(counts, 0, count_bytes, s) != cudaSuccess) {
            rc = KMASSIGN_ERR_CUDA;
            break;
        }
        // assignment with the current centroids (norms computed inside); with
        // the sorted update it also counts the points per centroid as it
        // stores idx, so the update starts from the scan ...
        rc = run_assign(X, C, nullptr, N, K, D, idx, nullptr, 0, 0, 0, 0, s,
                        scratch != nullptr ? counts : nullptr);
        if (rc != KMASSIGN_OK)
            break;
        // ... then the means of the assigned points replace them in place
        if (cudaMemsetAsync(sums, 0, sum_bytes, s) != cudaSuccess) {
            rc = KMASSIGN_ERR_CUDA;
            break;
        }
        const cudaError_t upd =
            scratch != nullptr
                ? kma::launch_update_sorted_counted(X, idx, N, K, D, sums, counts, scratch,
                                                    dev.sms, s)
                : kma::launch_update(X, idx, N, K, D, sums, counts, dev.sms, s);
        if (upd != cudaSuccess ||
            kma::launch_centroids(sums, counts, C, K, D, C, nullptr, s) != cudaSuccess)
            rc = KMASSIGN_ERR_CUDA;
    }
    if (scratch != nullptr && cudaFreeAsync(scratch, s) != cudaSuccess)
        rc = KMASSIGN_ERR_CUDA;
    if (cudaFreeAsync(sums, s) != cudaSuccess || cudaFreeAsync(counts, s) != cudaSuccess)
        rc = KMASSIGN_ERR_CUDA;
    return rc;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// kmassign_noalloc: the assignment call for callers that must not allocate.
//
// Some callers cannot have a library allocate device memory behind their
// back: a host framework that hands a plugin only its buffers and a stream
// and owns every byte of device memory, or a service that fixes its memory
// budget at start-up because cudaMalloc/cudaFree can synchronise the device
// and stall other work.  For them, the two temporaries of kmassign (the norm
// buffer when cnorm is NULL, and the packed keys of a split centroid range)
// live in the file-scope array below instead of the stream-ordered allocator.
// Every GPU that loads this library holds the array until the process exits.
constexpr int64_t kNoAllocNormMax = int64_t(1) << 20;   // K, when cnorm is NULL
constexpr int64_t kNoAllocKeyMax = int64_t(1) << 18;    // N, for a split centroid range
constexpr size_t kNoAllocNormBytes = static_cast<size_t>(kNoAllocNormMax) * 4;
// the keys and, after them, one arrival counter per 128 split points
constexpr size_t kNoAllocBytes =
    kNoAllocNormBytes + static_cast<size_t>(kNoAllocKeyMax) * 8 + kNoAllocKeyMax / 128 * 4;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocBytes];

namespace {

void *g_noalloc_addr[kMaxDevices] = {};

// Device address of the scratch array on the current device, looked up once
// per device.  The array's name in host code is only a host-side handle.
int noalloc_scratch(unsigned char **out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return KMASSIGN_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mutex);
    if (g_noalloc_addr[dev] == nullptr) {
        void *ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || ptr == nullptr) {
            cudaGetLastError();
            return KMASSIGN_ERR_CUDA;
        }
        g_noalloc_addr[dev] = ptr;
    }
    *out = static_cast<unsigned char *>(g_noalloc_addr[dev]);
    return KMASSIGN_OK;
}

int run_assign_noalloc(const void *X, const void *C, const float *cnorm, int64_t N, int64_t K,
                       int64_t D, int32_t *idx, float *minscore, cudaStream_t stream)
{
    int rc = check_shape(N, K, D);
    if (rc != KMASSIGN_OK)
        return rc;
    if (N == 0)
        return KMASSIGN_OK;
    if (X == nullptr || C == nullptr || idx == nullptr)
        return KMASSIGN_ERR_NULL;
    if (!aligned(X, 16) || !aligned(C, 16) || (cnorm && !aligned(cnorm, 16)) || !aligned(idx, 4) ||
        (minscore && !aligned(minscore, 4)))
        return KMASSIGN_ERR_ALIGN;
    if (cnorm == nullptr && K > kNoAllocNormMax)
        return KMASSIGN_ERR_SCRATCH;
    const void *ptrs[5] = {X, C, cnorm, idx, minscore};
    if ((rc = check_device_ptrs(ptrs, 5)) != KMASSIGN_OK)
        return rc;

    DeviceInfo dev;
    if ((rc = current_device_info(&dev)) != KMASSIGN_OK)
        return rc;
    int dev_id = 0;
    cudaGetDevice(&dev_id);
    // The automatic plan, unless it needs memory this entry point does not
    // have: a CTA pair that folds the norms reads a fold operand from global
    // memory (plan without CTA pairs instead), and a split centroid range
    // over more points than the array's keys hold (plan without a split).
    // Plans come from the same cache as kmassign's.
    const int kblocks = static_cast<int>(cdiv(D, kma::kKBlock));
    auto needs_operand = [&](const Plan &pl) {
        return pl.v.pair && kma::assign_folds(pl.v, kblocks);
    };
    auto too_many_keys = [&](const Plan &pl) {
        return pl.ksplit > 1 && N - split_first_row(pl) > kNoAllocKeyMax;
    };
    Plan plan;
    int ksplit = 0;
    bool no_pair = false;
    for (int pass = 0; pass < 3; ++pass) {
        if ((rc = cached_plan(N, K, D, dev, dev_id, ksplit, 0, 0, 0, &plan, false, no_pair)) !=
            KMASSIGN_OK)
            return rc;
        if (needs_operand(plan))
            no_pair = true;
        else if (too_many_keys(plan))
            ksplit = 1;
        else
            break;
    }
    if (needs_operand(plan) || too_many_keys(plan))
        return KMASSIGN_ERR_ARG;   // unreachable: the last pass excludes both

    CUtensorMap xmap, cmap;
    if (!encode_map(&xmap, X, static_cast<uint64_t>(N), static_cast<uint64_t>(D), kma::kTileM) ||
        !encode_map(&cmap, C, static_cast<uint64_t>(K), static_cast<uint64_t>(D),
                    c_box_rows(plan)))
        return KMASSIGN_ERR_CUDA;

    unsigned char *scratch = nullptr;
    if ((rc = noalloc_scratch(&scratch)) != KMASSIGN_OK)
        return rc;
    // The array keeps the previous call's contents: the preparation launch
    // writes every norm the kernel reads and resets the split rows' keys and
    // counters.
    float *norms = cnorm == nullptr ? reinterpret_cast<float *>(scratch) : nullptr;
    const int64_t row_split = split_first_row(plan);
    const int64_t n_split = plan.ksplit > 1 ? N - row_split : 0;
    unsigned char *split = n_split > 0 ? scratch + kNoAllocNormBytes : nullptr;
    const size_t split_bytes = n_split > 0 ? kma::split_scratch_bytes(n_split) : 0;
    bool prepped = false;
    if ((norms != nullptr || split != nullptr) &&
        kma::launch_prep(C, K, D, cnorm, norms, nullptr, split, split_bytes, stream, &prepped) !=
            cudaSuccess)
        return KMASSIGN_ERR_CUDA;
    AssignParams p = make_params(plan, cnorm != nullptr ? cnorm : norms, idx, minscore,
                                 reinterpret_cast<unsigned long long *>(split), N, K, D);
    if (split != nullptr)
        p.counters = reinterpret_cast<uint32_t *>(split + kma::split_counter_offset(n_split));
    const CUtensorMap no_fold{};
    if (kma::launch_assign(plan.v, p.kblocks, p, xmap, cmap, no_fold, plan.grid, plan.smem,
                           stream, prepped) != cudaSuccess)
        return KMASSIGN_ERR_CUDA;
    return KMASSIGN_OK;
}

}  // namespace

extern "C" {

int kmassign_noalloc(const void *X, const void *C, const float *cnorm, int64_t N, int64_t K,
                     int64_t D, int32_t *idx, float *minscore, void *stream)
{
    DeviceRestore restore;
    return run_assign_noalloc(X, C, cnorm, N, K, D, idx, minscore,
                              static_cast<cudaStream_t>(stream));
}

int kmassign_norms(const void *C, int64_t K, int64_t D, float *cnorm, void *stream)
{
    DeviceRestore restore;
    int rc = check_shape(0, K, D);
    if (rc != KMASSIGN_OK)
        return rc;
    if (C == nullptr || cnorm == nullptr)
        return KMASSIGN_ERR_NULL;
    if (!aligned(C, 16) || !aligned(cnorm, 4))
        return KMASSIGN_ERR_ALIGN;
    const void *ptrs[2] = {C, cnorm};
    if ((rc = check_device_ptrs(ptrs, 2)) != KMASSIGN_OK)
        return rc;
    if (kma::launch_norms(C, K, D, cnorm, static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return KMASSIGN_ERR_CUDA;
    return KMASSIGN_OK;
}

int kmassign(const void *X, const void *C, const float *cnorm, int64_t N, int64_t K, int64_t D,
             int32_t *idx, float *minscore, void *stream)
{
    DeviceRestore restore;
    return run_assign(X, C, cnorm, N, K, D, idx, minscore, 0, 0, 0, 0,
                      static_cast<cudaStream_t>(stream));
}

int kmassign_ex(const void *X, const void *C, const float *cnorm, int64_t N, int64_t K, int64_t D,
                int32_t *idx, float *minscore, int ksplit, int rows_per_cta,
                int centroids_per_tile, int consumer_warps, void *stream)
{
    DeviceRestore restore;
    return run_assign(X, C, cnorm, N, K, D, idx, minscore, ksplit, rows_per_cta,
                      centroids_per_tile, consumer_warps, static_cast<cudaStream_t>(stream));
}

int kmassign_topk(const void *X, const void *C, const float *cnorm, int64_t N, int64_t K,
                  int64_t D, int32_t k, int32_t *idx, float *score, int32_t distances,
                  void *stream)
{
    DeviceRestore restore;
    return run_topk(X, C, cnorm, N, K, D, k, idx, score, distances, 0,
                    static_cast<cudaStream_t>(stream));
}

int kmassign_topk_ex(const void *X, const void *C, const float *cnorm, int64_t N, int64_t K,
                     int64_t D, int32_t k, int32_t *idx, float *score, int32_t distances,
                     int32_t ksplit, void *stream)
{
    DeviceRestore restore;
    return run_topk(X, C, cnorm, N, K, D, k, idx, score, distances, ksplit,
                    static_cast<cudaStream_t>(stream));
}

}  // extern "C"

namespace {

// kmassign_plan_ex and kmassign_plan_for: the forcing arguments' checks, the
// planner, and the plan in the 9-value layout.
int plan_to_out9(int64_t N, int64_t K, int64_t D, const DeviceInfo *dev_or_null, int ksplit,
                 int rows_per_cta, int centroids_per_tile, int consumer_warps, int32_t *out9)
{
    if (out9 == nullptr)
        return KMASSIGN_ERR_NULL;
    int rc = check_shape(N, K, D);
    if (rc != KMASSIGN_OK)
        return rc;
    if (ksplit == -1 || (rows_per_cta != 0 && rows_per_cta != 128 && rows_per_cta != 256) ||
        (centroids_per_tile != 0 && centroids_per_tile != 128 && centroids_per_tile != 256) ||
        (consumer_warps != 0 && consumer_warps != 4 && consumer_warps != 8 &&
         consumer_warps != 16))
        return KMASSIGN_ERR_ARG;
    DeviceInfo dev;
    if (dev_or_null != nullptr)
        dev = *dev_or_null;
    else if ((rc = current_device_info(&dev)) != KMASSIGN_OK)
        return rc;
    Plan plan;
    if ((rc = make_plan(std::max<int64_t>(N, 1), K, D, dev, ksplit, rows_per_cta,
                        centroids_per_tile, consumer_warps, false, &plan)) != KMASSIGN_OK)
        return rc;
    out9[0] = plan.ksplit;
    out9[1] = (plan.v.pair ? 2 : plan.v.sub) * kma::kTileM;
    out9[2] = plan.v.nt;
    out9[3] = plan.grid;
    out9[4] = plan.stages;
    out9[5] = plan.xbufs;
    out9[6] = plan.full_units;
    out9[7] = plan.rowtiles - plan.split_row0;
    out9[8] = 4 * plan.v.sub * plan.v.ch;
    return KMASSIGN_OK;
}

}  // namespace

extern "C" {

int kmassign_plan_ex(int64_t N, int64_t K, int64_t D, int ksplit, int rows_per_cta,
                     int centroids_per_tile, int consumer_warps, int32_t *out9)
{
    return plan_to_out9(N, K, D, nullptr, ksplit, rows_per_cta, centroids_per_tile,
                        consumer_warps, out9);
}

int kmassign_plan_for(int64_t N, int64_t K, int64_t D, int sms, int smem_per_block,
                      int pair_clusters, int ksplit, int rows_per_cta, int centroids_per_tile,
                      int consumer_warps, int32_t *out9)
{
    if (sms < 1 || smem_per_block < 0 || pair_clusters < 0)
        return KMASSIGN_ERR_ARG;
    DeviceInfo dev;
    dev.ready = true;
    dev.sms = sms;
    dev.smem_optin = smem_per_block;
    dev.pair_clusters = std::min(pair_clusters, sms / 2);
    return plan_to_out9(N, K, D, &dev, ksplit, rows_per_cta, centroids_per_tile, consumer_warps,
                        out9);
}

int kmassign_plan(int64_t N, int64_t K, int64_t D, int32_t *out9)
{
    return kmassign_plan_ex(N, K, D, 0, 0, 0, 0, out9);
}

int kmassign_set_wait_timeout(uint64_t ns)
{
    g_wait_timeout_ns.store(ns == 0 ? kDefaultTimeoutNs : ns);
    return KMASSIGN_OK;
}

int kmassign_check(void *stream)
{
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return KMASSIGN_ERR_CUDA;
    int code = 0, code_topk = 0;
    if (kma::status_read_and_clear(&code) != cudaSuccess ||
        kma::topk_status_read_and_clear(&code_topk) != cudaSuccess)
        return KMASSIGN_ERR_CUDA;
    return code != 0 ? code : code_topk;
}

const char *kmassign_strerror(int code)
{
    switch (code) {
    case KMASSIGN_OK:
        return "success";
    case KMASSIGN_ERR_NULL:
        return "a required pointer is NULL";
    case KMASSIGN_ERR_ALIGN:
        return "X and C (and cnorm) must be 16-byte aligned; idx and minscore 4-byte aligned";
    case KMASSIGN_ERR_SHAPE:
        return "shape out of range: need 0 <= N < 2^31 and 1 <= K < 2^31";
    case KMASSIGN_ERR_UNSUPPORTED_D:
        return "unsupported D: need a multiple of 16 in [16, 256]";
    case KMASSIGN_ERR_CUDA:
        return "a CUDA runtime or driver call failed";
    case KMASSIGN_ERR_TIMEOUT:
        return "a bounded pipeline wait inside a kernel ran out; the kernel drained and returned";
    case KMASSIGN_ERR_NOT_DEVICE:
        return "a pointer is not device memory of the current device";
    case KMASSIGN_ERR_DEBUG_CHECK:
        return "a device-side consistency check of the debug build (KMASSIGN_DEBUG) failed";
    case KMASSIGN_ERR_NOT_HOST:
        return "kmassign_host: a pointer is device memory, not host memory";
    case KMASSIGN_ERR_SCRATCH:
        return "kmassign_noalloc: K exceeds its static norm buffer (cnorm NULL needs K <= 1048576)";
    case KMASSIGN_ERR_ARG:
        return "invalid argument (plan values: ksplit != -1, rows_per_cta 128/256, "
               "centroids_per_tile 128/256, consumer_warps 4/8/16 matching a compiled shape; "
               "top-k: 1 <= k <= min(K, 32), distances 0 or 1)";
    default:
        return "unknown kmassign status code";
    }
}

}  // extern "C"
