// internal.h -- declarations shared by the translation units of libkmassign.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

namespace kma {

constexpr int kTileM = 128;        // points per tensor-core tile (TMEM lanes)
constexpr int kKBlock = 64;        // bf16 elements per 128-byte swizzled row
constexpr uint32_t kXTileBytes = kTileM * 128;  // one k-block of one 128-row X tile
constexpr int kMaxStages = 16;     // upper bound of the shared-memory ring
constexpr int kMaxXBufs = 2;
constexpr int kNone = 0x7fffffff;  // "no candidate yet" index

struct AssignParams {
    const float *cnorm;            // [K] fp32
    int32_t *idx;                  // [N] (direct store when ksplit == 1)
    float *minscore;               // [N] or nullptr (direct store when ksplit == 1)
    // Packed (ordered score << 32 | index) keys of the split rows, indexed by
    // row - split_row0 * rows per tile: one per row for the assignment, L per
    // (row, centroid range) for the k-nearest kernel.
    unsigned long long *keys;
    // Arrival counters of the split rows, one per group of 128 (all-ones
    // before the launch): with more than two units per row, the last of a
    // group's ksplit units turns its keys into idx and minscore (two units
    // merge through the keys alone).
    uint32_t *counters;
    // Optional (the Lloyd loop): counts[idx[i]] += 1 for every point stored,
    // the update's histogram formed by the assignment itself.
    int32_t *counts;
    int32_t topk;                  // k of the k-nearest kernel (idx, minscore hold [N, k])
    const float *xnorm;            // [N] ||x||^2: the k-nearest kernel writes distances
    int32_t N, K, D;
    int32_t ksteps;                // D / 16 tensor-core k-steps
    int32_t kblocks;               // ceil(D / 64) swizzled k-blocks
    int32_t rowtiles;              // ceil(N / (128 * sub))
    int32_t full_units;            // row tiles [0, full_units) form one unit each, all of K
    int32_t split_row0;            // row tiles [split_row0, rowtiles) are split over K
    int32_t ksplit;                // centroid ranges per split row tile
    int32_t chunk_tiles;           // centroid tiles per range
    int32_t ntiles;                // ceil(K / nt)
    int32_t num_units;             // full_units + (rowtiles - split_row0) * ksplit
    int32_t stages;                // shared-memory ring depth
    int32_t stage_group;           // C stages per barrier pair (assign_stage_group)
    int32_t xbufs;                 // X tile buffers (1 or 2)
    uint64_t timeout_ns;           // bound on every pipeline wait
};

// Compiled shapes of the assignment kernel: `sub` 128-point sub-tiles per
// block, `nt` centroids per tensor-core tile, each tile's columns split over
// `ch` groups of consumer warps; `pair` kernels tile 256 points per cluster of
// two blocks.
struct Variant {
    int sub, nt, ch;
    bool pair;   // cluster of two CTAs issuing cta_group::2 MMAs (sub 1 per CTA, nt 256)
};
constexpr int kNumVariants = 7;
extern const Variant kVariants[kNumVariants];

size_t assign_smem_bytes(const Variant &v, int kblocks, int stages, int xbufs);
cudaError_t assign_prepare(const Variant &v, int kblocks, size_t smem_bytes);
// Clusters of the pair kernel that can be resident at once.
cudaError_t assign_max_clusters(const Variant &v, int kblocks, size_t smem, int *clusters);
// fmap: the fold operand's tensor map, read only by kernels that fold the
// norms into the MMA through it (assign_folds on a CTA pair); others ignore it.
// after_prep: the launch directly before this one in the stream is the
// call's preparation kernel.  The assignment kernel is then launched as its
// programmatic dependent: its set-up (barriers, tensor memory, the X copies)
// overlaps the preparation, and only the warps that read the preparation's
// outputs (norms, fold operand, split keys) wait for it.  Everything queued
// before the preparation kernel has completed when that kernel starts, so
// the inputs are ready either way.
cudaError_t launch_assign(const Variant &v, int kblocks, const AssignParams &p,
                          const CUtensorMap &xmap, const CUtensorMap &cmap,
                          const CUtensorMap &fmap, int grid, size_t smem_bytes,
                          cudaStream_t stream, bool after_prep = false);
// Whether the shape's kernel folds the norms into the MMA (every shape at up
// to two k-blocks, D <= 128).
bool assign_folds(const Variant &v, int kblocks);
// The CTA pair's fold operand: fold_operand_blocks(K) blocks of 128
// centroids, 4 KiB each ([K half][128 rows][16 B] bf16), written from the
// norms by launch_prep (rows past K hold NaN).
int64_t fold_operand_blocks(int64_t K);
// C stages per barrier pair of the shape: a folding CTA pair groups the
// k-blocks of a tile (its ring depth is a multiple of this), others use 1.
int assign_stage_group(const Variant &v, int kblocks);
size_t fold_operand_bytes(int64_t K);

// The k-nearest kernel: one shape (256 points x 128 centroids per tile, 8
// consumer warps), a sorted list of `list` in {4, 8, 16, 32} >= k candidates
// per point.
extern const Variant kTopkVariant;
int topk_list_size(int k);
size_t topk_smem_bytes(int kblocks, int stages, int xbufs);
cudaError_t topk_prepare(int kblocks, int list, size_t smem_bytes);
cudaError_t launch_topk(int kblocks, int list, const AssignParams &p, const CUtensorMap &xmap,
                        const CUtensorMap &cmap, int grid, size_t smem_bytes, cudaStream_t stream);
// Merge the per-range lists of `rows` split points ([rows][ksplit][list]
// keys) into the k best; idx, score (may be NULL) and xnorm (NULL: scores,
// else distances) point at the first split point.
cudaError_t launch_topk_merge(int list, const unsigned long long *part, int64_t rows, int ksplit,
                              int k, const float *xnorm, int32_t *idx, float *score,
                              cudaStream_t stream);

cudaError_t launch_norms(const void *C, int64_t K, int64_t D, float *cnorm, cudaStream_t stream);
// The update step: atomic (one launch, L2-atomic bound) or sorted (counting
// sort by centroid, then run reductions; needs update_sorted_scratch_bytes of
// device scratch, 8-byte aligned).
cudaError_t launch_update(const void *X, const int32_t *idx, int64_t N, int64_t K, int64_t D,
                          float *sums, int32_t *counts, int sms, cudaStream_t stream);
size_t update_sorted_scratch_bytes(int64_t N, int64_t K);
cudaError_t launch_update_sorted(const void *X, const int32_t *idx, int64_t N, int64_t K,
                                 int64_t D, float *sums, int32_t *counts, void *scratch, int sms,
                                 cudaStream_t stream);
// The sorted update when counts already holds the histogram of idx (the
// assignment formed it): counts has update_padded_bins(K) entries, 16-byte
// aligned, zero past K; only sums is accumulated.
int64_t update_padded_bins(int64_t K);
cudaError_t launch_update_sorted_counted(const void *X, const int32_t *idx, int64_t N, int64_t K,
                                         int64_t D, float *sums, const int32_t *counts,
                                         void *scratch, int sms, cudaStream_t stream);
cudaError_t launch_centroids(const float *sums, const int32_t *counts, const void *C_old, int64_t K,
                             int64_t D, void *C_new, float *means, cudaStream_t stream);
// score[i] = max(xnorm[i] + score[i], 0) (NaN kept): distances from scores.
cudaError_t launch_add_norms(float *score, const float *xnorm, int64_t N, cudaStream_t stream);
// One launch before an assignment kernel, doing any of: the norms of C into
// cnorm_out (when cnorm_in is NULL), the fold operand from the norms (when
// fold is not NULL), and fill_bytes (a multiple of 16) of all-ones at fill.
// *launched tells whether a kernel was launched (nothing to do: none).  The
// kernel lets the next launch in the stream start early (see launch_assign).
cudaError_t launch_prep(const void *C, int64_t K, int64_t D, const float *cnorm_in,
                        float *cnorm_out, void *fold, void *fill, size_t fill_bytes,
                        cudaStream_t stream, bool *launched);
// Bytes of packed keys and arrival counters for n_split split rows (a
// multiple of 16; the counters start at byte split_counter_offset).
size_t split_scratch_bytes(int64_t n_split);
size_t split_counter_offset(int64_t n_split);

// Read and clear the device status word of the assignment kernels, and of
// the k-nearest kernels (0 or a kmassign_status code).
cudaError_t status_read_and_clear(int *code);
cudaError_t topk_status_read_and_clear(int *code);

// For the host-buffer path (kmassign status codes): the stream-ordered memory
// pool of the current device, and the points one full wave of the automatic
// assignment plan covers (thread blocks in flight, a CTA pair counted once,
// times points per block).
int library_pool(cudaMemPool_t *pool);
int assign_wave_rows(int64_t N, int64_t K, int64_t D, int64_t *rows);

}  // namespace kma
