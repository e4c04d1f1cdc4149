/*
 * kmassign.h -- C ABI of libkmassign, the k-means assignment step on one
 * NVIDIA GB300 (sm_103a).
 *
 * The operation (flashlib PR #22 "Optimize Blackwell k-means assignment
 * reduction", Summary): for every point x_i, form the scores of all
 * centroids from their dot products with x_i, apply the centroid norms, and
 * select the winning centroid, ties going to the lowest index:
 *
 *     s_ij   = ||c_j||^2 - 2 * x_i . c_j
 *     idx[i] = the lowest j whose s_ij is minimal
 *
 * ||x_i||^2 is the same for every j, so idx[i] is the centroid nearest to
 * x_i in Euclidean distance.  Ordering of scores: -0 equals +0; NaN is above
 * every number (a NaN score never beats a number, +inf included).  A row whose
 * scores are all NaN (for example a row holding a NaN) gets idx 0 and minscore
 * NaN; the pages test NaN rows but fix no convention, this is the one chosen.
 *
 * Arithmetic (what the GPU computes): x and c are bf16; ||c_j||^2 is an fp32
 * sum of exact bf16 squares (or the caller's cnorm).  The tensor cores sum in
 * fp32, in an order the hardware fixes:
 *   - D <= 128: the accumulator takes x_i . c_j and then -||c_j||^2 / 2,
 *     entered as three bf16 parts h + m + l that carry all 24 bits of the
 *     fp32 value (one more K = 16 tensor-core step, A = ones), so it holds
 *     t_ij = x_i . c_j - ||c_j||^2 / 2; the winner is the largest t and
 *     s_ij = -2 t_ij (exact);
 *   - D > 128: the accumulator holds x_i . c_j and s_ij = fmaf(-2, dot,
 *     cnorm_j) in fp32.
 * Which of the two applies depends on D alone: every plan, batch size and
 * split gives a point the same idx and minscore bits.  On integer-valued
 * inputs whose sums stay below 2^24 every step is exact.
 *
 * Layout: every matrix is row-major and contiguous, D innermost.  Row pitch
 * is D * 2 bytes.  All pointers are device pointers (cudaMalloc, the stream
 * allocator or PyTorch CUDA tensors); host or unregistered pointers are
 * rejected with KMASSIGN_ERR_NOT_DEVICE before anything is launched.  The
 * exception is kmassign_host (and _ex), which takes host buffers.
 *
 * Devices: the pointers' device is made current for the launches; the calling
 * thread's current device is restored before every entry point returns.
 *
 * Ownership: the caller owns every buffer it passes.  The library keeps no
 * pointer after a call returns.  Temporaries (the norm buffer when cnorm is
 * NULL, and the packed-key workspace when the centroid range is split across
 * thread blocks) are stream-ordered allocations on the caller's stream from a
 * memory pool the library creates per device; the pool keeps up to 1 GiB
 * reserved between calls so that repeated calls do not re-map memory.
 *
 * Execution: every call is asynchronous on `stream` (a cudaStream_t passed as
 * void*; NULL is the legacy default stream) and never synchronises the host,
 * except kmassign_check and the host-buffer call kmassign_host, which return
 * once their stream's work is done.
 * Argument errors are returned before any launch; launch errors are returned
 * as KMASSIGN_ERR_CUDA.  The pipeline waits inside the main kernel are
 * bounded in time: a wait that runs out records KMASSIGN_ERR_TIMEOUT in a
 * device status word, the kernel drains its copies, frees its tensor memory
 * and returns; kmassign_check() reports it.  Calls on one stream are ordered;
 * calls on different streams that write the same outputs race.
 */
#ifndef KMASSIGN_H
#define KMASSIGN_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum kmassign_status {
    KMASSIGN_OK = 0,
    KMASSIGN_ERR_NULL = -1,          /* a required pointer is NULL */
    KMASSIGN_ERR_ALIGN = -2,         /* X or C not 16-byte aligned, or an output not 4-byte aligned */
    KMASSIGN_ERR_SHAPE = -3,         /* N < 0, K < 1, or N or K >= 2^31 */
    KMASSIGN_ERR_UNSUPPORTED_D = -4, /* D not a multiple of 16, or outside [16, 256] */
    KMASSIGN_ERR_CUDA = -5,          /* a CUDA runtime/driver call failed */
    KMASSIGN_ERR_TIMEOUT = -6,       /* a bounded wait inside a kernel ran out */
    KMASSIGN_ERR_NOT_DEVICE = -7,    /* a pointer is not device memory */
    KMASSIGN_ERR_ARG = -8,           /* an invalid plan value, k or flag */
    KMASSIGN_ERR_SCRATCH = -9,       /* too large for kmassign_noalloc's static scratch */
    KMASSIGN_ERR_NOT_HOST = -10,     /* kmassign_host: a pointer is device memory */
    KMASSIGN_ERR_DEBUG_CHECK = -11   /* a device-side check of a KMASSIGN_DEBUG build failed */
};

/*
 * cnorm[j] = ||c_j||^2 for j in [0, K)  (Summary: "applying centroid norms").
 *   C      device, bf16 [K, D] row-major, 16-byte aligned
 *   cnorm  device, fp32 [K], 4-byte aligned, written
 * fp32 sum of the exact bf16 squares, in a fixed order (deterministic).
 */
int kmassign_norms(const void *C, int64_t K, int64_t D, float *cnorm, void *stream);

/*
 * idx[i] = argmin_j (||c_j||^2 - 2 x_i . c_j), lowest index on ties.
 *   X         device, bf16 [N, D] row-major, 16-byte aligned
 *   C         device, bf16 [K, D] row-major, 16-byte aligned
 *   cnorm     device fp32 [K] from kmassign_norms, or NULL (then computed
 *             inside the call into a stream-ordered temporary)
 *   N         0 <= N < 2^31 (N == 0 launches nothing and returns OK;
 *             X and idx may then be NULL)
 *   K         1 <= K < 2^31
 *   D         multiple of 16 in [16, 256]
 *   idx       device int32 [N], written
 *   minscore  device fp32 [N] or NULL; when given, the winning score s
 *             computed as above, with -0 written as +0, or NaN for an
 *             all-NaN row
 * The result does not depend on how the work is tiled or split, nor on the
 * other points of the call: every plan returns the same idx and minscore
 * bits, and a point assigned alone gets the bits it gets in any batch.
 */
int kmassign(const void *X, const void *C, const float *cnorm, int64_t N, int64_t K,
             int64_t D, int32_t *idx, float *minscore, void *stream);

/*
 * kmassign with an explicit plan (0 = the automatic choice for each field):
 *   ksplit              number of centroid ranges the K axis of every row
 *                       tile is split into; > 1 merges partial winners with a
 *                       64-bit atomicMin on (ordered score bits << 32 | index)
 *                       keys.  ksplit <= -2 splits only the row tiles of the
 *                       last, partial wave of thread blocks into -ksplit
 *                       ranges (wave-tail balancing); -1 is invalid
 *   rows_per_cta        128 or 256 points per work unit
 *   centroids_per_tile  128 or 256 centroids per tensor-core tile; 256 with
 *                       256 rows selects the CTA-pair kernel (two thread
 *                       blocks on two SMs share each 256x256 tile; at
 *                       D <= 128 every shape folds the norms into the MMA)
 *   consumer_warps      warps reducing the score tiles per thread block: 4
 *                       (128x128 tiles), 8 or 16 (all other shapes)
 * Same arguments, layout and errors as kmassign; a value outside these sets,
 * or a combination no compiled kernel has (or no pair of SMs can run),
 * returns KMASSIGN_ERR_ARG.  Tests
 * use it to cover every path.
 */
int kmassign_ex(const void *X, const void *C, const float *cnorm, int64_t N, int64_t K,
                int64_t D, int32_t *idx, float *minscore, int ksplit, int rows_per_cta,
                int centroids_per_tile, int consumer_warps, void *stream);

/*
 * kmassign for points, centroids and results held in HOST memory: the whole
 * assignment step end to end, host to host (the Summary's operation, with
 * the copies to and from the GPU inside the call).
 *   X         host, bf16 [N, D] row-major
 *   C         host, bf16 [K, D] row-major
 *   cnorm     host fp32 [K], or NULL (then computed on the GPU)
 *   N, K, D   as in kmassign (N == 0 does nothing and returns OK)
 *   idx       host int32 [N], written
 *   minscore  host fp32 [N] or NULL, written as in kmassign
 *   stream    the caller's stream on the calling thread's current device
 *             (NULL: the legacy default stream); the GPU work runs on it and
 *             on two streams of the library, ordered after the work already
 *             queued on it
 * Host memory may be pinned (cudaHostAlloc, cudaHostRegister), pageable or
 * managed; only pinned memory lets the copies overlap the kernels.  No
 * alignment is required.  Device pointers return KMASSIGN_ERR_NOT_HOST.
 *
 * C (and cnorm) is copied first; X follows in row slices of about N / 8
 * points, rounded to whole waves of the assignment kernel's thread blocks
 * (the first slice, whose copy nothing overlaps, is a single wave),
 * through two device buffers: the copy of one slice overlaps the assignment
 * of the previous one, and each slice's answers are copied back while the
 * next slice runs.  Each slice is one kmassign call, so the results are
 * kmassign's bits for the whole batch.  Device temporaries (C, the norms,
 * two X slices, two idx and minscore slices) come from the library's
 * stream-ordered pool and are returned before the call ends.
 *
 * Synchronous: returns once idx and minscore hold the answers and every
 * temporary is released.  A pipeline wait that ran out in one of the
 * kernels returns KMASSIGN_ERR_TIMEOUT and clears the device status word as
 * kmassign_check does.  The first call on a device creates the library's two
 * streams and events there (kept until the process exits).  Calls on one
 * device are serialised.
 */
int kmassign_host(const void *X, const void *C, const float *cnorm, int64_t N, int64_t K,
                  int64_t D, int32_t *idx, float *minscore, void *stream);

/*
 * kmassign_host with the slice size forced: rows_per_slice > 0 points per
 * slice (the last takes the rest), 0 the automatic choice above; negative
 * returns KMASSIGN_ERR_ARG.  The results do not depend on it.
 */
int kmassign_host_ex(const void *X, const void *C, const float *cnorm, int64_t N, int64_t K,
                     int64_t D, int32_t *idx, float *minscore, int64_t rows_per_slice,
                     void *stream);

/*
 * The plan kmassign would choose for (N, K, D) on the current device:
 * out[0] = ksplit of the split row tiles (1: none split), out[1] =
 * rows_per_cta, out[2] = centroids_per_tile, out[3] = thread blocks
 * launched, out[4] = shared-memory ring stages, out[5] = X tile buffers,
 * out[6] = row tiles processed whole, out[7] = row tiles split, out[8] =
 * consumer warps.  Launches nothing.
 */
int kmassign_plan(int64_t N, int64_t K, int64_t D, int32_t *out9);

/*
 * The plan kmassign_ex would run with the same forcing arguments (same
 * meaning and errors as there; 0 leaves a field to the planner), in
 * kmassign_plan's layout.  Launches nothing.
 */
int kmassign_plan_ex(int64_t N, int64_t K, int64_t D, int ksplit, int rows_per_cta,
                     int centroids_per_tile, int consumer_warps, int32_t *out9);

/*
 * The plan kmassign_ex would run with the same forcing arguments on a
 * described device instead of the current one: sms streaming multiprocessors,
 * smem_per_block bytes of opt-in shared memory per thread block, and
 * pair_clusters two-block clusters of the CTA-pair kernel that can be
 * resident at once (0: no CTA pairs; capped at sms / 2).  Host only: makes no
 * CUDA call, so it also runs where no GPU is present (GB300: 152 SMs,
 * 232,448 bytes, 76 pairs).  Layout of out9 and errors as kmassign_plan_ex;
 * sms < 1 or a negative size returns KMASSIGN_ERR_ARG.
 */
int kmassign_plan_for(int64_t N, int64_t K, int64_t D, int sms, int smem_per_block,
                      int pair_clusters, int ksplit, int rows_per_cta, int centroids_per_tile,
                      int consumer_warps, int32_t *out9);

/*
 * Synchronise `stream`, then report and clear the device status word:
 * KMASSIGN_ERR_TIMEOUT if a kernel gave up on a bounded wait since the last
 * check, KMASSIGN_ERR_CUDA if the stream reports an error, else KMASSIGN_OK.
 * The status word belongs to the current device and is shared by every
 * stream and thread of the process: a timeout raised by a kernel on one
 * stream is reported, and cleared, by a check on any stream of that device.
 */
int kmassign_check(void *stream);

/*
 * kmassign without any device allocation.  The pages have no counterpart to
 * this call; it exists for callers that cannot let a library allocate device
 * memory while they run -- a host framework that hands a plugin only its
 * buffers and a stream and owns all device memory, or a service that fixes
 * its memory budget at start-up because cudaMalloc/cudaFree can synchronise
 * the device.
 *
 * Same arguments, layout, results (bit for bit) and errors as kmassign.  Its temporaries
 * live in one static device array of this library (6 MiB, held on every GPU
 * that loads the library until the process exits) instead of the stream
 * allocator; it calls no cudaMalloc, cudaFree or other allocating routine.
 *   - cnorm == NULL needs K <= 1,048,576 (the norms go into the array);
 *     larger K returns KMASSIGN_ERR_SCRATCH before anything is launched.
 *   - A split centroid range keeps one 8-byte key per point in the array;
 *     for N > 262,144 the call plans without a split instead.
 *   - Where kmassign would run CTA pairs that fold the norms into the MMA
 *     (every D <= 128) and read a fold operand from memory, this call plans
 *     without CTA pairs; every plan gives the same bits, so the results are
 *     still kmassign's.
 * The first call on a device does that device's set-up with it current: the
 * kernels' shared-memory attributes, the library's memory pool (used only by
 * the other entry points) and the array's device address
 * (cudaGetSymbolAddress); make that first call before any stream capture.  Every call shares the one array and overwrites
 * what the previous call left there, so calls whose work overlaps on the GPU
 * (different streams, or different host threads) race; order them on one
 * stream or synchronise between them.
 */
int kmassign_noalloc(const void *X, const void *C, const float *cnorm, int64_t N, int64_t K,
                     int64_t D, int32_t *idx, float *minscore, void *stream);

/*
 * The update step of a Lloyd iteration (the textbook step after the
 * assignment; flashlib PR #22 covers the assignment only):
 *     counts[j] += |{i : idx[i] == j}|,   sums[j][d] += sum of x_id over them
 *   X       device, bf16 [N, D] row-major, 16-byte aligned
 *   idx     device int32 [N] (ids outside [0, K) are skipped)
 *   sums    device fp32 [K, D], 16-byte aligned, accumulated into
 *   counts  device int32 [K], accumulated into
 * The caller zeroes sums and counts first, or keeps accumulating over batches
 * (or adds the results of several GPUs).  Sums are fp32 additions in an
 * unspecified order: on non-integer data their last bits can differ from run
 * to run; integer-valued data whose sums stay below 2^24 is exact.
 */
int kmassign_update(const void *X, const int32_t *idx, int64_t N, int64_t K, int64_t D,
                    float *sums, int32_t *counts, void *stream);

/*
 * kmassign_update with the method forced: 0 = automatic (by N * D), 1 =
 * atomic (every point adds its row into the sums with vector reductions; one
 * launch), 2 = sorted (a counting sort groups the points by centroid, then
 * runs of sorted points are summed in registers and added once per centroid
 * met; a temporary of 8K + 4N bytes from the library's pool).  Same
 * arguments and results as kmassign_update; another method returns
 * KMASSIGN_ERR_ARG.  Tests use it to cover both.
 */
int kmassign_update_ex(const void *X, const int32_t *idx, int64_t N, int64_t K, int64_t D,
                       float *sums, int32_t *counts, int method, void *stream);

/*
 * New centroids from kmassign_update's results: C_new[j] = bf16(sums[j] /
 * counts[j]) (fp32 division, then round to nearest even) where counts[j] > 0,
 * else C_old[j].  means (fp32 [K, D], 16-byte aligned) receives the unrounded
 * means when not NULL.  C_new may be C_old.  All pointers device memory.
 */
int kmassign_centroids(const float *sums, const int32_t *counts, const void *C_old, int64_t K,
                       int64_t D, void *C_new, float *means, void *stream);

/*
 * `iters` Lloyd iterations on the device: each assigns X to C (norms computed
 * inside) into idx, then replaces every centroid that received points by
 * their mean (kmassign_update + kmassign_centroids), in place in C.  Where
 * the update is the sorted one (N * D >= 2^24), the assignment kernel counts
 * the points per centroid as it stores idx and the update starts from those
 * counts; the results are those of the separate calls.  On return idx holds
 * the last assignment, made with the centroids before the last update.
 * Temporaries (sums, counts, norms, the sort's scratch) come from the
 * library's stream-ordered pool.  iters < 0 returns KMASSIGN_ERR_ARG.
 */
int kmassign_lloyd(const void *X, void *C, int64_t N, int64_t K, int64_t D, int iters,
                   int32_t *idx, void *stream);

/* Largest k kmassign_topk accepts. */
#define KMASSIGN_TOPK_MAX 32

/*
 * The k nearest centroids of every point, and optionally the true squared
 * distances to them.  Not part of flashlib PR #22, which selects one winner
 * per point; this widens its Summary's selection step to the k best pairs
 * (s_ij, j) under the same order as kmassign: s_ij = ||c_j||^2 - 2 x_i . c_j
 * ascending, NaN above every number, -0 equal to +0, the lower index first
 * among equal scores.  k = 1 returns kmassign's idx.
 *   X, C, cnorm, N, K, D   as in kmassign
 *   k          1 <= k <= min(K, KMASSIGN_TOPK_MAX); N * k < 2^31
 *   idx        device int32 [N, k] row-major, written: row i ascending
 *   score      device fp32 [N, k] row-major, or NULL (then distances must be
 *              0); written in idx's order:
 *                distances == 0: s_ij = -2 t_ij from an accumulator that
 *                                folds the norms in (as kmassign does at
 *                                D <= 128, here at every D; k = 1 returns
 *                                kmassign's minscore), -0 as +0, NaN for a
 *                                NaN score
 *                distances == 1: ||x_i||^2 + s_ij in fp32 with ||x_i||^2 the
 *                                fp32 sum of exact bf16 squares, a negative
 *                                result (rounding) written as 0.  For
 *                                non-finite inputs this is the same formula,
 *                                not the direct sum of (x_d - c_d)^2
 * k = 1 runs the assignment kernel (then adds ||x_i||^2 for distances).
 * Each selection uses the fp32 scores, so points whose k-th and (k+1)-th
 * scores lie within fp32 rounding of each other may pick either.  Temporaries
 * (norms, ||x||^2, partial lists of split centroid ranges) come from the
 * library's stream-ordered pool.  Errors: as kmassign; k or distances out of
 * range returns KMASSIGN_ERR_ARG, N * k >= 2^31 KMASSIGN_ERR_SHAPE,
 * distances == 1 with score NULL KMASSIGN_ERR_NULL.
 */
int kmassign_topk(const void *X, const void *C, const float *cnorm, int64_t N, int64_t K,
                  int64_t D, int32_t k, int32_t *idx, float *score, int32_t distances,
                  void *stream);

/*
 * kmassign_topk with an explicit centroid split (0 = automatic; > 1 splits
 * the K axis of every row tile into ksplit ranges whose sorted candidate
 * lists a merge kernel combines; <= -2 splits only the last, partial wave of
 * row tiles into -ksplit ranges; -1 returns KMASSIGN_ERR_ARG).  k = 1 takes
 * the assignment kernel with kmassign_ex's split.  Every split returns the
 * same results.  Tests use it to cover the merge path.
 */
int kmassign_topk_ex(const void *X, const void *C, const float *cnorm, int64_t N, int64_t K,
                     int64_t D, int32_t k, int32_t *idx, float *score, int32_t distances,
                     int32_t ksplit, void *stream);

/*
 * Bound, in nanoseconds of the GPU's global timer, on every pipeline wait in
 * the kernels launched afterwards by this process (0 restores the default,
 * 2 s).  A wait that runs out aborts its kernel cleanly and makes
 * kmassign_check() return KMASSIGN_ERR_TIMEOUT; outputs are then undefined.
 * Tests shrink it to make a timeout happen without faulting the GPU.
 */
int kmassign_set_wait_timeout(uint64_t ns);

/* Static English text for a status code (never NULL). */
const char *kmassign_strerror(int code);

#ifdef __cplusplus
}
#endif

#endif /* KMASSIGN_H */
