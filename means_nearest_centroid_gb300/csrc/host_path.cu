// host_path.cu -- kmassign_host: the assignment step for points and centroids
// held in host memory.
//
// No arithmetic of the method lives here: this file only moves data and
// orders work.  C (and the caller's norms, if any) is copied to the device
// first; X then goes over in row slices of whole waves of the assignment
// kernel, two device buffers in turn, on a copy stream of the library's,
// while the previous slice is assigned on the caller's stream; each slice's
// idx (and minscore) is copied back on a third stream as soon as it is ready,
// so the link carries the next slice's X while the kernels run.  Every
// assignment is a kmassign call, whose answers do not depend on how the points
// are batched, so the slices give the bits of one call over all points.
//
//   copy stream:    C | X0 | X1 | X2 ...            (X_s waits until the kernel
//   caller stream:      norms | A(X0) | A(X1) ...     of slice s-2 has read its
//   back stream:                 idx0 | idx1 ...      buffer)
#include "kmassign.h"
#include "internal.h"

#include <algorithm>
#include <cstdint>
#include <mutex>

namespace {

constexpr int kMaxDevices = 64;
constexpr int64_t kSlices = 8;   // aimed-for number of slices (each whole waves)

// Streams and events of the host path on one device, made by its first call
// and kept until the process exits.  The mutex serialises calls on the device
// (the call is synchronous; the events are reused from call to call).
struct HostPath {
    std::mutex mutex;
    bool ready = false;
    cudaStream_t copy = nullptr, back = nullptr;
    cudaEvent_t start = nullptr, c_in = nullptr, copy_end = nullptr, back_end = nullptr;
    cudaEvent_t landed[2] = {}, done[2] = {}, freed[2] = {};
};
HostPath g_host[kMaxDevices];

int setup(HostPath &h)
{
    if (h.ready)
        return KMASSIGN_OK;
    const unsigned ev = cudaEventDisableTiming;
    bool ok = cudaStreamCreateWithFlags(&h.copy, cudaStreamNonBlocking) == cudaSuccess &&
              cudaStreamCreateWithFlags(&h.back, cudaStreamNonBlocking) == cudaSuccess &&
              cudaEventCreateWithFlags(&h.start, ev) == cudaSuccess &&
              cudaEventCreateWithFlags(&h.c_in, ev) == cudaSuccess &&
              cudaEventCreateWithFlags(&h.copy_end, ev) == cudaSuccess &&
              cudaEventCreateWithFlags(&h.back_end, ev) == cudaSuccess;
    for (int b = 0; ok && b < 2; ++b)
        ok = cudaEventCreateWithFlags(&h.landed[b], ev) == cudaSuccess &&
             cudaEventCreateWithFlags(&h.done[b], ev) == cudaSuccess &&
             cudaEventCreateWithFlags(&h.freed[b], ev) == cudaSuccess;
    if (!ok)
        return KMASSIGN_ERR_CUDA;
    h.ready = true;
    return KMASSIGN_OK;
}

// Device memory cannot be read by the host path's copies as host memory:
// reject it (pinned, registered, pageable and managed memory are accepted).
int check_host_ptrs(const void *const *ptrs, int n)
{
    for (int i = 0; i < n; ++i) {
        if (ptrs[i] == nullptr)
            continue;
        cudaPointerAttributes a;
        if (cudaPointerGetAttributes(&a, ptrs[i]) != cudaSuccess) {
            cudaGetLastError();   // not known to CUDA: plain host memory
            continue;
        }
        if (a.type == cudaMemoryTypeDevice)
            return KMASSIGN_ERR_NOT_HOST;
    }
    return KMASSIGN_OK;
}

// Rows per slice: the caller's, else about N / kSlices rounded to whole waves
// (at least one), so that no slice but the last ends in a partly filled wave
// (run_host makes the first slice a single wave).
int64_t slice_rows(int64_t N, int64_t wave, int64_t forced)
{
    if (forced > 0)
        return std::min(forced, N);
    const int64_t share = (N + kSlices - 1) / kSlices;
    const int64_t waves = (share + wave / 2) / wave;
    return std::min(N, std::max<int64_t>(1, waves) * wave);
}

int run_host(const void *X, const void *C, const float *cnorm, int64_t N, int64_t K, int64_t D,
             int32_t *idx, float *minscore, int64_t rows_per_slice, cudaStream_t compute)
{
    if (N < 0 || N >= (int64_t(1) << 31) || K < 1 || K >= (int64_t(1) << 31))
        return KMASSIGN_ERR_SHAPE;
    if (D < 16 || D > 256 || D % 16 != 0)
        return KMASSIGN_ERR_UNSUPPORTED_D;
    if (rows_per_slice < 0)
        return KMASSIGN_ERR_ARG;
    if (N == 0)
        return KMASSIGN_OK;
    if (X == nullptr || C == nullptr || idx == nullptr)
        return KMASSIGN_ERR_NULL;
    const void *ptrs[5] = {X, C, cnorm, idx, minscore};
    int rc = check_host_ptrs(ptrs, 5);
    if (rc != KMASSIGN_OK)
        return rc;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return KMASSIGN_ERR_CUDA;
    cudaMemPool_t pool;
    int64_t wave = 1;
    if ((rc = kma::library_pool(&pool)) != KMASSIGN_OK ||
        (rc = kma::assign_wave_rows(N, K, D, &wave)) != KMASSIGN_OK)
        return rc;
    const int64_t rows = slice_rows(N, wave, rows_per_slice);
    // Nothing overlaps the first slice's copy, so unless the caller fixed the
    // slices the first one is a single wave (when the others hold more).
    const int64_t first_rows = rows_per_slice > 0 ? rows : std::min(rows, wave);

    HostPath &h = g_host[dev];
    std::lock_guard<std::mutex> lock(h.mutex);
    if ((rc = setup(h)) != KMASSIGN_OK)
        return rc;

    // Device buffers from the library's pool, in the caller's stream order.
    const size_t row_bytes = static_cast<size_t>(D) * 2;
    void *cd = nullptr, *xd = nullptr;
    float *cn = nullptr, *msd = nullptr;
    int32_t *idxd = nullptr;
    auto take = [&](void **p, size_t bytes) {
        return cudaMallocFromPoolAsync(p, bytes, pool, compute) == cudaSuccess;
    };
    if (!take(&cd, static_cast<size_t>(K) * row_bytes) ||
        !take(reinterpret_cast<void **>(&cn), static_cast<size_t>(K) * 4) ||
        !take(&xd, 2 * static_cast<size_t>(rows) * row_bytes) ||
        !take(reinterpret_cast<void **>(&idxd), 2 * static_cast<size_t>(rows) * 4) ||
        (minscore != nullptr &&
         !take(reinterpret_cast<void **>(&msd), 2 * static_cast<size_t>(rows) * 4)))
        rc = KMASSIGN_ERR_CUDA;
    // Everything after this point is ordered after the caller's earlier work
    // on its stream and after the allocations.
    auto ok = [&](cudaError_t e) {
        if (e != cudaSuccess && rc == KMASSIGN_OK)
            rc = KMASSIGN_ERR_CUDA;
        return rc == KMASSIGN_OK;
    };
    if (rc == KMASSIGN_OK && ok(cudaEventRecord(h.start, compute)) &&
        ok(cudaStreamWaitEvent(h.copy, h.start, 0)) &&
        ok(cudaStreamWaitEvent(h.back, h.start, 0)) &&
        ok(cudaMemcpyAsync(cd, C, static_cast<size_t>(K) * row_bytes, cudaMemcpyDefault,
                           h.copy)) &&
        (cnorm == nullptr ||
         ok(cudaMemcpyAsync(cn, cnorm, static_cast<size_t>(K) * 4, cudaMemcpyDefault,
                            h.copy))) &&
        ok(cudaEventRecord(h.c_in, h.copy)) && ok(cudaStreamWaitEvent(compute, h.c_in, 0))) {
        if (cnorm == nullptr) {
            const int r = kmassign_norms(cd, K, D, cn, compute);
            if (r != KMASSIGN_OK)
                rc = r;
        }
    }
    const uint8_t *xh = static_cast<const uint8_t *>(X);
    for (int64_t s = 0, b0 = 0, nr = 0; rc == KMASSIGN_OK && b0 < N; ++s, b0 += nr) {
        const int slot = static_cast<int>(s & 1);
        nr = std::min(s == 0 ? first_rows : rows, N - b0);
        void *xs = static_cast<uint8_t *>(xd) + static_cast<size_t>(slot) * rows * row_bytes;
        int32_t *is = idxd + static_cast<size_t>(slot) * rows;
        float *ms = msd != nullptr ? msd + static_cast<size_t>(slot) * rows : nullptr;
        // the copy into a buffer waits for the kernel that last read it; the
        // kernel waits for the copy, and for the copy-out of its last answers
        if (s >= 2 && !ok(cudaStreamWaitEvent(h.copy, h.done[slot], 0)))
            break;
        if (!ok(cudaMemcpyAsync(xs, xh + static_cast<size_t>(b0) * row_bytes,
                                static_cast<size_t>(nr) * row_bytes, cudaMemcpyDefault,
                                h.copy)) ||
            !ok(cudaEventRecord(h.landed[slot], h.copy)) ||
            !ok(cudaStreamWaitEvent(compute, h.landed[slot], 0)) ||
            (s >= 2 && !ok(cudaStreamWaitEvent(compute, h.freed[slot], 0))))
            break;
        const int r = kmassign(xs, cd, cn, nr, K, D, is, ms, compute);
        if (r != KMASSIGN_OK) {
            rc = r;
            break;
        }
        if (!ok(cudaEventRecord(h.done[slot], compute)) ||
            !ok(cudaStreamWaitEvent(h.back, h.done[slot], 0)) ||
            !ok(cudaMemcpyAsync(idx + b0, is, static_cast<size_t>(nr) * 4, cudaMemcpyDefault,
                                h.back)) ||
            (ms != nullptr &&
             !ok(cudaMemcpyAsync(minscore + b0, ms, static_cast<size_t>(nr) * 4,
                                 cudaMemcpyDefault, h.back))) ||
            !ok(cudaEventRecord(h.freed[slot], h.back)))
            break;
    }
    // Whatever happened above: the caller's stream waits for both other
    // streams, returns the buffers, and the host waits for all of it.
    int end = KMASSIGN_OK;
    if (cudaEventRecord(h.copy_end, h.copy) != cudaSuccess ||
        cudaEventRecord(h.back_end, h.back) != cudaSuccess ||
        cudaStreamWaitEvent(compute, h.copy_end, 0) != cudaSuccess ||
        cudaStreamWaitEvent(compute, h.back_end, 0) != cudaSuccess)
        end = KMASSIGN_ERR_CUDA;
    for (void *p : {cd, static_cast<void *>(cn), xd, static_cast<void *>(idxd),
                    static_cast<void *>(msd)})
        if (p != nullptr && cudaFreeAsync(p, compute) != cudaSuccess)
            end = KMASSIGN_ERR_CUDA;
    if (cudaStreamSynchronize(compute) != cudaSuccess ||
        cudaStreamSynchronize(h.copy) != cudaSuccess ||
        cudaStreamSynchronize(h.back) != cudaSuccess)
        end = KMASSIGN_ERR_CUDA;
    if (rc == KMASSIGN_OK)
        rc = end;
    // a pipeline wait that ran out inside one of the kernels
    int code = 0;
    if (kma::status_read_and_clear(&code) != cudaSuccess)
        return rc == KMASSIGN_OK ? KMASSIGN_ERR_CUDA : rc;
    return rc == KMASSIGN_OK ? code : rc;
}

}  // namespace

extern "C" {

int kmassign_host(const void *X, const void *C, const float *cnorm, int64_t N, int64_t K,
                  int64_t D, int32_t *idx, float *minscore, void *stream)
{
    return run_host(X, C, cnorm, N, K, D, idx, minscore, 0, static_cast<cudaStream_t>(stream));
}

int kmassign_host_ex(const void *X, const void *C, const float *cnorm, int64_t N, int64_t K,
                     int64_t D, int32_t *idx, float *minscore, int64_t rows_per_slice,
                     void *stream)
{
    return run_host(X, C, cnorm, N, K, D, idx, minscore, rows_per_slice,
                    static_cast<cudaStream_t>(stream));
}

}  // extern "C"
