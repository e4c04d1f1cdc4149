"""libkmassign: the k-means assignment step on one NVIDIA GB300 (sm_103a).

For points X[N, D] and centroids C[K, D] (bf16), returns

    idx[i] = argmin_j (||c_j||^2 - 2 x_i . c_j)      (lowest j on ties)

(flashlib PR #22 "Optimize Blackwell k-means assignment reduction",
Summary).  Every step runs in the CUDA kernels of ``libkmassign.so``; this
module only marshals torch tensors into the C ABI declared in
``include/kmassign.h`` and raises on error codes.  There is no CPU path: if
the shared library is missing, every call raises.
"""

from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import _build

__all__ = [
    "KmassignError", "library", "library_path", "kmassign", "kmassign_ex", "kmassign_norms",
    "kmassign_noalloc", "kmassign_set_wait_timeout", "shard_rows", "kmassign_update",
    "kmassign_centroids", "kmassign_lloyd",
    "kmassign_plan", "kmassign_plan_for", "kmassign_check", "kmassign_strerror", "assign", "norms", "assign_host",
    "STATUS",
]

STATUS = {
    "KMASSIGN_OK": 0,
    "KMASSIGN_ERR_NULL": -1,
    "KMASSIGN_ERR_ALIGN": -2,
    "KMASSIGN_ERR_SHAPE": -3,
    "KMASSIGN_ERR_UNSUPPORTED_D": -4,
    "KMASSIGN_ERR_CUDA": -5,
    "KMASSIGN_ERR_TIMEOUT": -6,
    "KMASSIGN_ERR_NOT_DEVICE": -7,
    "KMASSIGN_ERR_ARG": -8,
    "KMASSIGN_ERR_SCRATCH": -9,
    "KMASSIGN_ERR_NOT_HOST": -10,
    "KMASSIGN_ERR_DEBUG_CHECK": -11,
}
_NAMES = {v: k for k, v in STATUS.items()}

_lock = threading.Lock()
_lib = None


class KmassignError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = int(code)
        super().__init__(f"{where}: {_NAMES.get(code, code)} ({kmassign_strerror(code)})")


def library_path() -> str:
    return _build.LIB_PATH


def _declare(lib):
    vp, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
    lib.kmassign_norms.argtypes = [vp, i64, i64, vp, vp]
    lib.kmassign_norms.restype = i32
    lib.kmassign.argtypes = [vp, vp, vp, i64, i64, i64, vp, vp, vp]
    lib.kmassign.restype = i32
    lib.kmassign_ex.argtypes = [vp, vp, vp, i64, i64, i64, vp, vp, i32, i32, i32, i32, vp]
    lib.kmassign_ex.restype = i32
    lib.kmassign_host.argtypes = [vp, vp, vp, i64, i64, i64, vp, vp, vp]
    lib.kmassign_host.restype = i32
    lib.kmassign_host_ex.argtypes = [vp, vp, vp, i64, i64, i64, vp, vp, i64, vp]
    lib.kmassign_host_ex.restype = i32
    lib.kmassign_noalloc.argtypes = [vp, vp, vp, i64, i64, i64, vp, vp, vp]
    lib.kmassign_noalloc.restype = i32
    lib.kmassign_plan.argtypes = [i64, i64, i64, vp]
    lib.kmassign_plan.restype = i32
    lib.kmassign_plan_ex.argtypes = [i64, i64, i64, i32, i32, i32, i32, vp]
    lib.kmassign_plan_ex.restype = i32
    lib.kmassign_plan_for.argtypes = [i64, i64, i64, i32, i32, i32, i32, i32, i32, i32, vp]
    lib.kmassign_plan_for.restype = i32
    lib.kmassign_update.argtypes = [vp, vp, i64, i64, i64, vp, vp, vp]
    lib.kmassign_update.restype = i32
    lib.kmassign_update_ex.argtypes = [vp, vp, i64, i64, i64, vp, vp, i32, vp]
    lib.kmassign_update_ex.restype = i32
    lib.kmassign_centroids.argtypes = [vp, vp, vp, i64, i64, vp, vp, vp]
    lib.kmassign_centroids.restype = i32
    lib.kmassign_lloyd.argtypes = [vp, vp, i64, i64, i64, i32, vp, vp]
    lib.kmassign_lloyd.restype = i32
    lib.kmassign_topk.argtypes = [vp, vp, vp, i64, i64, i64, i32, vp, vp, i32, vp]
    lib.kmassign_topk.restype = i32
    lib.kmassign_topk_ex.argtypes = [vp, vp, vp, i64, i64, i64, i32, vp, vp, i32, i32, vp]
    lib.kmassign_topk_ex.restype = i32
    lib.kmassign_set_wait_timeout.argtypes = [ctypes.c_uint64]
    lib.kmassign_set_wait_timeout.restype = i32
    lib.kmassign_check.argtypes = [vp]
    lib.kmassign_check.restype = i32
    lib.kmassign_strerror.argtypes = [i32]
    lib.kmassign_strerror.restype = ctypes.c_char_p
    return lib


def library(path: str | None = None):
    """The loaded libkmassign (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            p = path or library_path()
            if not os.path.exists(p):
                raise RuntimeError(
                    f"libkmassign.so not found at {p}; build it with "
                    "`python -m means_nearest_centroid_gb300._build` (there is no CPU fallback)")
            _lib = _declare(ctypes.CDLL(p))
        return _lib


def kmassign_strerror(code: int) -> str:
    return library().kmassign_strerror(int(code)).decode()


def _check(code: int, where: str):
    if code != 0:
        raise KmassignError(code, where)


_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream_ptr(stream, device=None) -> int:
    """The cudaStream_t to launch on: ``stream``, else the current stream of
    ``device`` (the tensors' device), else of the current device."""
    if stream is None:
        if _raw_stream is not None:
            idx = torch.cuda.current_device() if device is None else device.index
            return _raw_stream(idx)
        stream = torch.cuda.current_stream(device)
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _ptr(t):
    return None if t is None else t.data_ptr()


def _need_cuda(t, name, dtype):
    # the common case in one expression; the detail only on failure
    if isinstance(t, torch.Tensor) and t.is_cuda and t.dtype == dtype and t.is_contiguous():
        return
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    raise ValueError(f"{name} must be contiguous")


def kmassign_norms(C: torch.Tensor, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """cnorm[j] = ||c_j||^2 (fp32) on the GPU."""
    _need_cuda(C, "C", torch.bfloat16)
    K, D = C.shape
    if out is None:
        out = torch.empty(K, dtype=torch.float32, device=C.device)
    _need_cuda(out, "out", torch.float32)
    _check(library().kmassign_norms(_ptr(C), K, D, _ptr(out), _stream_ptr(stream, C.device)),
           "kmassign_norms")
    return out


def kmassign_ex(X, C, cnorm=None, idx=None, minscore=None, ksplit: int = 0,
                rows_per_cta: int = 0, centroids_per_tile: int = 0, consumer_warps: int = 0,
                stream=None):
    """Assignment with an explicit plan (0 = automatic).  Returns idx (int32)."""
    _need_cuda(X, "X", torch.bfloat16)
    _need_cuda(C, "C", torch.bfloat16)
    N, D = X.shape
    K, D2 = C.shape
    if D != D2:
        raise ValueError("X and C disagree on D")
    if cnorm is not None:
        _need_cuda(cnorm, "cnorm", torch.float32)
    if idx is None:
        idx = torch.empty(N, dtype=torch.int32, device=X.device)
    _need_cuda(idx, "idx", torch.int32)
    if minscore is not None:
        _need_cuda(minscore, "minscore", torch.float32)
    rc = library().kmassign_ex(_ptr(X), _ptr(C), _ptr(cnorm), N, K, D, _ptr(idx), _ptr(minscore),
                               int(ksplit), int(rows_per_cta), int(centroids_per_tile),
                               int(consumer_warps), _stream_ptr(stream, X.device))
    _check(rc, "kmassign_ex")
    return idx


def kmassign(X, C, cnorm=None, idx=None, minscore=None, stream=None):
    """idx[i] = argmin_j (||c_j||^2 - 2 x_i . c_j) on the GPU; returns idx."""
    _need_cuda(X, "X", torch.bfloat16)
    _need_cuda(C, "C", torch.bfloat16)
    N, D = X.shape
    K, D2 = C.shape
    if D != D2:
        raise ValueError("X and C disagree on D")
    if cnorm is not None:
        _need_cuda(cnorm, "cnorm", torch.float32)
    if idx is None:
        idx = torch.empty(N, dtype=torch.int32, device=X.device)
    _need_cuda(idx, "idx", torch.int32)
    if minscore is not None:
        _need_cuda(minscore, "minscore", torch.float32)
    rc = library().kmassign(_ptr(X), _ptr(C), _ptr(cnorm), N, K, D, _ptr(idx), _ptr(minscore),
                            _stream_ptr(stream, X.device))
    _check(rc, "kmassign")
    return idx


def kmassign_noalloc(X, C, cnorm=None, idx=None, minscore=None, stream=None):
    """kmassign for callers that cannot let the library allocate device memory.

    The library's temporaries come from its static device array instead of
    the stream allocator (see ``include/kmassign.h``).  ``idx`` should be
    passed preallocated by such callers; it is allocated here only for
    convenience.  Calls that overlap on the GPU share that array and race.
    """
    _need_cuda(X, "X", torch.bfloat16)
    _need_cuda(C, "C", torch.bfloat16)
    N, D = X.shape
    K, D2 = C.shape
    if D != D2:
        raise ValueError("X and C disagree on D")
    if cnorm is not None:
        _need_cuda(cnorm, "cnorm", torch.float32)
    if idx is None:
        idx = torch.empty(N, dtype=torch.int32, device=X.device)
    _need_cuda(idx, "idx", torch.int32)
    if minscore is not None:
        _need_cuda(minscore, "minscore", torch.float32)
    rc = library().kmassign_noalloc(_ptr(X), _ptr(C), _ptr(cnorm), N, K, D, _ptr(idx),
                                    _ptr(minscore), _stream_ptr(stream, X.device))
    _check(rc, "kmassign_noalloc")
    return idx


def kmassign_topk(X, C, k: int, cnorm=None, idx=None, score=None, distances: bool = False,
                  with_score: bool = True, ksplit: int = 0, stream=None):
    """The k nearest centroids of every point: (idx int32 [N, k], score fp32 [N, k]).

    Row i lists centroids in ascending score s_ij = ||c_j||^2 - 2 x_i . c_j
    (lowest index first on ties); ``distances`` returns ||x_i||^2 + s_ij
    instead.  ``score`` is None when ``with_score`` is false and no output
    tensor is given.  ``ksplit`` forces a split of the centroid axis (0 =
    automatic; see ``kmassign_topk_ex`` in ``include/kmassign.h``).
    """
    _need_cuda(X, "X", torch.bfloat16)
    _need_cuda(C, "C", torch.bfloat16)
    N, D = X.shape
    K, D2 = C.shape
    if D != D2:
        raise ValueError("X and C disagree on D")
    if cnorm is not None:
        _need_cuda(cnorm, "cnorm", torch.float32)
    k = int(k)
    if idx is None:
        idx = torch.empty((N, max(k, 0)), dtype=torch.int32, device=X.device)
    _need_cuda(idx, "idx", torch.int32)
    if score is None and (with_score or distances):
        score = torch.empty((N, max(k, 0)), dtype=torch.float32, device=X.device)
    if score is not None:
        _need_cuda(score, "score", torch.float32)
    lib = library()
    if ksplit:
        rc = lib.kmassign_topk_ex(_ptr(X), _ptr(C), _ptr(cnorm), N, K, D, k, _ptr(idx),
                                  _ptr(score), int(bool(distances)), int(ksplit),
                                  _stream_ptr(stream, X.device))
    else:
        rc = lib.kmassign_topk(_ptr(X), _ptr(C), _ptr(cnorm), N, K, D, k, _ptr(idx), _ptr(score),
                               int(bool(distances)), _stream_ptr(stream, X.device))
    _check(rc, "kmassign_topk")
    return idx, score


def kmassign_plan(N: int, K: int, D: int, ksplit: int = 0, rows_per_cta: int = 0,
                  centroids_per_tile: int = 0, consumer_warps: int = 0) -> dict:
    """The plan kmassign (or, with forcing arguments, kmassign_ex) would run."""
    out = (ctypes.c_int32 * 9)()
    _check(library().kmassign_plan_ex(int(N), int(K), int(D), int(ksplit), int(rows_per_cta),
                                      int(centroids_per_tile), int(consumer_warps),
                                      ctypes.cast(out, ctypes.c_void_p)),
           "kmassign_plan")
    keys = ["ksplit", "rows_per_cta", "centroids_per_tile", "grid", "stages", "xbufs",
            "whole_row_tiles", "split_row_tiles", "consumer_warps"]
    return dict(zip(keys, list(out)))


def kmassign_plan_for(N: int, K: int, D: int, sms: int = 152, smem_per_block: int = 232448,
                      pair_clusters: int = 76, ksplit: int = 0, rows_per_cta: int = 0,
                      centroids_per_tile: int = 0, consumer_warps: int = 0) -> dict:
    """The plan for a described device (default: a GB300); needs no GPU."""
    out = (ctypes.c_int32 * 9)()
    _check(library().kmassign_plan_for(int(N), int(K), int(D), int(sms), int(smem_per_block),
                                       int(pair_clusters), int(ksplit), int(rows_per_cta),
                                       int(centroids_per_tile), int(consumer_warps),
                                       ctypes.cast(out, ctypes.c_void_p)),
           "kmassign_plan_for")
    keys = ["ksplit", "rows_per_cta", "centroids_per_tile", "grid", "stages", "xbufs",
            "whole_row_tiles", "split_row_tiles", "consumer_warps"]
    return dict(zip(keys, list(out)))


def kmassign_update(X, idx, K: int, sums=None, counts=None, method: int = 0, stream=None):
    """Per-centroid fp32 sums [K, D] and int32 counts [K] of X's rows by idx.

    When sums/counts are given they are accumulated into; otherwise zeroed
    tensors are created.  ``method``: 0 automatic, 1 atomic, 2 sorted (see
    ``kmassign_update_ex`` in ``include/kmassign.h``).  Returns (sums, counts).
    """
    _need_cuda(X, "X", torch.bfloat16)
    _need_cuda(idx, "idx", torch.int32)
    N, D = X.shape
    if idx.shape != (N,):
        raise ValueError("idx must hold one id per point")
    if sums is None:
        sums = torch.zeros((K, D), dtype=torch.float32, device=X.device)
    if counts is None:
        counts = torch.zeros(K, dtype=torch.int32, device=X.device)
    _need_cuda(sums, "sums", torch.float32)
    _need_cuda(counts, "counts", torch.int32)
    _check(library().kmassign_update_ex(_ptr(X), _ptr(idx), N, int(K), D, _ptr(sums),
                                        _ptr(counts), int(method),
                                        _stream_ptr(stream, X.device)),
           "kmassign_update")
    return sums, counts


def kmassign_centroids(sums, counts, C_old, C_new=None, means=None, stream=None):
    """bf16 means of the assigned points (C_old where a centroid has none)."""
    _need_cuda(sums, "sums", torch.float32)
    _need_cuda(counts, "counts", torch.int32)
    _need_cuda(C_old, "C_old", torch.bfloat16)
    K, D = C_old.shape
    if C_new is None:
        C_new = torch.empty_like(C_old)
    _need_cuda(C_new, "C_new", torch.bfloat16)
    if means is not None:
        _need_cuda(means, "means", torch.float32)
    _check(library().kmassign_centroids(_ptr(sums), _ptr(counts), _ptr(C_old), K, D, _ptr(C_new),
                                        _ptr(means), _stream_ptr(stream, sums.device)),
           "kmassign_centroids")
    return C_new


def kmassign_lloyd(X, C, iters: int, idx=None, stream=None):
    """``iters`` Lloyd iterations on the GPU, updating C (bf16) in place.

    Returns idx, the last assignment (made before the last update).
    """
    _need_cuda(X, "X", torch.bfloat16)
    _need_cuda(C, "C", torch.bfloat16)
    N, D = X.shape
    K = C.shape[0]
    if idx is None:
        idx = torch.empty(N, dtype=torch.int32, device=X.device)
    _need_cuda(idx, "idx", torch.int32)
    _check(library().kmassign_lloyd(_ptr(X), _ptr(C), N, K, D, int(iters), _ptr(idx),
                                    _stream_ptr(stream, X.device)), "kmassign_lloyd")
    return idx


def kmassign_set_wait_timeout(ns: int) -> None:
    """Bound on every kernel pipeline wait, in ns (0 = default 2 s)."""
    _check(library().kmassign_set_wait_timeout(int(ns)), "kmassign_set_wait_timeout")


def shard_rows(N: int, rank: int, world: int) -> tuple:
    """Contiguous, balanced share [begin, end) of N points for one of `world` GPUs.

    The assignment needs no exchange between GPUs: each holds all centroids
    and assigns its own rows; the answers concatenate in rank order.
    """
    if world < 1 or not 0 <= rank < world or N < 0:
        raise ValueError("need N >= 0 and 0 <= rank < world")
    base, extra = divmod(int(N), int(world))
    begin = rank * base + min(rank, extra)
    return begin, begin + base + (1 if rank < extra else 0)


def kmassign_check(stream=None) -> int:
    """Synchronise the stream and return the device status code (0 = OK)."""
    return int(library().kmassign_check(_stream_ptr(stream)))


def norms(C, stream=None):
    return kmassign_norms(C, stream=stream)


def assign(X, C, cnorm=None, with_minscore: bool = False, stream=None):
    """Convenience: returns idx, or (idx, minscore) when ``with_minscore``."""
    ms = None
    if with_minscore:
        ms = torch.empty(X.shape[0], dtype=torch.float32, device=X.device)
    idx = kmassign(X, C, cnorm=cnorm, minscore=ms, stream=stream)
    return (idx, ms) if with_minscore else idx


def _need_host(t, name, dtype):
    if isinstance(t, torch.Tensor) and not t.is_cuda and t.dtype == dtype and t.is_contiguous():
        return
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.is_cuda:
        raise ValueError(f"{name} must be a CPU tensor (ideally pinned)")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    raise ValueError(f"{name} must be contiguous")


def assign_host(X_host, C_host, idx_host=None, cnorm_host=None, minscore_host=None,
                device=None, stream=None, rows_per_slice: int = 0):
    """End-to-end assignment of host tensors through ``kmassign_host``.

    X (bf16 [N, D]), C (bf16 [K, D]) and the optional cnorm (fp32 [K]) are
    CPU tensors, ideally pinned so that the copies overlap the kernels.  The
    library copies C in, then X in row slices of whole kernel waves while the
    previous slice is assigned, and copies each slice's idx (and minscore)
    back as soon as it is ready; the call returns when the answers are in
    ``idx_host`` (int32 [N], pinned, allocated if None) and ``minscore_host``
    (fp32 [N] or None).  ``device`` is the GPU to run on (default: current),
    ``stream`` a stream of it (default: its current stream),
    ``rows_per_slice`` forces the slice size (0: automatic).  Returns idx_host.
    """
    _need_host(X_host, "X_host", torch.bfloat16)
    _need_host(C_host, "C_host", torch.bfloat16)
    N, D = X_host.shape
    K, D2 = C_host.shape
    if D != D2:
        raise ValueError("X and C disagree on D")
    if cnorm_host is not None:
        _need_host(cnorm_host, "cnorm_host", torch.float32)
    if idx_host is None:
        idx_host = torch.empty(N, dtype=torch.int32, pin_memory=True)
    _need_host(idx_host, "idx_host", torch.int32)
    if minscore_host is not None:
        _need_host(minscore_host, "minscore_host", torch.float32)
    device = torch.device("cuda") if device is None else torch.device(device)
    if device.index is None:
        device = torch.device("cuda", torch.cuda.current_device())
    with torch.cuda.device(device):
        rc = library().kmassign_host_ex(_ptr(X_host), _ptr(C_host), _ptr(cnorm_host), N, K, D,
                                        _ptr(idx_host), _ptr(minscore_host), int(rows_per_slice),
                                        _stream_ptr(stream, device))
    _check(rc, "kmassign_host")
    return idx_host
