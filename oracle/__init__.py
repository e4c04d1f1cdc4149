"""fp64 CPU oracle for the k-means assignment step -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg (and its ``--impl reference`` arm) may import this package.  The product
path (``means_nearest_centroid_gb300``) never imports it and shares no code
with it.

The arithmetic lives in ``kmassign_oracle.c`` (plain C, fp64, OpenMP over
rows).  This module compiles it with gcc on first use and marshals numpy
arrays into it.  Inputs are bf16 bit patterns (``numpy.uint16``), the same
bits the CUDA path reads, so both sides see identical data.

Parity status: every function here is pinned by ``tests/test_oracle_pins.py``
(exact-rational brute force, the distance identity, numpy argmin and stable
argsort on integer data, hand-built cases with known answers, the Lloyd
descent property).  The all-NaN-row
convention (idx 0, minscore NaN) is a documented choice, pinned by its
definition only.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kmassign_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None

_i64p = ctypes.POINTER(ctypes.c_int64)


def build(force: bool = False, src: str = _SRC, out: str = _LIB_PATH) -> str:
    """Compile the oracle into a shared library; returns its path."""
    if (not force and os.path.exists(out)
            and os.path.getmtime(out) >= os.path.getmtime(src)):
        return out
    os.makedirs(os.path.dirname(out), exist_ok=True)
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared",
           "-fno-fast-math", "-ffp-contract=off", src, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True, capture_output=True, text=True)
    os.replace(tmp, out)
    return out


def load_library(path: str):
    """Load an oracle shared library and declare its signatures."""
    lib = ctypes.CDLL(path)
    vp = ctypes.c_void_p
    lib.oracle_max_threads.argtypes = [ctypes.c_int]
    lib.oracle_max_threads.restype = ctypes.c_int
    lib.oracle_norms.argtypes = [vp, ctypes.c_int64, ctypes.c_int64, vp, ctypes.c_int]
    lib.oracle_norms.restype = None
    lib.oracle_assign.argtypes = [vp, vp, vp, ctypes.c_int64, ctypes.c_int64,
                                  ctypes.c_int64, vp, ctypes.c_int64, vp, vp,
                                  ctypes.c_int]
    lib.oracle_assign.restype = None
    lib.oracle_scores.argtypes = [vp, vp, vp, ctypes.c_int64, vp, vp, ctypes.c_int64,
                                  vp, ctypes.c_int]
    lib.oracle_scores.restype = None
    lib.oracle_update.argtypes = [vp, vp, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, vp, vp]
    lib.oracle_update.restype = None
    lib.oracle_topk.argtypes = [vp, vp, vp, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, vp,
                                ctypes.c_int64, ctypes.c_int64, vp, vp, ctypes.c_int]
    lib.oracle_topk.restype = None
    lib.oracle_sqdist.argtypes = [vp, vp, ctypes.c_int64, vp, vp, ctypes.c_int64, vp, ctypes.c_int]
    lib.oracle_sqdist.restype = None
    return lib


def _get():
    global _lib
    with _lock:
        if _lib is None:
            _lib = load_library(build())
        return _lib


def _bits(a) -> np.ndarray:
    """Accept uint16/int16 numpy bf16 bit arrays or a torch bf16 CPU tensor."""
    if hasattr(a, "dtype") and str(a.dtype) == "torch.bfloat16":
        import torch  # local: the oracle itself does not need torch
        a = a.contiguous().view(torch.int16).numpy()
    a = np.ascontiguousarray(a)
    if a.dtype == np.int16:
        a = a.view(np.uint16)
    if a.dtype != np.uint16:
        raise TypeError(f"expected bf16 bit patterns (uint16), got {a.dtype}")
    if a.ndim != 2:
        raise ValueError("expected a 2-D [rows, D] array")
    return a


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


class Oracle:
    """Thin marshalling wrapper around one oracle shared library."""

    def __init__(self, lib=None):
        self.lib = lib if lib is not None else _get()

    def max_threads(self, nthreads: int = 0) -> int:
        return int(self.lib.oracle_max_threads(int(nthreads)))

    def norms(self, C, nthreads: int = 0) -> np.ndarray:
        C = _bits(C)
        K, D = C.shape
        out = np.empty(K, dtype=np.float64)
        self.lib.oracle_norms(_ptr(C), K, D, _ptr(out), int(nthreads))
        return out

    def assign(self, X, C, rows=None, cnorm=None, nthreads: int = 0):
        """Return (idx int32, minscore float64) for ``rows`` (default: all)."""
        X = _bits(X)
        C = _bits(C)
        N, D = X.shape
        K, D2 = C.shape
        if D != D2:
            raise ValueError("X and C disagree on D")
        if K < 1:
            raise ValueError("K must be >= 1")
        if cnorm is None:
            cnorm = self.norms(C, nthreads)
        cnorm = np.ascontiguousarray(cnorm, dtype=np.float64)
        if rows is None:
            rows_arr = None
            nrows = N
        else:
            rows_arr = np.ascontiguousarray(rows, dtype=np.int64)
            if rows_arr.size and (rows_arr.min() < 0 or rows_arr.max() >= N):
                raise IndexError("row index out of range")
            nrows = rows_arr.size
        idx = np.empty(nrows, dtype=np.int32)
        mins = np.empty(nrows, dtype=np.float64)
        if nrows:
            self.lib.oracle_assign(_ptr(X), _ptr(C), _ptr(cnorm), N, K, D,
                                   None if rows_arr is None else _ptr(rows_arr),
                                   nrows, _ptr(idx), _ptr(mins), int(nthreads))
        return idx, mins

    def scores(self, X, C, ii, jj, cnorm=None, nthreads: int = 0) -> np.ndarray:
        """fp64 score s_ij for each pair (ii[p], jj[p])."""
        X = _bits(X)
        C = _bits(C)
        D = X.shape[1]
        if cnorm is None:
            cnorm = self.norms(C, nthreads)
        cnorm = np.ascontiguousarray(cnorm, dtype=np.float64)
        ii = np.ascontiguousarray(ii, dtype=np.int64)
        jj = np.ascontiguousarray(jj, dtype=np.int64)
        if ii.shape != jj.shape:
            raise ValueError("ii and jj must have the same shape")
        if ii.size and (ii.min() < 0 or ii.max() >= X.shape[0]
                        or jj.min() < 0 or jj.max() >= C.shape[0]):
            raise IndexError("pair index out of range")
        out = np.empty(ii.size, dtype=np.float64)
        if ii.size:
            self.lib.oracle_scores(_ptr(X), _ptr(C), _ptr(cnorm), D, _ptr(ii),
                                   _ptr(jj), ii.size, _ptr(out), int(nthreads))
        return out


def _update(self, X, idx, K):
    """fp64 per-centroid sums [K, D] and int64 counts [K] of the points by idx."""
    X = _bits(X)
    N, D = X.shape
    idx = np.ascontiguousarray(idx, dtype=np.int32)
    if idx.shape != (N,):
        raise ValueError("idx must have one entry per point")
    sums = np.empty((K, D), dtype=np.float64)
    counts = np.empty(K, dtype=np.int64)
    self.lib.oracle_update(_ptr(X), _ptr(idx), N, K, D, _ptr(sums), _ptr(counts))
    return sums, counts


def _centroids(self, X, idx, C_old):
    """Means of the assigned points (fp64), the old centroid where none are assigned."""
    C_old = _bits(C_old)
    K, D = C_old.shape
    sums, counts = self.update(X, idx, K)
    old = (C_old.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    means = np.where(counts[:, None] > 0, sums / np.maximum(counts, 1)[:, None], old)
    return means, counts


def _topk(self, X, C, k, rows=None, cnorm=None, nthreads: int = 0):
    """(idx int32 [rows, k], score float64 [rows, k]): the k nearest centroids."""
    X = _bits(X)
    C = _bits(C)
    N, D = X.shape
    K = C.shape[0]
    if not 1 <= k <= K:
        raise ValueError("need 1 <= k <= K")
    if cnorm is None:
        cnorm = self.norms(C, nthreads)
    cnorm = np.ascontiguousarray(cnorm, dtype=np.float64)
    rows_arr = None if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
    nrows = N if rows_arr is None else rows_arr.size
    idx = np.empty((nrows, k), dtype=np.int32)
    sc = np.empty((nrows, k), dtype=np.float64)
    if nrows:
        self.lib.oracle_topk(_ptr(X), _ptr(C), _ptr(cnorm), N, K, D,
                             None if rows_arr is None else _ptr(rows_arr), nrows, k, _ptr(idx),
                             _ptr(sc), int(nthreads))
    return idx, sc


def _sqdist(self, X, C, ii, jj, nthreads: int = 0) -> np.ndarray:
    """fp64 ||x_ii[p] - c_jj[p]||^2 for each pair, summed directly over d."""
    X = _bits(X)
    C = _bits(C)
    D = X.shape[1]
    if C.shape[1] != D:
        raise ValueError("X and C disagree on D")
    ii = np.ascontiguousarray(ii, dtype=np.int64).ravel()
    jj = np.ascontiguousarray(jj, dtype=np.int64).ravel()
    if ii.shape != jj.shape:
        raise ValueError("ii and jj must have the same shape")
    if ii.size and (ii.min() < 0 or ii.max() >= X.shape[0]
                    or jj.min() < 0 or jj.max() >= C.shape[0]):
        raise IndexError("pair index out of range")
    out = np.empty(ii.size, dtype=np.float64)
    if ii.size:
        self.lib.oracle_sqdist(_ptr(X), _ptr(C), D, _ptr(ii), _ptr(jj), ii.size, _ptr(out),
                               int(nthreads))
    return out


Oracle.sqdist = _sqdist
Oracle.topk = _topk
Oracle.update = _update
Oracle.centroids = _centroids


def default() -> Oracle:
    return Oracle()


def norms(C, nthreads: int = 0):
    return default().norms(C, nthreads)


def assign(X, C, rows=None, cnorm=None, nthreads: int = 0):
    return default().assign(X, C, rows=rows, cnorm=cnorm, nthreads=nthreads)


def scores(X, C, ii, jj, cnorm=None, nthreads: int = 0):
    return default().scores(X, C, ii, jj, cnorm=cnorm, nthreads=nthreads)


def update(X, idx, K):
    return default().update(X, idx, K)


def topk(X, C, k, rows=None, cnorm=None, nthreads: int = 0):
    return default().topk(X, C, k, rows=rows, cnorm=cnorm, nthreads=nthreads)


def centroids(X, idx, C_old):
    return default().centroids(X, idx, C_old)


def sqdist(X, C, ii, jj, nthreads: int = 0):
    return default().sqdist(X, C, ii, jj, nthreads=nthreads)
