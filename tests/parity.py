"""Comparison of the CUDA path's answers with the fp64 oracle.

Rules (the assignment rule of flashlib PR #22 "Optimize Blackwell k-means
assignment reduction", Summary; tolerance as the library specifies it):

* integer-valued inputs: every fp32 step on the GPU is exact, so idx must be
  identical to the oracle's and minscore equal to the oracle's fp64 score
  (NaN where the oracle has NaN);
* float inputs: an idx j' that differs from the oracle's j* is accepted only
  if s64(i, j') - s64(i, j*) <= TOL * (||x_i||^2 + ||c_j'||^2), with s64 the
  oracle's fp64 score; the number of such rows is reported.  The GPU
  minscore must be within the same bound of s64(i, j').

TOL = 2e-5.  Where it comes from: the GPU score is an fp32 dot product of D
terms plus an fp32 norm; summation error is bounded by about D * 2^-24 times
(|x|.|c| + ||c||^2) in the worst case (1.5e-5 at D = 256) and is typically
~sqrt(D) * 2^-24.
"""

from __future__ import annotations

import dataclasses

import numpy as np
import torch

import oracle

TOL = 2e-5


@dataclasses.dataclass
class Report:
    rows: int
    idx_mismatches: int          # rows whose idx differs from the oracle's
    rejected: int                # mismatches outside the tolerance
    minscore_bad: int            # minscore outside the rule
    worst_gap: float             # largest accepted relative score gap

    def ok(self) -> bool:
        return self.rejected == 0 and self.minscore_bad == 0


def _as_np(t):
    if isinstance(t, torch.Tensor):
        return t.detach().cpu().numpy()
    return np.asarray(t)


def compare(X, C, gpu_idx, gpu_ms, rows=None, integer=False, orc=None, nthreads=0) -> Report:
    """Check GPU answers for ``rows`` (default all) against the oracle."""
    orc = orc or oracle.default()
    gpu_idx = _as_np(gpu_idx).astype(np.int64)
    gpu_ms = None if gpu_ms is None else _as_np(gpu_ms).astype(np.float64)
    N = X.shape[0]
    rows = np.arange(N) if rows is None else np.asarray(rows, dtype=np.int64)
    cn64 = orc.norms(C, nthreads)
    o_idx, o_min = orc.assign(X, C, rows=rows, cnorm=cn64, nthreads=nthreads)
    g_idx = gpu_idx[rows]
    g_ms = None if gpu_ms is None else gpu_ms[rows]
    if np.any(g_idx < 0) or np.any(g_idx >= C.shape[0]):
        return Report(len(rows), len(rows), len(rows), 0, float("inf"))
    diff = g_idx != o_idx
    if integer:
        ms_bad = 0
        if g_ms is not None:
            both_nan = np.isnan(g_ms) & np.isnan(o_min)
            ms_bad = int(np.sum(~(both_nan | (g_ms == o_min))))
        nd = int(diff.sum())
        return Report(len(rows), nd, nd, ms_bad, 0.0)
    # float rule
    xs = X.to(torch.float64).numpy()[rows]
    xn = np.einsum("rd,rd->r", xs, xs)
    s_g = orc.scores(X, C, rows, g_idx, cnorm=cn64, nthreads=nthreads)
    scale = xn + cn64[g_idx]
    gap = s_g - o_min
    finite = np.isfinite(o_min) & np.isfinite(s_g)
    accept = np.where(diff, finite & (gap <= TOL * scale), True)
    # non-finite oracle minima must be matched exactly (special values)
    accept &= np.where(~np.isfinite(o_min), (g_idx == o_idx), True)
    rejected = int((~accept).sum())
    worst = float(np.max(np.where(diff & finite, gap / np.maximum(scale, 1e-300), 0.0))) if len(rows) else 0.0
    ms_bad = 0
    if g_ms is not None:
        both_nan = np.isnan(g_ms) & np.isnan(s_g)
        same_inf = np.isinf(g_ms) & (g_ms == s_g)
        close = np.abs(g_ms - s_g) <= TOL * scale
        ms_bad = int(np.sum(~(both_nan | same_inf | (np.isfinite(s_g) & close))))
    return Report(len(rows), int(diff.sum()), rejected, ms_bad, worst)


# ---------------------------------------------------------------- top-k
@dataclasses.dataclass
class TopkReport:
    rows: int
    invalid: int            # rows with an index out of range or repeated
    order_bad: int          # rows whose exact scores stray from the oracle's order statistics
    score_bad: int          # reported scores/distances outside the rule
    unsorted: int           # rows whose reported values are not ascending
    idx_mismatches: int     # rows whose idx list differs from the oracle's

    def ok(self) -> bool:
        return self.invalid == 0 and self.order_bad == 0 and self.score_bad == 0 and self.unsorted == 0


def compare_topk(X, C, gpu_idx, gpu_score, k, rows=None, integer=False, distances=False,
                 orc=None, nthreads=0) -> TopkReport:
    """Check the GPU's k nearest centroids for ``rows`` against the oracle.

    * integer data: every fp32 step is exact, so idx must equal the oracle's
      lists and the values its scores (or direct squared distances);
    * float data: the GPU ranks by fp32 scores within TOL * scale of the exact
      ones (scale = ||x||^2 + max_j ||c_j||^2), so the exact score of its e-th
      pick must lie within 2 * TOL * scale of the oracle's e-th smallest score
      (order statistics move by at most the uniform error); each reported
      value within TOL (scores) or 2 TOL (distances, which add the fp32
      ||x||^2) times ||x||^2 + ||c||^2 of the exact one.
    Every row must hold k distinct valid indices with non-decreasing values.
    """
    orc = orc or oracle.default()
    gi = _as_np(gpu_idx).astype(np.int64).reshape(-1, k)
    gs = None if gpu_score is None else _as_np(gpu_score).astype(np.float64).reshape(-1, k)
    N, K = X.shape[0], C.shape[0]
    rows = np.arange(N) if rows is None else np.asarray(rows, dtype=np.int64)
    cn64 = orc.norms(C, nthreads)
    o_idx, o_s = orc.topk(X, C, k, rows=rows, cnorm=cn64, nthreads=nthreads)
    g = gi[rows]
    sg = None if gs is None else gs[rows]
    bad_range = np.any((g < 0) | (g >= K), axis=1)
    srt = np.sort(g, axis=1)
    repeated = np.any(srt[:, 1:] == srt[:, :-1], axis=1) if k > 1 else np.zeros(len(rows), bool)
    invalid = bad_range | repeated
    n = len(rows)
    if invalid.any():
        return TopkReport(n, int(invalid.sum()), 0, 0, 0, n)
    mism = int(np.sum(np.any(g != o_idx, axis=1)))
    rr = np.repeat(rows, k)
    exact_s = orc.scores(X, C, rr, g.ravel(), cnorm=cn64, nthreads=nthreads).reshape(-1, k)
    exact_v = (orc.sqdist(X, C, rr, g.ravel(), nthreads=nthreads).reshape(-1, k)
               if distances else exact_s)
    unsorted = 0
    if sg is not None and k > 1:
        a, b = sg[:, :-1], sg[:, 1:]
        ok_pair = (a <= b) | np.isnan(b) | (np.isnan(a) & np.isnan(b))
        unsorted = int(np.sum(~np.all(ok_pair, axis=1)))
    if integer:
        order_bad = mism
        score_bad = 0
        if sg is not None:
            same = (sg == exact_v) | (np.isnan(sg) & np.isnan(exact_v))
            score_bad = int(np.sum(~np.all(same, axis=1)))
        return TopkReport(n, 0, order_bad, score_bad, unsorted, mism)
    xs = X.to(torch.float64).numpy()[rows]
    xn = np.einsum("rd,rd->r", xs, xs)
    scale = xn + cn64.max()
    fin = np.isfinite(o_s) & np.isfinite(exact_s)
    close = np.abs(exact_s - o_s) <= 2 * TOL * scale[:, None]
    order_bad = int(np.sum(~np.all(np.where(fin, close, g == o_idx), axis=1)))
    score_bad = 0
    if sg is not None:
        pair_scale = xn[:, None] + cn64[g]
        tol = (2 * TOL if distances else TOL) * pair_scale
        good = (np.abs(sg - exact_v) <= tol) | (np.isnan(sg) & np.isnan(exact_v))
        score_bad = int(np.sum(~np.all(good, axis=1)))
    return TopkReport(n, 0, order_bad, score_bad, unsorted, mism)
