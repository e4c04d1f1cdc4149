"""Checks that pin the fp64 oracle to facts outside itself.

Each ``check_*`` function takes an ``oracle.Oracle`` and raises
``AssertionError`` when the oracle disagrees with:

* hand-derived answers (``tests/golden/hand_cases.json``);
* an exact-rational brute force (``fractions.Fraction``) on tiny inputs --
  every bf16 value is a dyadic rational, so the exact argmin is known;
* the identity ||x - c||^2 = ||x||^2 + s, with the distance computed
  directly from the difference vector;
* ``numpy.argmin`` (documented to return the first occurrence) over an exact
  fp64 score matrix on integer data;
* closed-form winners for rows holding one infinity;
* self-consistency of the row-subset and pair-score entry points.

The same functions run against deliberately broken copies of the oracle in
``test_oracle_mutants.py``: every planted mistake must trip at least one.
"""

from __future__ import annotations

import json
import math
import os
from fractions import Fraction

import numpy as np
import torch

import workloads

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden",
                      "hand_cases.json")


def _val(v):
    if isinstance(v, str):
        return {"nan": math.nan, "inf": math.inf, "-inf": -math.inf, "-0": -0.0}[v]
    return float(v)


def _bf16_rows(rows):
    t = torch.tensor([[_val(v) for v in r] for r in rows], dtype=torch.float32)
    b = t.to(torch.bfloat16)
    # the fixtures are exact in bf16: nothing may round
    back = b.to(torch.float32)
    same = (back == t) | (torch.isnan(back) & torch.isnan(t))
    assert bool(same.all()), "golden value not exact in bf16"
    return b.contiguous()


def _same_score(a: float, b: float) -> bool:
    if math.isnan(a) or math.isnan(b):
        return math.isnan(a) and math.isnan(b)
    return a == b


def load_golden():
    with open(GOLDEN) as f:
        return json.load(f)["cases"]


def check_golden(orc):
    for case in load_golden():
        X = _bf16_rows(case["X"])
        C = _bf16_rows(case["C"])
        idx, mins = orc.assign(X, C)
        exp_idx = case["idx"]
        exp_min = [_val(v) for v in case["minscore"]]
        assert list(idx) == exp_idx, (case["name"], list(idx), exp_idx)
        for got, exp in zip(mins, exp_min):
            assert _same_score(float(got), exp), (case["name"], float(got), exp)


def _exact(b16: torch.Tensor):
    return [[Fraction(float(v)) for v in row] for row in b16.to(torch.float32).tolist()]


def _exact_assign(Xf, Cf):
    """Exact-rational argmin with lowest-index ties (finite inputs only)."""
    norms = [sum(c * c for c in row) for row in Cf]
    out_idx, out_s = [], []
    for x in Xf:
        s = [norms[j] - 2 * sum(a * b for a, b in zip(x, Cf[j])) for j in range(len(Cf))]
        m = min(s)
        j = s.index(m)          # list.index: the first occurrence
        out_idx.append(j)
        out_s.append(m)
    return out_idx, out_s, norms


def check_bruteforce_rational(orc, trials: int = 24):
    rng = np.random.default_rng(12345)
    for t in range(trials):
        N = int(rng.integers(1, 9))
        K = int(rng.integers(1, 13))
        D = int(rng.integers(1, 17))
        if t % 3 == 0:
            X, C = workloads.integers(N, K, D, seed=1000 + t, lo=-2, hi=2)
        elif t % 3 == 1:
            X, C = workloads.iid(N, K, D, seed=2000 + t)
        else:
            X, C = workloads.blobs(N, K, D, seed=3000 + t)
            # force cross-index duplicates so exact ties occur
            if K >= 2:
                C[K - 1] = C[0]
        Xf, Cf = _exact(X), _exact(C)
        exp_idx, exp_s, exp_norms = _exact_assign(Xf, Cf)
        idx, mins = orc.assign(X, C)
        assert list(idx) == exp_idx, (t, list(idx), exp_idx)
        for got, exp in zip(mins, exp_s):
            # fp64 sums of <= 16 bf16 products are exact here; keep a
            # rounding-sized allowance in case a sum spans many binades
            assert abs(Fraction(float(got)) - exp) <= Fraction(1, 2**40) * (1 + abs(exp)), (t, got, exp)
        norms = orc.norms(C)
        for got, exp in zip(norms, exp_norms):
            assert Fraction(float(got)) == exp, (t, got, exp)


def check_distance_identity(orc):
    # float data: ||x - c||^2 computed from the difference vector
    X, C = workloads.iid(40, 30, 48, seed=77)
    xs = X.to(torch.float64).numpy()
    cs = C.to(torch.float64).numpy()
    ii, jj = np.meshgrid(np.arange(40), np.arange(30), indexing="ij")
    ii, jj = ii.ravel(), jj.ravel()
    s = orc.scores(X, C, ii, jj)
    diff = xs[ii] - cs[jj]
    dist = np.einsum("pd,pd->p", diff, diff)
    xn = np.einsum("pd,pd->p", xs[ii], xs[ii])
    cn = np.einsum("pd,pd->p", cs[jj], cs[jj])
    err = np.abs((xn + s) - dist)
    assert np.all(err <= 1e-12 * (xn + cn + 1.0)), float(err.max())
    # integer data: the identity holds exactly
    X, C = workloads.integers(25, 19, 33, seed=78)
    xs = X.to(torch.float64).numpy()
    cs = C.to(torch.float64).numpy()
    ii, jj = np.meshgrid(np.arange(25), np.arange(19), indexing="ij")
    ii, jj = ii.ravel(), jj.ravel()
    s = orc.scores(X, C, ii, jj)
    diff = xs[ii] - cs[jj]
    dist = np.einsum("pd,pd->p", diff, diff)
    xn = np.einsum("pd,pd->p", xs[ii], xs[ii])
    assert np.array_equal(xn + s, dist)
    # the winner is the nearest centroid in Euclidean distance
    idx, _ = orc.assign(X, C)
    full = ((xs[:, None, :] - cs[None, :, :]) ** 2).sum(-1)
    assert np.array_equal(idx, np.argmin(full, axis=1))


def check_numpy_argmin(orc):
    for seed, (N, K, D) in enumerate([(200, 97, 24), (64, 300, 8), (33, 5, 64)]):
        X, C = workloads.integers(N, K, D, seed=500 + seed)
        if K > 4:
            C[K // 2:K // 2 + 3] = C[1]        # ties far apart in the index
        xs = X.to(torch.float64).numpy()
        cs = C.to(torch.float64).numpy()
        S = (cs * cs).sum(1)[None, :] - 2.0 * (xs @ cs.T)   # exact on integers
        idx, mins = orc.assign(X, C)
        exp = np.argmin(S, axis=1)                          # first occurrence
        assert np.array_equal(idx, exp), seed
        assert np.array_equal(mins, S[np.arange(N), exp]), seed


def check_single_infinity_rows(orc):
    """Closed form for a row with one +-inf at dimension d, finite elsewhere.

    x.c_j is +inf * sign(c_jd) (NaN when c_jd == 0), so s_j is -inf where
    x_d * c_jd > 0, +inf where < 0 and NaN where c_jd == 0.  Winner: the
    lowest j with -inf, else the lowest j with +inf, else 0 (all NaN).
    """
    rng = np.random.default_rng(7)
    for t in range(30):
        K = int(rng.integers(1, 12))
        D = int(rng.integers(1, 6))
        X, C = workloads.integers(1, K, D, seed=900 + t, lo=-1, hi=1)
        d = int(rng.integers(0, D))
        sign = 1.0 if t % 2 == 0 else -1.0
        X[0, d] = sign * math.inf
        col = C[:, d].to(torch.float32).numpy() * sign
        neg = np.nonzero(col > 0)[0]
        pos = np.nonzero(col < 0)[0]
        if neg.size:
            exp_j, exp_s = int(neg[0]), -math.inf
        elif pos.size:
            exp_j, exp_s = int(pos[0]), math.inf
        else:
            exp_j, exp_s = 0, math.nan
        idx, mins = orc.assign(X, C)
        assert int(idx[0]) == exp_j, (t, int(idx[0]), exp_j)
        assert _same_score(float(mins[0]), exp_s), (t, float(mins[0]), exp_s)
    # NaN anywhere in x makes every score NaN
    X, C = workloads.integers(3, 9, 7, seed=901)
    X[1, 3] = math.nan
    idx, mins = orc.assign(X, C)
    assert int(idx[1]) == 0 and math.isnan(mins[1])


def check_subsets_consistent(orc):
    X, C = workloads.blobs(50, 20, 12, seed=31)
    full_idx, full_min = orc.assign(X, C)
    rows = np.array([49, 0, 7, 7, 23])
    idx, mins = orc.assign(X, C, rows=rows)
    assert np.array_equal(idx, full_idx[rows])
    assert np.array_equal(mins, full_min[rows])
    s = orc.scores(X, C, rows, full_idx[rows])
    assert np.array_equal(s, full_min[rows])


ALL_CHECKS = [check_golden, check_bruteforce_rational, check_distance_identity,
              check_numpy_argmin, check_single_infinity_rows, check_subsets_consistent]


# ---------------------------------------------------------------- update step
def _exact_update(Xf, idx, K, D):
    sums = [[Fraction(0)] * D for _ in range(K)]
    counts = [0] * K
    for x, j in zip(Xf, idx):
        if 0 <= j < K:
            counts[j] += 1
            for d in range(D):
                sums[j][d] += x[d]
    return sums, counts


def check_update_rational(orc, trials: int = 12):
    rng = np.random.default_rng(321)
    for t in range(trials):
        N = int(rng.integers(0, 30))
        K = int(rng.integers(1, 9))
        D = int(rng.integers(1, 12))
        X, _ = workloads.iid(N, 1, D, seed=70 + t)
        idx = rng.integers(-1, K + 1, N).astype(np.int32)     # includes invalid ids
        sums, counts = orc.update(X, idx, K)
        exp_s, exp_c = _exact_update(_exact(X), idx.tolist(), K, D)
        assert list(counts) == exp_c, t
        for j in range(K):
            for d in range(D):
                assert Fraction(float(sums[j, d])) == exp_s[j][d], (t, j, d)


def check_update_invariants(orc):
    X, C = workloads.integers(500, 23, 40, seed=11)
    idx, _ = orc.assign(X, C)
    sums, counts = orc.update(X, idx, 23)
    xs = X.to(torch.float64).numpy()
    assert counts.sum() == 500
    assert np.array_equal(sums.sum(0), xs.sum(0))                   # integers: exact
    perm = np.random.default_rng(3).permutation(500)
    s2, c2 = orc.update(X[perm], idx[perm], 23)
    assert np.array_equal(s2, sums) and np.array_equal(c2, counts)   # order-free on integers
    for j in (0, 5, 22):
        assert np.array_equal(sums[j], xs[idx == j].sum(0))


def check_lloyd_descent(orc):
    """For a fixed assignment the mean minimises the summed squared distance:
    replacing each used centroid by its points' mean never raises it."""
    X, C = workloads.blobs(400, 12, 16, seed=5)
    idx, _ = orc.assign(X, C)
    xs = X.to(torch.float64).numpy()
    cs = C.to(torch.float64).numpy()
    means, counts = orc.centroids(X, idx, C)
    before = ((xs - cs[idx]) ** 2).sum()
    after = ((xs - means[idx]) ** 2).sum()
    assert after <= before * (1 + 1e-12)
    # and any perturbation of a mean raises it (first-order optimality)
    j = int(np.argmax(counts))
    for delta in (1e-3, -1e-3):
        m2 = means.copy()
        m2[j, 0] += delta
        assert ((xs - m2[idx]) ** 2).sum() > after


def check_empty_cluster_keeps_centroid(orc):
    X, C = workloads.integers(20, 6, 8, seed=4)
    idx = np.zeros(20, dtype=np.int32)
    idx[10:] = 3
    means, counts = orc.centroids(X, idx, C)
    cs = C.to(torch.float64).numpy()
    xs = X.to(torch.float64).numpy()
    assert list(counts) == [10, 0, 0, 10, 0, 0]
    for j in (1, 2, 4, 5):
        assert np.array_equal(means[j], cs[j])
    assert np.array_equal(means[0], xs[:10].mean(0))
    assert np.array_equal(means[3], xs[10:].mean(0))


ALL_CHECKS += [check_update_rational, check_update_invariants, check_lloyd_descent,
               check_empty_cluster_keeps_centroid]


# ---------------------------------------------------------------- top-k
def check_topk_rational(orc, trials: int = 12):
    rng = np.random.default_rng(99)
    for t in range(trials):
        N = int(rng.integers(1, 7))
        K = int(rng.integers(1, 14))
        D = int(rng.integers(1, 10))
        k = int(rng.integers(1, K + 1))
        X, C = (workloads.integers(N, K, D, seed=40 + t, lo=-2, hi=2) if t % 2 == 0
                else workloads.iid(N, K, D, seed=40 + t))
        Xf, Cf = _exact(X), _exact(C)
        norms = [sum(c * c for c in row) for row in Cf]
        idx, sc = orc.topk(X, C, k)
        for r, x in enumerate(Xf):
            s = [(norms[j] - 2 * sum(a * b for a, b in zip(x, Cf[j])), j) for j in range(K)]
            s.sort()                                   # exact: by score, then index
            assert [j for _, j in s[:k]] == list(idx[r]), (t, r)
            for e in range(k):
                assert abs(Fraction(float(sc[r, e])) - s[e][0]) <= Fraction(1, 2**40) * (1 + abs(s[e][0]))


def check_topk_consistency(orc):
    # k = 1 is the assignment; numpy's stable argsort on exact integer scores
    X, C = workloads.integers(120, 60, 16, seed=3)
    C[30:35] = C[2]                                  # ties across the index range
    i1, s1 = orc.topk(X, C, 1)
    ia, sa = orc.assign(X, C)
    assert np.array_equal(i1[:, 0], ia) and np.array_equal(s1[:, 0], sa)
    xs = X.to(torch.float64).numpy()
    cs = C.to(torch.float64).numpy()
    S = (cs * cs).sum(1)[None, :] - 2.0 * (xs @ cs.T)
    ik, sk = orc.topk(X, C, 7)
    exp = np.argsort(S, axis=1, kind="stable")[:, :7]
    assert np.array_equal(ik, exp)
    assert np.array_equal(sk, np.take_along_axis(S, exp, 1))
    # an all-NaN row: the k lowest indices, every score NaN
    X2, C2 = workloads.integers(2, 9, 5, seed=8, lo=-1, hi=1)
    X2[0, 2] = math.nan
    ik, sk = orc.topk(X2, C2, 4)
    assert list(ik[0]) == [0, 1, 2, 3] and np.all(np.isnan(sk[0]))


ALL_CHECKS += [check_topk_rational, check_topk_consistency]


# ---------------------------------------------------------------- squared distance
def check_sqdist(orc):
    # exact rational brute force of sum_d (x_d - c_d)^2
    for t in range(6):
        X, C = workloads.iid(5, 6, 3 + 5 * t, seed=70 + t)
        Xf, Cf = _exact(X), _exact(C)
        ii = np.repeat(np.arange(5), 6)
        jj = np.tile(np.arange(6), 5)
        got = orc.sqdist(X, C, ii, jj)
        for p, (i, j) in enumerate(zip(ii, jj)):
            exact = sum((a - b) ** 2 for a, b in zip(Xf[i], Cf[j]))
            assert abs(Fraction(float(got[p])) - exact) <= Fraction(1, 2**45) * (1 + exact), (t, i, j)
    # zero exactly at the point itself, positive elsewhere
    X, _ = workloads.iid(8, 1, 32, seed=5)
    n = np.arange(8)
    assert np.all(orc.sqdist(X, X, n, n) == 0.0)
    assert np.all(orc.sqdist(X, X, n, (n + 1) % 8) > 0.0)
    # the norm expansion ||x||^2 + s agrees exactly on small integers
    Xi, Ci = workloads.integers(40, 30, 16, seed=9)
    ii = np.repeat(np.arange(40), 30)
    jj = np.tile(np.arange(30), 40)
    xs = Xi.to(torch.float64).numpy()
    xn = (xs * xs).sum(1)
    assert np.array_equal(orc.sqdist(Xi, Ci, ii, jj), xn[ii] + orc.scores(Xi, Ci, ii, jj))


ALL_CHECKS += [check_sqdist]
