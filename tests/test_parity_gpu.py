"""CUDA path vs the fp64 oracle, through the C ABI (needs a GB300)."""

import json
import math
import os
import time

import numpy as np
import pytest
import torch

import means_nearest_centroid_gb300 as km
import oracle
import parity
import pins
import workloads

pytestmark = pytest.mark.gpu

PLANS = [
    dict(),                                                    # automatic
    dict(rows_per_cta=128, centroids_per_tile=128),
    dict(rows_per_cta=128, centroids_per_tile=256),
    dict(rows_per_cta=256, centroids_per_tile=128),
    dict(ksplit=3, rows_per_cta=256, centroids_per_tile=128),
    dict(ksplit=2, rows_per_cta=128, centroids_per_tile=256),
    dict(ksplit=5, rows_per_cta=128, centroids_per_tile=128),
    dict(ksplit=-2, rows_per_cta=256, centroids_per_tile=128),
    dict(rows_per_cta=256, centroids_per_tile=128, consumer_warps=16),
    dict(ksplit=2, rows_per_cta=128, centroids_per_tile=256, consumer_warps=16),
    dict(rows_per_cta=256, centroids_per_tile=256, consumer_warps=8),        # CTA pair
    dict(ksplit=3, rows_per_cta=256, centroids_per_tile=256, consumer_warps=16),
]


def is_pair(plan):
    return plan.get("rows_per_cta") == 256 and plan.get("centroids_per_tile") == 256


def plans_for(D):
    """The plans a shape can run: every compiled shape, at every D."""
    return list(PLANS)


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from means_nearest_centroid_gb300 import _build
    _build.build()
    km.library()
    return torch.device("cuda:0")


def run(dev, X, C, cnorm=None, with_cnorm=False, plan=None, minscore=True):
    Xd, Cd = X.to(dev), C.to(dev)
    cn = None
    if with_cnorm:
        cn = km.kmassign_norms(Cd)
    if cnorm is not None:
        cn = cnorm
    ms = torch.full((X.shape[0],), 12345.0, dtype=torch.float32, device=dev) if minscore else None
    idx = torch.full((X.shape[0],), -7, dtype=torch.int32, device=dev)
    if plan:
        km.kmassign_ex(Xd, Cd, cnorm=cn, idx=idx, minscore=ms, **plan)
    else:
        km.kmassign(Xd, Cd, cnorm=cn, idx=idx, minscore=ms)
    assert km.kmassign_check() == 0
    return idx.cpu(), (ms.cpu() if ms is not None else None)


def pad_d(t, D=16):
    out = torch.zeros(t.shape[0], D, dtype=torch.bfloat16)
    out[:, :t.shape[1]] = t
    return out


# ---------------------------------------------------------------- norms
@pytest.mark.parametrize("K,D", [(1, 16), (7, 64), (1000, 128), (4099, 256), (300, 48)])
def test_norms_match_oracle(dev, K, D):
    _, C = workloads.iid(1, K, D, seed=K + D)
    got = km.kmassign_norms(C.to(dev)).cpu().double().numpy()
    ref = oracle.norms(C)
    # sum of positive terms: relative error <= (D - 1) * 2^-24
    assert np.all(np.abs(got - ref) <= D * 2.0**-24 * ref + 1e-30)
    _, Ci = workloads.integers(1, K, D, seed=K * D)
    assert np.array_equal(km.kmassign_norms(Ci.to(dev)).cpu().double().numpy(), oracle.norms(Ci))


# ---------------------------------------------------------------- hand cases
@pytest.mark.parametrize("plan", PLANS[:4], ids=str)
def test_golden_cases(dev, plan):
    for case in pins.load_golden():
        X = pad_d(pins._bf16_rows(case["X"]))
        C = pad_d(pins._bf16_rows(case["C"]))
        idx, ms = run(dev, X, C, plan=plan)
        assert idx.tolist() == case["idx"], case["name"]
        for got, exp in zip(ms.tolist(), case["minscore"]):
            assert pins._same_score(got, pins._val(exp)), (case["name"], got, exp)


# ---------------------------------------------------------------- small shapes
SHAPES = [(1, 1, 16), (1, 3, 64), (5, 7, 32), (300, 130, 64), (129, 257, 256),
          (1000, 777, 128), (2000, 1000, 48), (4096, 128, 64), (333, 2049, 96),
          # D = 192 (CTA pairs by default), K past 65,536, ragged tails
          (97, 70001, 192), (513, 3001, 192), (260, 4100, 256)]


@pytest.mark.parametrize("N,K,D", SHAPES)
@pytest.mark.parametrize("pi", range(len(PLANS)))
def test_float_shapes_all_plans(dev, N, K, D, pi):
    X, C = workloads.blobs(N, K, D, seed=N * 7 + K * 3 + D)
    idx, ms = run(dev, X, C, plan=PLANS[pi], with_cnorm=(pi % 2 == 1))
    rep = parity.compare(X, C, idx, ms)
    assert rep.ok(), rep


@pytest.mark.parametrize("N,K,D", SHAPES)
def test_integer_shapes_bit_exact(dev, N, K, D):
    X, C = workloads.integers(N, K, D, seed=N + K + D)
    results = []
    for plan in plans_for(D):
        idx, ms = run(dev, X, C, plan=plan)
        rep = parity.compare(X, C, idx, ms, integer=True)
        assert rep.ok() and rep.idx_mismatches == 0, (plan, rep)
        results.append((idx, ms))
    for idx, ms in results[1:]:
        assert torch.equal(idx, results[0][0])
        assert torch.equal(ms.view(torch.int32), results[0][1].view(torch.int32))


def test_adversarial_reduced_bit_exact(dev):
    X, C = workloads.adversarial(6000, 2048, 64, seed=44)
    for plan in plans_for(64):
        idx, ms = run(dev, X, C, plan=plan)
        rep = parity.compare(X, C, idx, ms, integer=True)
        assert rep.ok() and rep.idx_mismatches == 0, (plan, rep)


SPLIT_PLANS = [
    dict(ksplit=2, rows_per_cta=128, centroids_per_tile=256),
    dict(ksplit=2, rows_per_cta=256, centroids_per_tile=256, consumer_warps=8),
    dict(ksplit=-2, rows_per_cta=256, centroids_per_tile=256, consumer_warps=8),
    dict(ksplit=3, rows_per_cta=256, centroids_per_tile=256, consumer_warps=8),
    dict(ksplit=4, rows_per_cta=256, centroids_per_tile=128),
]


@pytest.mark.parametrize("D", [64, 128, 256])
@pytest.mark.parametrize("nan_range", ["first", "last", "both"])
def test_split_ranges_that_see_no_number(dev, D, nan_range):
    """Split centroid ranges where one range, or every range, sees only NaN
    scores (centroids holding a NaN), and rows that are NaN themselves: the
    merged answer is the other range's winner, or idx 0 with a NaN score.
    Integer data, so every plan must match the oracle and each other bit for
    bit, whichever unit of a row finishes first."""
    N, K = 3000, 2048
    X, C = workloads.integers(N, K, D, seed=D + 5)
    X[7] = float("nan")
    X[2999, 3] = float("nan")
    half = K // 2
    if nan_range in ("first", "both"):
        C[:half, 0] = float("nan")
    if nan_range in ("last", "both"):
        C[half:, 1] = float("nan")
    ref = None
    for plan in SPLIT_PLANS:
        idx, ms = run(dev, X, C, plan=plan)
        rep = parity.compare(X, C, idx, ms, integer=True)
        assert rep.ok() and rep.idx_mismatches == 0, (plan, rep)
        if nan_range == "both":
            assert bool((idx == 0).all()) and bool(torch.isnan(ms).all()), plan
        elif nan_range == "first":
            finite = ~torch.isnan(X.float()).any(1)
            assert bool((idx[finite] >= half).all()), plan
        if ref is None:
            ref = (idx, ms)
            continue
        assert torch.equal(idx, ref[0]), plan
        assert torch.equal(ms.view(torch.int32), ref[1].view(torch.int32)), plan


@pytest.mark.parametrize("D", [96, 128, 192, 256])
def test_adversarial_specials_every_plan_wider_rows(dev, D):
    """Ties, twins, all-equal centroids and rows with NaN, +-inf and -0 on
    integer data at the widths the CTA pairs run (folding the norms up to
    D = 128): every plan bit-exact against the oracle and against each other."""
    N, K = 4000, 2048
    X, C = workloads.adversarial(N, K, D, seed=D)
    ref = None
    for plan in plans_for(D):
        idx, ms = run(dev, X, C, plan=plan)
        rep = parity.compare(X, C, idx, ms, integer=True)
        assert rep.ok() and rep.idx_mismatches == 0, (plan, rep)
        nan_rows = torch.isnan(X.float()).any(1)
        assert bool((idx[nan_rows] == 0).all()) and bool(torch.isnan(ms[nan_rows]).all()), plan
        if ref is None:
            ref = (idx, ms)
            continue
        assert torch.equal(idx, ref[0]), plan
        assert torch.equal(ms.view(torch.int32), ref[1].view(torch.int32)), plan


@pytest.mark.parametrize("D", [16, 48, 64, 96, 128, 192, 256])
def test_plans_give_identical_bits_on_float_data(dev, D):
    """Every plan (every tile shape, warp count and split, the CTA pairs
    included) returns the same idx and minscore bits on float data: at
    D <= 128 every kernel folds the norms into the MMA, above it none does, so
    a point's arithmetic does not depend on the plan.  The first plan is also
    checked against the oracle."""
    N, K = 1500, 1300
    X, C = workloads.iid(N, K, D, seed=99 + D)
    ref = None
    for plan in plans_for(D):
        idx, ms = run(dev, X, C, plan=plan)
        if ref is None:
            rep = parity.compare(X, C, idx, ms)
            assert rep.ok(), (plan, rep)
            ref = (idx, ms)
            continue
        assert torch.equal(idx, ref[0]), plan
        assert torch.equal(ms.view(torch.int32), ref[1].view(torch.int32)), plan


@pytest.mark.parametrize("D", [64, 96, 128, 192, 256])
def test_answers_do_not_depend_on_the_batch(dev, D):
    """A point's idx and minscore bits are the same whether it is assigned
    alone, in a slice of the rows or with all of them, although the planner
    picks different shapes and splits for the different N (at D = 96 and 128
    the whole batch runs on CTA pairs, the small slices on single blocks)."""
    N, K = 70000, 4096
    X, C = workloads.iid(N, K, D, seed=7 * D)
    Xd, Cd = X.to(dev), C.to(dev)
    cn = km.kmassign_norms(Cd)
    ms = torch.empty(N, dtype=torch.float32, device=dev)
    idx = km.kmassign(Xd, Cd, cnorm=cn, minscore=ms)
    plans = {str(km.kmassign_plan(N, K, D))}
    for a, b in [(0, 1), (5, 300), (1000, 9000), (40000, 70000), (123, 65659)]:
        ms_s = torch.empty(b - a, dtype=torch.float32, device=dev)
        idx_s = km.kmassign(Xd[a:b].contiguous(), Cd, cnorm=cn, minscore=ms_s)
        plans.add(str(km.kmassign_plan(b - a, K, D)))
        assert torch.equal(idx_s, idx[a:b]), (a, b)
        assert torch.equal(ms_s.view(torch.int32), ms[a:b].view(torch.int32)), (a, b)
    assert km.kmassign_check() == 0
    assert len(plans) >= 2


def test_repeat_runs_are_bitwise_identical(dev):
    X, C = workloads.iid(3000, 2500, 64, seed=3)
    Xd, Cd = X.to(dev), C.to(dev)
    first = km.kmassign(Xd, Cd).clone()
    for _ in range(20):
        assert torch.equal(km.kmassign(Xd, Cd), first)


def test_minscore_optional_and_idx_only(dev):
    X, C = workloads.blobs(700, 300, 64, seed=8)
    idx_a, _ = run(dev, X, C, minscore=False)
    idx_b, _ = run(dev, X, C, minscore=True)
    assert torch.equal(idx_a, idx_b)


def test_empty_input(dev):
    X = torch.empty(0, 64, dtype=torch.bfloat16, device=dev)
    C = torch.ones(4, 64, dtype=torch.bfloat16, device=dev)
    idx = km.kmassign(X, C)
    assert idx.numel() == 0


def test_host_pointer_rejected(dev):
    X, C = workloads.iid(10, 4, 64, seed=1)
    lib = km.library()
    idx = torch.empty(10, dtype=torch.int32, device=dev)
    rc = lib.kmassign(km._ptr(X), km._ptr(C.to(dev)), km._ptr(None), 10, 4, 64, km._ptr(idx),
                      km._ptr(None), km._stream_ptr(None))
    assert rc == km.STATUS["KMASSIGN_ERR_NOT_DEVICE"]


def test_assign_host_end_to_end(dev):
    X, C = workloads.blobs(1000, 200, 128, seed=12)
    got = km.assign_host(X.pin_memory(), C.pin_memory())
    rep = parity.compare(X, C, got, None)
    assert rep.ok(), rep


def _host_call(X, C, cnorm=None, minscore=False, rows=0, pin=True):
    """kmassign_host_ex straight through the C ABI with host buffers."""
    N, D = X.shape
    K = C.shape[0]
    hold = (lambda t: t.pin_memory()) if pin else (lambda t: t.contiguous())
    Xh, Ch = hold(X), hold(C)
    cn = None if cnorm is None else hold(cnorm)
    idx = hold(torch.full((N,), -1, dtype=torch.int32))
    ms = hold(torch.full((N,), 7.0)) if minscore else None
    rc = km.library().kmassign_host_ex(km._ptr(Xh), km._ptr(Ch), km._ptr(cn), N, K, D,
                                       km._ptr(idx), km._ptr(ms), rows, km._stream_ptr(None))
    return rc, idx, ms


@pytest.mark.parametrize("N,K,D,gen", [
    (70001, 3000, 64, workloads.integers),     # several slices, ragged last one
    (5000, 16384, 96, workloads.integers),     # one slice, split centroid range
    (40000, 700, 256, workloads.integers),
])
def test_host_path_matches_oracle_bit_exact(dev, N, K, D, gen):
    """The host-buffer entry point against the oracle on integer data, where
    every fp32 step is exact: idx and minscore bit for bit."""
    X, C = gen(N, K, D, seed=N + K)
    rc, idx, ms = _host_call(X, C, minscore=True)
    assert rc == 0, km.kmassign_strerror(rc)
    rep = parity.compare(X, C, idx, ms, integer=True)
    assert rep.ok() and rep.idx_mismatches == 0, rep


@pytest.mark.parametrize("N,K,D,rows", [
    (3, 300, 64, 0), (1001, 300, 64, 250), (5000, 300, 64, 1), (6000, 1000, 128, 777),
    (90000, 16384, 96, 0), (90000, 4096, 128, 20000), (50000, 2000, 192, 0),
    (30000, 5000, 256, 4096),
])
def test_host_path_slices_match_whole_call(dev, N, K, D, rows):
    """Any slicing (forced or automatic) gives the bits of one kmassign call
    over all points, with the norms computed inside or given."""
    X, C = workloads.blobs(N, K, D, seed=N + D)
    Xd, Cd = X.to(dev), C.to(dev)
    cn = km.kmassign_norms(Cd)
    ref_ms = torch.empty(N, dtype=torch.float32, device=dev)
    ref = km.kmassign(Xd, Cd, cnorm=cn, minscore=ref_ms).cpu()
    for given in (False, True):
        rc, idx, ms = _host_call(X, C, cnorm=cn.cpu() if given else None, minscore=True,
                                 rows=rows)
        assert rc == 0, km.kmassign_strerror(rc)
        assert torch.equal(idx, ref)
        assert torch.equal(ms.view(torch.int32), ref_ms.cpu().view(torch.int32))


def test_host_path_pageable_memory(dev):
    """Pageable (unpinned) host buffers work too; the copies just do not overlap."""
    X, C = workloads.blobs(20000, 500, 128, seed=3)
    rc, idx, _ = _host_call(X, C, rows=3000, pin=False)
    assert rc == 0
    assert torch.equal(idx, km.kmassign(X.to(dev), C.to(dev)).cpu())


def test_host_path_rejects_device_pointers(dev):
    X, C = workloads.blobs(100, 50, 64, seed=4)
    idx = torch.empty(100, dtype=torch.int32, device=dev)
    rc = km.library().kmassign_host(km._ptr(X), km._ptr(C), None, 100, 50, 64, km._ptr(idx),
                                    None, km._stream_ptr(None))
    assert rc == km.STATUS["KMASSIGN_ERR_NOT_HOST"]


def test_host_path_on_a_side_stream(dev):
    """The caller's stream orders the call after its earlier work."""
    X, C = workloads.blobs(8000, 900, 64, seed=5)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        torch.cuda._sleep(1000000)
        got = km.assign_host(X.pin_memory(), C.pin_memory(), stream=s, rows_per_slice=1500)
    assert torch.equal(got, km.kmassign(X.to(dev), C.to(dev)).cpu())


def test_non_default_stream(dev):
    X, C = workloads.blobs(2000, 600, 64, seed=13)
    s = torch.cuda.Stream()
    Xd, Cd = X.to(dev), C.to(dev)
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        idx = km.kmassign(Xd, Cd, stream=s)
    s.synchronize()
    rep = parity.compare(X, C, idx.cpu(), None)
    assert rep.ok(), rep


def test_many_centroids(dev):
    """K = 100,000 (many tiles, a ragged last tile, plans that split K)."""
    X, C = workloads.blobs(3000, 100000, 16, seed=77)
    idx, ms = run(dev, X, C)
    rows = np.arange(0, 3000, 7)
    rep = parity.compare(X, C, idx, ms, rows=rows)
    assert rep.ok(), rep


# ---------------------------------------------------------------- full sizes
def _record(entry):
    """Append one JSON line to the file named by KMASSIGN_PARITY_REPORT, if set."""
    path = os.environ.get("KMASSIGN_PARITY_REPORT")
    if path:
        with open(path, "a") as f:
            f.write(json.dumps(entry) + "\n")


@pytest.mark.parametrize("key", workloads.ORDER)
def test_full_size_workloads(dev, key):
    """Every row of each of the five workloads, at full size, against the
    oracle: bit-exact idx and minscore on integer data, the tolerance rule on
    float data.  The number of rows whose idx differs from the oracle's (each
    within the tolerance) and the largest accepted gap are printed and, with
    KMASSIGN_PARITY_REPORT set, appended to that file."""
    w = workloads.WORKLOADS[key]
    X, C = workloads.make(key)
    Xd, Cd = X.to(dev), C.to(dev)
    cn = km.kmassign_norms(Cd) if w.precomputed_norms else None
    ms = torch.empty(w.N, dtype=torch.float32, device=dev)
    idx = km.kmassign(Xd, Cd, cnorm=cn, minscore=ms)
    assert km.kmassign_check() == 0
    plan = km.kmassign_plan(w.N, w.K, w.D)
    idx, ms = idx.cpu(), ms.cpu()
    t0 = time.time()
    rep = parity.compare(X, C, idx, ms, rows=None, integer=w.integer)
    entry = dict(workload=key, N=w.N, K=w.K, D=w.D, rows=rep.rows,
                 idx_mismatches=rep.idx_mismatches, rejected=rep.rejected,
                 minscore_bad=rep.minscore_bad, worst_gap=rep.worst_gap,
                 integer=bool(w.integer), oracle_s=round(time.time() - t0, 1),
                 plan=plan)
    print(entry)
    _record(entry)
    assert rep.rows == w.N
    assert rep.ok(), rep
    if w.integer:
        assert rep.idx_mismatches == 0
    # properties that hold on every row at any size
    assert int(idx.min()) >= 0 and int(idx.max()) < w.K
    if w.key == "adversarial_ties":
        # twins: the lower copy always wins over its duplicate at j + K/2
        finite = torch.isfinite(ms)
        assert bool((idx[finite] < w.K // 2).all())
        nan_rows = torch.isnan(X.float()).any(1)
        assert bool((idx[nan_rows] == 0).all()) and bool(torch.isnan(ms[nan_rows]).all())


# ---------------------------------------------------------------- wave-tail split
# More row tiles than thread blocks: the tail split keeps the first full waves
# whole and splits only the last, partial wave (on a 152-SM GB300: 152 whole
# row tiles, 5 split).
TAIL_CASES = [
    (20000, 700, 64, dict(ksplit=-2, rows_per_cta=128, centroids_per_tile=128)),
    (20000, 700, 64, dict(ksplit=-3, rows_per_cta=128, centroids_per_tile=256)),
    (40000, 300, 32, dict(ksplit=-2, rows_per_cta=256, centroids_per_tile=128)),
    (40000, 1000, 48, dict(ksplit=-4, rows_per_cta=256, centroids_per_tile=128)),
    (40000, 1000, 48, dict(ksplit=-3, rows_per_cta=256, centroids_per_tile=128,
                           consumer_warps=16)),
    (20000, 700, 64, dict(ksplit=-2, rows_per_cta=128, centroids_per_tile=256,
                          consumer_warps=16)),
    (40000, 700, 256, dict(ksplit=-2, rows_per_cta=256, centroids_per_tile=256,
                           consumer_warps=8)),
]


@pytest.mark.parametrize("N,K,D,plan", TAIL_CASES, ids=str)
def test_tail_split_matches_oracle_and_whole_plan(dev, N, K, D, plan):
    X, C = workloads.blobs(N, K, D, seed=N + K)
    idx, ms = run(dev, X, C, plan=plan)
    whole = dict(plan, ksplit=1)
    idx1, ms1 = run(dev, X, C, plan=whole)
    assert torch.equal(idx, idx1)
    assert torch.equal(ms.view(torch.int32), ms1.view(torch.int32))
    g = np.random.default_rng(N)
    rows = np.unique(np.concatenate([g.choice(N, 3000, replace=False), np.arange(N - 2000, N)]))
    rep = parity.compare(X, C, idx, ms, rows=rows)
    assert rep.ok(), rep
    Xi, Ci = workloads.integers(N, K, D, seed=N - K)
    idx, ms = run(dev, Xi, Ci, plan=plan)
    rep = parity.compare(Xi, Ci, idx, ms, rows=rows, integer=True)
    assert rep.ok() and rep.idx_mismatches == 0, rep


def test_invalid_tail_value_rejected(dev):
    X, C = workloads.iid(10, 4, 64, seed=2)
    with pytest.raises(km.KmassignError):
        km.kmassign_ex(X.to(dev), C.to(dev), ksplit=-1)


# ---------------------------------------------------------------- random shapes
def _random_cases(n, seed=2026):
    g = np.random.default_rng(seed)
    cases = []
    for c in range(n):
        N = int(g.integers(1, 3000))
        K = int(g.integers(1, 5000))
        D = int(g.choice([16, 32, 48, 64, 80, 96, 112, 128, 160, 192, 224, 256]))
        plan = PLANS[int(g.integers(0, len(PLANS)))]
        cases.append((N, K, D, plan))
    return cases


@pytest.mark.parametrize("N,K,D,plan", _random_cases(40), ids=str)
def test_random_shapes_and_plans(dev, N, K, D, plan):
    """Seeded random ragged shapes on a random forced plan (every shape runs
    at every D): integer data bit-exact against the oracle, float data within
    the tolerance."""
    Xi, Ci = workloads.integers(N, K, D, seed=N * 3 + K + D)
    idx, ms = run(dev, Xi, Ci, plan=plan)
    rep = parity.compare(Xi, Ci, idx, ms, integer=True)
    assert rep.ok() and rep.idx_mismatches == 0, (plan, rep)
    X, C = workloads.blobs(N, K, D, seed=N + K * 3 + D)
    idx, ms = run(dev, X, C, plan=plan)
    rep = parity.compare(X, C, idx, ms)
    assert rep.ok(), (plan, rep)
