"""The k nearest centroids and squared distances on the GPU vs the fp64 oracle
(needs a GB300).  Rules in ``parity.compare_topk``: exact lists and values on
integer data; on float data the exact score of every pick within the fp32
error of the oracle's order statistic."""

import numpy as np
import pytest
import torch

import means_nearest_centroid_gb300 as km
import oracle
import parity
import pins
import workloads

pytestmark = pytest.mark.gpu

SPLITS = [0, 2, 3, 5, -2, -3]
# (N, K, D, k): ragged N and K, every list size (4, 8, 16, 32), k == K
SHAPES = [(1, 1, 16, 1), (1, 3, 64, 3), (5, 7, 32, 4), (300, 130, 64, 8), (129, 257, 256, 16),
          (1000, 777, 128, 32), (2000, 1000, 48, 5), (333, 2049, 96, 10), (600, 32, 64, 32),
          (4100, 300, 16, 2), (300, 2049, 192, 8)]


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from means_nearest_centroid_gb300 import _build
    _build.build()
    km.library()
    return torch.device("cuda:0")


def run(dev, X, C, k, distances=False, ksplit=0, with_cnorm=False, with_score=True):
    Xd, Cd = X.to(dev), C.to(dev)
    cn = km.kmassign_norms(Cd) if with_cnorm else None
    idx = torch.full((X.shape[0], k), -7, dtype=torch.int32, device=dev)
    sc = (torch.full((X.shape[0], k), 12345.0, dtype=torch.float32, device=dev)
          if with_score or distances else None)
    km.kmassign_topk(Xd, Cd, k, cnorm=cn, idx=idx, score=sc, distances=distances, ksplit=ksplit)
    assert km.kmassign_check() == 0
    return idx.cpu(), (None if sc is None else sc.cpu())


@pytest.mark.parametrize("N,K,D,k", SHAPES)
@pytest.mark.parametrize("ksplit", SPLITS)
def test_float_shapes_every_split(dev, N, K, D, k, ksplit):
    X, C = workloads.blobs(N, K, D, seed=N * 5 + K + D)
    idx, sc = run(dev, X, C, k, ksplit=ksplit, with_cnorm=(ksplit % 2 == 1))
    rep = parity.compare_topk(X, C, idx, sc, k)
    assert rep.ok(), rep


@pytest.mark.parametrize("N,K,D,k", SHAPES)
def test_integer_shapes_bit_exact_every_split(dev, N, K, D, k):
    X, C = workloads.integers(N, K, D, seed=N + 2 * K + D)
    ref = None
    for ks in SPLITS:
        idx, sc = run(dev, X, C, k, ksplit=ks)
        rep = parity.compare_topk(X, C, idx, sc, k, integer=True)
        assert rep.ok() and rep.idx_mismatches == 0, (ks, rep)
        if ref is None:
            ref = (idx, sc)
        assert torch.equal(idx, ref[0]) and torch.equal(sc.view(torch.int32), ref[1].view(torch.int32))


@pytest.mark.parametrize("N,K,D,k", [(700, 300, 64, 8), (129, 2049, 256, 32), (5000, 64, 16, 4),
                                     (900, 500, 128, 1)])
@pytest.mark.parametrize("ksplit", [0, 3])
def test_distances(dev, N, K, D, k, ksplit):
    Xi, Ci = workloads.integers(N, K, D, seed=K + k)
    idx, d = run(dev, Xi, Ci, k, distances=True, ksplit=ksplit)
    rep = parity.compare_topk(Xi, Ci, idx, d, k, integer=True, distances=True)
    assert rep.ok() and rep.idx_mismatches == 0, rep
    X, C = workloads.blobs(N, K, D, seed=N + k)
    idx, d = run(dev, X, C, k, distances=True, ksplit=ksplit)
    rep = parity.compare_topk(X, C, idx, d, k, distances=True)
    assert rep.ok(), rep
    assert torch.all(d >= 0)
    # the same picks as the score output
    idx2, _ = run(dev, X, C, k, ksplit=ksplit)
    assert torch.equal(idx, idx2)


def test_k1_is_the_assignment(dev):
    X, C = workloads.adversarial(5000, 3000, 64, seed=9)
    Xd, Cd = X.to(dev), C.to(dev)
    ms = torch.empty(5000, dtype=torch.float32, device=dev)
    ref = km.kmassign(Xd, Cd, minscore=ms).cpu()
    for ks in SPLITS:
        idx, sc = run(dev, X, C, 1, ksplit=ks)
        assert torch.equal(idx[:, 0], ref), ks
        assert torch.equal(sc[:, 0].view(torch.int32), ms.cpu().view(torch.int32)), ks


def test_golden_cases(dev):
    """Every hand case through the full ordering (k = K) and k = 1."""
    for case in pins.load_golden():
        X = pins._bf16_rows(case["X"])
        C = pins._bf16_rows(case["C"])
        Xp = torch.zeros(X.shape[0], 16, dtype=torch.bfloat16)
        Cp = torch.zeros(C.shape[0], 16, dtype=torch.bfloat16)
        Xp[:, :X.shape[1]] = X
        Cp[:, :C.shape[1]] = C
        K = C.shape[0]
        idx, sc = run(dev, Xp, Cp, 1)
        assert idx[:, 0].tolist() == case["idx"], case["name"]
        for got, exp in zip(sc[:, 0].tolist(), case["minscore"]):
            assert pins._same_score(got, pins._val(exp)), (case["name"], got, exp)
        k = min(K, 32)
        idx, sc = run(dev, Xp, Cp, k)
        rep = parity.compare_topk(Xp, Cp, idx, sc, k, integer=True)
        assert rep.ok() and rep.idx_mismatches == 0, (case["name"], rep)


@pytest.mark.parametrize("k", [4, 16])
def test_adversarial_ties_bit_exact(dev, k):
    X, C = workloads.adversarial(6000, 2048, 64, seed=44)
    for ks in SPLITS:
        idx, sc = run(dev, X, C, k, ksplit=ks)
        rep = parity.compare_topk(X, C, idx, sc, k, integer=True)
        assert rep.ok() and rep.idx_mismatches == 0, (ks, rep)


def test_nan_rows_and_nan_centroids(dev):
    """All-NaN rows list the lowest indices with NaN scores; a NaN centroid
    ranks after every number; +-inf rows keep their order."""
    X, C = workloads.integers(600, 300, 32, seed=5)
    X[::7, 3] = float("nan")
    X[1::11, 0] = float("inf")
    X[2::13, 5] = float("-inf")
    C[::17, 1] = float("nan")
    for k in (3, 8, 20):
        for ks in SPLITS[:4]:
            idx, sc = run(dev, X, C, k, ksplit=ks)
            rep = parity.compare_topk(X, C, idx, sc, k, integer=True)
            assert rep.ok() and rep.idx_mismatches == 0, (k, ks, rep)
    assert idx[0].tolist() == list(range(20)) and torch.all(torch.isnan(sc[0]))


def test_descending_scores_insert_every_column(dev):
    """Centroids ordered so every new column beats the list (worst case)."""
    D, K, N = 16, 2000, 300
    C = torch.zeros(K, D, dtype=torch.bfloat16)
    C[:, 0] = torch.linspace(-1.0, 1.0, K).to(torch.bfloat16)    # x . c grows with j
    X = torch.zeros(N, D, dtype=torch.bfloat16)
    X[:, 0] = 1.0
    X[:, 1] = torch.arange(N).to(torch.bfloat16) / 64
    for k in (1, 7, 32):
        idx, sc = run(dev, X, C, k)
        rep = parity.compare_topk(X, C, idx, sc, k, integer=False)
        assert rep.ok(), (k, rep)


def test_score_optional(dev):
    X, C = workloads.blobs(900, 500, 64, seed=4)
    a, _ = run(dev, X, C, 8, with_score=False)
    b, _ = run(dev, X, C, 8)
    assert torch.equal(a, b)


def test_repeat_runs_are_bitwise_identical(dev):
    X, C = workloads.iid(3000, 2500, 128, seed=3)
    first = run(dev, X, C, 10)
    for _ in range(5):
        again = run(dev, X, C, 10)
        assert torch.equal(again[0], first[0])
        assert torch.equal(again[1].view(torch.int32), first[1].view(torch.int32))


def test_empty_input(dev):
    X = torch.empty(0, 64, dtype=torch.bfloat16, device=dev)
    C = torch.ones(40, 64, dtype=torch.bfloat16, device=dev)
    idx, sc = km.kmassign_topk(X, C, 8)
    assert idx.shape == (0, 8) and sc.shape == (0, 8)


def test_argument_errors(dev):
    X, C = workloads.iid(10, 5, 64, seed=1)
    Xd, Cd = X.to(dev), C.to(dev)
    for k in (0, 6):
        with pytest.raises(km.KmassignError):
            km.kmassign_topk(Xd, Cd, k)


@pytest.mark.parametrize("key,k", [("sampled_centroids", 8), ("iid_normal", 16),
                                   ("adversarial_ties", 32), ("lognormal_clusters", 4)])
def test_full_size_workloads_sampled_rows(dev, key, k):
    """Full-size inputs; the oracle checks a sample of rows (every 97th, the
    first and last 128, every row of the ragged last tile)."""
    w = workloads.WORKLOADS[key]
    X, C = workloads.make(key)
    idx, sc = run(dev, X, C, k)
    N = w.N
    rows = sorted(set(range(0, N, 97 if N < 500000 else 397)) | set(range(128))
                  | set(range(N - 128, N)))
    rep = parity.compare_topk(X, C, idx, sc, k, rows=rows, integer=w.integer)
    assert rep.ok(), rep
    if w.integer:
        assert rep.idx_mismatches == 0, rep
