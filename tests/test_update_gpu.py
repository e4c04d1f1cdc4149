"""The update step and the Lloyd loop on the GPU vs the fp64 oracle (GB300).

Rules: counts are integers and must match exactly.  Sums are fp32 additions
in an unspecified order; for centroid j and dimension d the bound is
    |gpu - exact| <= n_j * 2^-24 * sum_i |x_id|        (order-free fp32 bound)
plus exact equality on integer-valued data (every partial sum is an integer
below 2^24).  Means are sums / counts with one more rounding.
"""

import numpy as np
import pytest
import torch

import means_nearest_centroid_gb300 as km
import oracle
import workloads

pytestmark = pytest.mark.gpu
U = 2.0 ** -24


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from means_nearest_centroid_gb300 import _build
    _build.build()
    km.library()
    return torch.device("cuda:0")


def _abs_sums(X, idx, K):
    xs = np.abs(X.to(torch.float64).numpy())
    out = np.zeros((K, X.shape[1]))
    ok = (idx >= 0) & (idx < K)
    np.add.at(out, idx[ok], xs[ok])
    return out


def check_sums(X, idx, K, sums, counts, integer):
    o_sums, o_counts = oracle.update(X, idx, K)
    assert np.array_equal(counts.cpu().numpy().astype(np.int64), o_counts)
    g = sums.cpu().double().numpy()
    if integer:
        assert np.array_equal(g, o_sums)
    else:
        bound = o_counts[:, None] * U * _abs_sums(X, idx, K) + 1e-30
        assert np.all(np.abs(g - o_sums) <= bound), float(np.max(np.abs(g - o_sums) - bound))


METHODS = [0, 1, 2]   # automatic, atomic, sorted


@pytest.mark.parametrize("N,K,D", [(1, 1, 16), (1000, 37, 64), (5000, 300, 128), (3000, 17, 256),
                                   (2048, 1000, 48), (999, 5, 80), (20000, 5000, 96),
                                   (9000, 70000, 16), (40000, 40000, 32), (300000, 16385, 16),
                                   (70000, 65536, 16)])
@pytest.mark.parametrize("method", METHODS)
def test_update_float_and_integer(dev, N, K, D, method):
    """Ragged shapes; K past one scan tile of 16,384 bins, at the one-block
    limit 65,536 and past it (the multi-block scan)."""
    X, C = workloads.blobs(N, min(K, 4096), D, seed=N + D)
    g = np.random.default_rng(N)
    idx = g.integers(-2, K + 2, N).astype(np.int32)          # includes ids to skip
    sums, counts = km.kmassign_update(X.to(dev), torch.from_numpy(idx).to(dev), K, method=method)
    check_sums(X, idx, K, sums, counts, integer=False)
    Xi, _ = workloads.integers(N, 1, D, seed=N * 3)
    sums, counts = km.kmassign_update(Xi.to(dev), torch.from_numpy(idx).to(dev), K, method=method)
    check_sums(Xi, idx, K, sums, counts, integer=True)


@pytest.mark.parametrize("method", [1, 2])
def test_update_skewed_clusters(dev, method):
    """Most points on a few centroids (long runs), the rest spread thinly."""
    N, K, D = 50000, 3000, 64
    Xi, _ = workloads.integers(N, 1, D, seed=5)
    g = np.random.default_rng(5)
    idx = np.where(g.random(N) < 0.8, g.integers(0, 3, N), g.integers(0, K, N)).astype(np.int32)
    sums, counts = km.kmassign_update(Xi.to(dev), torch.from_numpy(idx).to(dev), K, method=method)
    check_sums(Xi, idx, K, sums, counts, integer=True)


@pytest.mark.parametrize("N,K,D", [(400_000, 1000, 64), (300_000, 2000, 16), (2_000_000, 500, 32)])
def test_update_sorted_many_points_per_centroid(dev, N, K, D):
    """N >> K: the sort counts in shared memory per block first."""
    Xi, _ = workloads.integers(N, 1, D, seed=K)
    g = np.random.default_rng(K)
    idx = g.integers(-1, K + 1, N).astype(np.int32)
    sums, counts = km.kmassign_update(Xi.to(dev), torch.from_numpy(idx).to(dev), K, method=2)
    check_sums(Xi, idx, K, sums, counts, integer=True)
    a = km.kmassign_update(Xi.to(dev), torch.from_numpy(idx).to(dev), K, method=1)
    assert torch.equal(a[0], sums) and torch.equal(a[1], counts)


def test_update_methods_agree_on_integers(dev):
    X, _ = workloads.integers(30000, 1, 128, seed=6)
    idx = torch.from_numpy(np.random.default_rng(6).integers(0, 900, 30000).astype(np.int32))
    Xd, idxd = X.to(dev), idx.to(dev)
    a = km.kmassign_update(Xd, idxd, 900, method=1)
    b = km.kmassign_update(Xd, idxd, 900, method=2)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


def test_update_rejects_unknown_method(dev):
    X, _ = workloads.integers(10, 1, 16, seed=1)
    idx = torch.zeros(10, dtype=torch.int32, device=dev)
    with pytest.raises(km.KmassignError):
        km.kmassign_update(X.to(dev), idx, 4, method=3)


@pytest.mark.parametrize("method", METHODS)
def test_update_accumulates_batches(dev, method):
    X, _ = workloads.integers(4000, 1, 64, seed=8)
    idx = np.random.default_rng(1).integers(0, 50, 4000).astype(np.int32)
    Xd, idxd = X.to(dev), torch.from_numpy(idx).to(dev)
    sums, counts = km.kmassign_update(Xd[:1500], idxd[:1500], 50, method=method)
    km.kmassign_update(Xd[1500:], idxd[1500:], 50, sums=sums, counts=counts, method=method)
    check_sums(X, idx, 50, sums, counts, integer=True)


def test_centroids_means_rounding_and_empty(dev):
    X, C = workloads.blobs(3000, 64, 128, seed=2)
    idx = np.random.default_rng(2).integers(0, 60, 3000).astype(np.int32)   # 60..63 empty
    Xd, Cd = X.to(dev), C.to(dev)
    sums, counts = km.kmassign_update(Xd, torch.from_numpy(idx).to(dev), 64)
    means = torch.empty(64, 128, dtype=torch.float32, device=dev)
    Cn = km.kmassign_centroids(sums, counts, Cd, means=means)
    o_means, o_counts = oracle.centroids(X, idx, C)
    m = means.cpu().double().numpy()
    bound = (o_counts[:, None] * U * _abs_sums(X, idx, 64) / np.maximum(o_counts, 1)[:, None]
             + np.abs(o_means) * U + 1e-30)
    assert np.all(np.abs(m - o_means) <= bound)
    # bf16 output is the round-to-nearest-even of the fp32 means
    assert torch.equal(Cn.cpu().view(torch.int16), means.cpu().to(torch.bfloat16).view(torch.int16))
    # empty clusters keep their centroid bit for bit
    assert torch.equal(Cn[60:].cpu().view(torch.int16), C[60:].view(torch.int16))
    # in place
    Cd2 = Cd.clone()
    km.kmassign_centroids(sums, counts, Cd2, C_new=Cd2)
    assert torch.equal(Cd2, Cn)


def test_lloyd_matches_host_driven_pieces(dev):
    X, C0 = workloads.adversarial(6000, 512, 64, seed=6)
    Xd = X.to(dev)
    C_loop = C0.to(dev).clone()
    idx_loop = km.kmassign_lloyd(Xd, C_loop, iters=3)
    assert km.kmassign_check() == 0
    C = C0.to(dev).clone()
    for _ in range(3):
        idx = km.kmassign(Xd, C)
        sums, counts = km.kmassign_update(Xd, idx, 512)
        km.kmassign_centroids(sums, counts, C, C_new=C)
    assert torch.equal(idx_loop, idx)
    assert torch.equal(C_loop.view(torch.int16), C.view(torch.int16))


def test_lloyd_one_iteration_vs_oracle(dev):
    X, C0 = workloads.integers(3000, 40, 32, seed=12)
    Xd = X.to(dev)
    C = C0.to(dev).clone()
    idx = km.kmassign_lloyd(Xd, C, iters=1)
    o_idx, _ = oracle.assign(X, C0)
    assert np.array_equal(idx.cpu().numpy(), o_idx)
    o_means, o_counts = oracle.centroids(X, o_idx, C0)
    # integer sums are exact; the GPU divides in fp32 then rounds to bf16, so
    # its centroid is within one bf16 step of the exact mean
    got = C.cpu().double().numpy()
    assert np.all(np.abs(got - o_means) <= np.abs(o_means) * 2.0 ** -8 + 1e-30)


def test_lloyd_rejects_negative_iterations(dev):
    X, C = workloads.integers(10, 4, 16, seed=1)
    with pytest.raises(km.KmassignError):
        km.kmassign_lloyd(X.to(dev), C.to(dev), iters=-1)


@pytest.mark.parametrize("method", [1, 2])
def test_update_full_size_lognormal(dev, method):
    w = workloads.WORKLOADS["lognormal_clusters"]
    X, C = workloads.make("lognormal_clusters")
    Xd, Cd = X.to(dev), C.to(dev)
    idx = km.kmassign(Xd, Cd)
    sums, counts = km.kmassign_update(Xd, idx, w.K, method=method)
    check_sums(X, idx.cpu().numpy(), w.K, sums, counts, integer=False)


def test_update_sorted_many_scan_tiles(dev):
    """K large enough that the tile offsets take several passes of one block."""
    N, K, D = 3000, 4_300_000, 16
    Xi, _ = workloads.integers(N, 1, D, seed=9)
    g = np.random.default_rng(9)
    idx = np.concatenate([g.integers(0, K, N - 100), np.full(100, K - 1)]).astype(np.int32)
    sums, counts = km.kmassign_update(Xi.to(dev), torch.from_numpy(idx).to(dev), K, method=2)
    o_sums, o_counts = oracle.update(Xi, idx, K)
    touched = np.unique(idx)
    assert np.array_equal(counts.cpu().numpy().astype(np.int64), o_counts)
    assert np.array_equal(sums[torch.from_numpy(touched).to(dev)].cpu().double().numpy(),
                          o_sums[touched])
    assert float(sums.abs().sum()) == float(np.abs(o_sums).sum())


@pytest.mark.parametrize("N,K,D", [
    (70000, 600, 256),      # sorted update, one-block scan, global scatter
    (131072, 256, 128),     # N >> K: block-local counting sort
    (66000, 70000, 256),    # K > 65,536: the scan takes three kernels
])
def test_lloyd_sorted_update_matches_host_driven_pieces(dev, N, K, D):
    """Sizes where the Lloyd loop takes the sorted update (N * D >= 2^24):
    the assignment counts the points per centroid as it stores idx, and the
    update starts from the scan of those counts.  On integer data every sum is
    exact, so two iterations must give the bits of the same steps made
    through the public calls (assignment, sorted update, new centroids)."""
    assert N * D >= 1 << 24
    X, C0 = workloads.integers(N, K, D, seed=N + K)
    Xd = X.to(dev)
    C_loop = C0.to(dev).clone()
    idx_loop = km.kmassign_lloyd(Xd, C_loop, iters=2)
    assert km.kmassign_check() == 0
    C = C0.to(dev).clone()
    for _ in range(2):
        idx = km.kmassign(Xd, C)
        sums, counts = km.kmassign_update(Xd, idx, K, method=2)
        km.kmassign_centroids(sums, counts, C, C_new=C)
    assert torch.equal(idx_loop, idx)
    assert torch.equal(C_loop.view(torch.int16), C.view(torch.int16))
