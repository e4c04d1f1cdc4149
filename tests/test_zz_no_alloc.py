"""kmassign_noalloc against kmassign, through the C ABI (needs a GB300).

kmassign_noalloc serves callers that cannot let a library allocate device
memory while they run (a host framework that owns all device memory and
hands a plugin only buffers and a stream, or a service whose memory budget
is fixed at start-up because cudaMalloc/cudaFree can synchronise the
device).  Its temporaries come from one static device array.  Each case
calls it twice in a row -- the second call finds the first call's leftovers
in that array -- and both answers must equal those of kmassign, which takes
its temporaries from the stream allocator.  Every plan gives the same bits,
so the comparison is bit for bit even where this entry point has to run a
different plan.  This file is collected last so that a stop at the first
failure has already run every other test.
"""

import pytest
import torch

import means_nearest_centroid_gb300 as km
import workloads

pytestmark = pytest.mark.gpu

KEY_MAX = 1 << 18   # points whose packed keys the static array holds

CASES = [
    # (N, K, D, cnorm given, generator, what the automatic plan needs)
    # small N: the plan splits the centroid range, keys in the static array
    (2048, 16384, 64, False, workloads.iid, "split"),
    (3000, 5000, 128, False, workloads.blobs, "split"),
    (1000, 4096, 256, True, workloads.integers, "split"),
    (70000, 3000, 64, False, workloads.blobs, None),
    (20000, 8192, 192, False, workloads.blobs, None),
    # CTA pairs that fold the norms read a fold operand from global memory:
    # this entry point plans without pairs instead
    (65536, 4096, 128, False, workloads.iid, "fold_pair"),
    (65536, 16384, 96, True, workloads.blobs, "fold_pair"),
]


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from means_nearest_centroid_gb300 import _build
    _build.build()
    km.library()
    return torch.device("cuda:0")


def _call_noalloc(X, C, cn, idx, ms):
    lib = km.library()
    return lib.kmassign_noalloc(km._ptr(X), km._ptr(C), km._ptr(cn), X.shape[0], C.shape[0],
                                X.shape[1], km._ptr(idx), km._ptr(ms), km._stream_ptr(None))


def _needs(plan, N):
    """What the automatic plan needs beyond the static array."""
    pair = (plan["rows_per_cta"], plan["centroids_per_tile"]) == (256, 256)
    split_rows = N - plan["whole_row_tiles"] * plan["rows_per_cta"]
    return dict(split=plan["ksplit"] > 1, fold_pair=pair,
                many_keys=plan["ksplit"] > 1 and split_rows > KEY_MAX)


@pytest.mark.parametrize("N,K,D,given,gen,need", CASES)
def test_noalloc_matches_kmassign_twice(dev, N, K, D, given, gen, need):
    X, C = gen(N, K, D, seed=N + K + D)
    if need is not None:
        # the case reaches the branch it is here for
        assert _needs(km.kmassign_plan(N, K, D), N)[need], km.kmassign_plan(N, K, D)
    Xd, Cd = X.to(dev), C.to(dev)
    cn = km.kmassign_norms(Cd) if given else None
    ref_idx = torch.empty(N, dtype=torch.int32, device=dev)
    ref_ms = torch.empty(N, dtype=torch.float32, device=dev)
    km.kmassign(Xd, Cd, cnorm=cn, idx=ref_idx, minscore=ref_ms)
    assert km.kmassign_check() == 0
    for _ in range(2):
        idx = torch.full((N,), -1, dtype=torch.int32, device=dev)
        ms = torch.full((N,), 7.0, dtype=torch.float32, device=dev)
        assert _call_noalloc(Xd, Cd, cn, idx, ms) == 0
        assert km.kmassign_check() == 0
        assert torch.equal(idx, ref_idx)
        assert torch.equal(ms.view(torch.int32), ref_ms.view(torch.int32))


def test_noalloc_many_split_points(dev):
    """A split centroid range over more points than the array's keys hold
    makes this entry point plan without a split.  The planner splits all row
    tiles only when there are too few of them to fill the GPU, and otherwise
    splits the last, partial wave (at most one wave of row tiles), so on a
    full GB300 no automatic plan needs that many keys: search a grid of shapes
    with large K for one, and run any that does."""
    found = []
    for D in (16, 64, 128):
        for N in (262400, 300000, 330000, 400000, 600000):
            for K in (1 << 17, 1 << 19, 1 << 21):
                if _needs(km.kmassign_plan(N, K, D), N)["many_keys"]:
                    found.append((N, K, D))
    for N, K, D in found[:2]:
        X, C = workloads.iid(N, K, D, seed=N + K)
        Xd, Cd = X.to(dev), C.to(dev)
        cn = km.kmassign_norms(Cd)
        ref = km.kmassign(Xd, Cd, cnorm=cn)
        idx = torch.full((N,), -1, dtype=torch.int32, device=dev)
        assert _call_noalloc(Xd, Cd, cn, idx, None) == 0
        assert km.kmassign_check() == 0
        assert torch.equal(idx, ref)
    print("automatic plans splitting more points than the array holds:", found)


def test_noalloc_rejects_norms_beyond_its_array(dev):
    X = torch.zeros(4, 16, dtype=torch.bfloat16, device=dev)
    C = torch.zeros((1 << 20) + 1, 16, dtype=torch.bfloat16, device=dev)
    idx = torch.empty(4, dtype=torch.int32, device=dev)
    rc = _call_noalloc(X, C, None, idx, None)
    assert rc == km.STATUS["KMASSIGN_ERR_SCRATCH"]
    assert "static" in km.kmassign_strerror(rc)
