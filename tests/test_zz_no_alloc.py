"""kmassign_noalloc against kmassign, through the C ABI (needs a GB300).

kmassign_noalloc serves callers that cannot let a library allocate device
memory while they run (a host framework that owns all device memory and
hands a plugin only buffers and a stream, or a service whose memory budget
is fixed at start-up because cudaMalloc/cudaFree can synchronise the
device).  Its temporaries come from one static device array.  Each case
calls it twice in a row -- the second call finds the first call's leftovers
in that array -- and both answers must equal those of kmassign, which takes
its temporaries from the stream allocator.  This file is collected last so
that a stop at the first failure has already run every other test.
"""

import ctypes

import pytest
import torch

import means_nearest_centroid_gb300 as km
import workloads

pytestmark = pytest.mark.gpu

CASES = [
    # (N, K, D, cnorm given, generator): small N makes the plan split the
    # centroid range, so the packed keys live in the static array too
    (2048, 16384, 64, False, workloads.iid),
    (3000, 5000, 128, False, workloads.blobs),
    (1000, 4096, 256, True, workloads.integers),
    (70000, 3000, 64, False, workloads.blobs),
    (20000, 8192, 192, False, workloads.blobs),   # CTA-pair plan, tail split
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


@pytest.mark.parametrize("N,K,D,given,gen", CASES)
def test_noalloc_matches_kmassign_twice(dev, N, K, D, given, gen):
    X, C = gen(N, K, D, seed=N + K + D)
    Xd, Cd = X.to(dev), C.to(dev)
    cn = km.kmassign_norms(Cd) if given else None
    ref_idx = torch.empty(N, dtype=torch.int32, device=dev)
    ref_ms = torch.empty(N, dtype=torch.float32, device=dev)
    # Where kmassign would run the CTA pair that folds the norms (64 < D <=
    # 128), this entry point has no room for its fold operand and runs the
    # 256-row single-block shape: compare with that plan, bit for bit.
    auto = km.kmassign_plan(N, K, D)
    pair_fold = 64 < D <= 128 and (auto["rows_per_cta"], auto["centroids_per_tile"]) == (256, 256)
    plan = dict(rows_per_cta=256, centroids_per_tile=128) if pair_fold else {}
    km.kmassign_ex(Xd, Cd, cnorm=cn, idx=ref_idx, minscore=ref_ms, **plan)
    assert km.kmassign_check() == 0
    for _ in range(2):
        idx = torch.full((N,), -1, dtype=torch.int32, device=dev)
        ms = torch.full((N,), 7.0, dtype=torch.float32, device=dev)
        assert _call_noalloc(Xd, Cd, cn, idx, ms) == 0
        assert km.kmassign_check() == 0
        assert torch.equal(idx, ref_idx)
        assert torch.equal(ms.view(torch.int32), ref_ms.view(torch.int32))


def test_noalloc_rejects_norms_beyond_its_array(dev):
    X = torch.zeros(4, 16, dtype=torch.bfloat16, device=dev)
    C = torch.zeros((1 << 20) + 1, 16, dtype=torch.bfloat16, device=dev)
    idx = torch.empty(4, dtype=torch.int32, device=dev)
    rc = _call_noalloc(X, C, None, idx, None)
    assert rc == km.STATUS["KMASSIGN_ERR_SCRATCH"]
    assert "static" in km.kmassign_strerror(rc)
