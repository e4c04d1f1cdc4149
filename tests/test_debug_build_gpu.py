"""The debug build (KMASSIGN_DEBUG) on the GPU: device-side consistency
checks of the planned layout, rings, work units and split-key indices, which
record KMASSIGN_ERR_DEBUG_CHECK instead of trapping.  Every plan shape and
split runs through it; the status must stay clean and the answers must equal
the normal build's bit for bit.  (compute-sanitizer is closed on this machine;
this is the device-side stand-in.)"""

import ctypes

import pytest
import torch

import means_nearest_centroid_gb300 as km
import workloads
from means_nearest_centroid_gb300 import _build

pytestmark = pytest.mark.gpu

PLANS = [dict(), dict(ksplit=3), dict(ksplit=-2), dict(rows_per_cta=128, centroids_per_tile=128),
         dict(rows_per_cta=256, centroids_per_tile=128, consumer_warps=16),
         dict(rows_per_cta=128, centroids_per_tile=256, consumer_warps=8),
         dict(rows_per_cta=256, centroids_per_tile=256), dict(rows_per_cta=256,
                                                                centroids_per_tile=256, ksplit=2)]
SHAPES = [(1, 1, 16), (300, 700, 64), (5000, 3000, 128), (20000, 700, 96), (3000, 5000, 192),
          (40000, 1000, 256), (777, 129, 48)]


@pytest.fixture(scope="module")
def libs():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    _build.build()
    normal = km.library()
    debug = km._declare(ctypes.CDLL(_build.build(debug=True)))
    return normal, debug


def _call(lib, Xd, Cd, cn, plan):
    N, D = Xd.shape
    K = Cd.shape[0]
    idx = torch.full((N,), -1, dtype=torch.int32, device=Xd.device)
    ms = torch.full((N,), 7.0, dtype=torch.float32, device=Xd.device)
    rc = lib.kmassign_ex(km._ptr(Xd), km._ptr(Cd), km._ptr(cn), N, K, D, km._ptr(idx),
                         km._ptr(ms), plan.get("ksplit", 0), plan.get("rows_per_cta", 0),
                         plan.get("centroids_per_tile", 0), plan.get("consumer_warps", 0),
                         km._stream_ptr(None))
    return rc, idx, ms


@pytest.mark.parametrize("N,K,D", SHAPES)
def test_debug_build_clean_and_identical(libs, N, K, D):
    normal, debug = libs
    dev = torch.device("cuda:0")
    X, C = workloads.blobs(N, K, D, seed=N + K + D)
    Xd, Cd = X.to(dev), C.to(dev)
    for given in (False, True):
        cn = km.kmassign_norms(Cd) if given else None
        for plan in PLANS:
            rc_n, idx_n, ms_n = _call(normal, Xd, Cd, cn, plan)
            if rc_n == km.STATUS["KMASSIGN_ERR_ARG"]:
                continue   # a shape no kernel has for this D
            rc_d, idx_d, ms_d = _call(debug, Xd, Cd, cn, plan)
            assert rc_n == 0 and rc_d == 0, (plan, rc_n, rc_d)
            assert normal.kmassign_check(km._stream_ptr(None)) == 0
            assert debug.kmassign_check(km._stream_ptr(None)) == 0, (N, K, D, plan)
            assert torch.equal(idx_n, idx_d), plan
            assert torch.equal(ms_n.view(torch.int32), ms_d.view(torch.int32)), plan


def test_debug_build_topk_and_noalloc_clean(libs):
    normal, debug = libs
    dev = torch.device("cuda:0")
    X, C = workloads.blobs(3000, 900, 128, seed=9)
    Xd, Cd = X.to(dev), C.to(dev)
    idx = torch.empty(3000 * 8, dtype=torch.int32, device=dev)
    sc = torch.empty(3000 * 8, dtype=torch.float32, device=dev)
    assert debug.kmassign_topk(km._ptr(Xd), km._ptr(Cd), None, 3000, 900, 128, 8, km._ptr(idx),
                               km._ptr(sc), 0, km._stream_ptr(None)) == 0
    i1 = torch.empty(3000, dtype=torch.int32, device=dev)
    assert debug.kmassign_noalloc(km._ptr(Xd), km._ptr(Cd), None, 3000, 900, 128, km._ptr(i1),
                                  None, km._stream_ptr(None)) == 0
    assert debug.kmassign_check(km._stream_ptr(None)) == 0
    assert torch.equal(i1, idx.view(3000, 8)[:, 0])
