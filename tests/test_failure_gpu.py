"""Failure detection on the GPU without faulting it (needs a GB300).

The kernel's pipeline waits are bounded by the GPU's global timer.  Shrinking
the bound to 100 ns makes the first wait that is not already satisfied run
out: the kernel must record a timeout, drain its copies and MMAs, free its
tensor memory and return.  The host then reads KMASSIGN_ERR_TIMEOUT, and the
same context must still give correct answers once the bound is restored.
"""

import pytest
import torch

import means_nearest_centroid_gb300 as km
import parity
import workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from means_nearest_centroid_gb300 import _build
    _build.build()
    km.library()
    return torch.device("cuda:0")


@pytest.mark.parametrize("plan", [dict(), dict(ksplit=3, rows_per_cta=256, centroids_per_tile=128),
                                  dict(rows_per_cta=128, centroids_per_tile=256, consumer_warps=16),
                                  dict(rows_per_cta=256, centroids_per_tile=256, consumer_warps=8)],
                         ids=str)
def test_short_wait_bound_reports_timeout_and_context_survives(dev, plan):
    X, C = workloads.iid(40000, 3000, 128, seed=21)
    Xd, Cd = X.to(dev), C.to(dev)
    assert km.kmassign_check() == 0
    try:
        km.kmassign_set_wait_timeout(100)
        km.kmassign_ex(Xd, Cd, **plan)
        rc = km.kmassign_check()
    finally:
        km.kmassign_set_wait_timeout(0)
    assert rc == km.STATUS["KMASSIGN_ERR_TIMEOUT"], km.kmassign_strerror(rc)
    # the status word was cleared by the check; the context is intact
    assert km.kmassign_check() == 0
    ms = torch.empty(40000, dtype=torch.float32, device=dev)
    idx = km.kmassign_ex(Xd, Cd, minscore=ms, **plan)
    assert km.kmassign_check() == 0
    rows = list(range(0, 40000, 97)) + list(range(39700, 40000))
    rep = parity.compare(X, C, idx.cpu(), ms.cpu(), rows=sorted(set(rows)))
    assert rep.ok(), rep


@pytest.mark.parametrize("ksplit", [0, 4])
def test_topk_short_wait_bound_reports_timeout(dev, ksplit):
    """The k-nearest kernel shares the bounded pipeline: same behaviour."""
    X, C = workloads.iid(40000, 3000, 128, seed=22)
    Xd, Cd = X.to(dev), C.to(dev)
    assert km.kmassign_check() == 0
    try:
        km.kmassign_set_wait_timeout(100)
        km.kmassign_topk(Xd, Cd, 8, ksplit=ksplit)
        rc = km.kmassign_check()
    finally:
        km.kmassign_set_wait_timeout(0)
    assert rc == km.STATUS["KMASSIGN_ERR_TIMEOUT"], km.kmassign_strerror(rc)
    assert km.kmassign_check() == 0
    idx, sc = km.kmassign_topk(Xd, Cd, 8, ksplit=ksplit)
    assert km.kmassign_check() == 0
    rows = sorted(set(range(0, 40000, 211)) | set(range(39800, 40000)))
    rep = parity.compare_topk(X, C, idx.cpu(), sc.cpu(), 8, rows=rows)
    assert rep.ok(), rep
