"""The fp64 oracle against facts outside itself (CPU only)."""

import numpy as np
import pytest

import oracle
import pins


@pytest.fixture(scope="module")
def orc():
    return oracle.Oracle()


@pytest.mark.parametrize("check", pins.ALL_CHECKS, ids=lambda f: f.__name__)
def test_pin(orc, check):
    check(orc)


def test_thread_count_does_not_change_answers(orc):
    import workloads
    X, C = workloads.iid(300, 70, 32, seed=5)
    a = orc.assign(X, C, nthreads=1)
    b = orc.assign(X, C, nthreads=4)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_rejects_bad_arguments(orc):
    import workloads
    X, C = workloads.iid(4, 3, 8, seed=1)
    with pytest.raises(IndexError):
        orc.assign(X, C, rows=[4])
    with pytest.raises(ValueError):
        orc.assign(X[:, :4], C)
