"""Host-side arithmetic of the binding, without a GPU."""

import pytest

from means_nearest_centroid_gb300 import _slices


@pytest.mark.parametrize("N", [0, 1, 3, 7, 1001, 262144])
@pytest.mark.parametrize("chunks", [1, 2, 4, 8])
@pytest.mark.parametrize("first", [None, 1, 5, 100000])
def test_slices_cover_rows_in_order(N, chunks, first):
    b = _slices(N, chunks, first)
    assert b[0] == 0 and b[-1] == N
    assert all(x < y for x, y in zip(b, b[1:])) or N == 0
    assert len(b) - 1 <= max(1, chunks)
    if N and chunks > 1 and first is not None:
        assert b[1] == min(first, N)


def test_even_slices_by_default():
    assert _slices(262144, 8, None) == [32768 * i for i in range(9)]
    assert _slices(1001, 4, None) == [0, 251, 501, 751, 1001]
