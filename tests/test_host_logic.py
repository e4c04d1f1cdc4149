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


@pytest.mark.parametrize("N", [1, 1001, 19456, 262144, 1048576])
@pytest.mark.parametrize("chunks", [1, 2, 8])
@pytest.mark.parametrize("align", [19456, 38912])
def test_wave_aligned_slices(N, chunks, align):
    b = _slices(N, chunks, None, align)
    assert b[0] == 0 and b[-1] == N
    assert all(x < y for x, y in zip(b, b[1:]))
    sizes = [y - x for x, y in zip(b, b[1:])]
    # every slice but the last is a whole number of waves
    assert all(s % align == 0 for s in sizes[:-1])
    if chunks == 1:
        assert sizes == [N]


def test_wave_aligned_slices_of_the_bench_workload():
    # 262,144 rows, waves of 76 CTA pairs x 256 rows: six slices of two waves,
    # then the remaining 1.47 waves, instead of eight slices of 1.68 waves
    assert _slices(262144, 8, None, 19456) == [0] + [38912 * i for i in range(1, 7)] + [262144]
