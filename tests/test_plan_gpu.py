"""The planner seen through kmassign_plan / kmassign_plan_ex (needs a GPU: the
plan depends on the device's SM count and shared memory)."""

import pytest
import torch

import means_nearest_centroid_gb300 as km

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from means_nearest_centroid_gb300 import _build
    _build.build()
    km.library()
    return torch.device("cuda:0")


SHAPES = [(4096, 128, 64), (65536, 4096, 128), (262144, 16384, 256), (65536, 8192, 192),
          (1048576, 4096, 256), (1000, 300, 48)]


@pytest.mark.parametrize("N,K,D", SHAPES)
def test_plan_ex_without_forcing_is_the_automatic_plan(dev, N, K, D):
    assert km.kmassign_plan(N, K, D) == km.kmassign_plan(N, K, D, 0, 0, 0, 0)


@pytest.mark.parametrize("N,K,D", SHAPES)
@pytest.mark.parametrize("rows,nt,cw", [(128, 256, 8), (256, 128, 8), (128, 128, 4),
                                        (256, 128, 16), (128, 256, 16)])
def test_forced_shape_is_honoured(dev, N, K, D, rows, nt, cw):
    p = km.kmassign_plan(N, K, D, rows_per_cta=rows, centroids_per_tile=nt, consumer_warps=cw)
    assert (p["rows_per_cta"], p["centroids_per_tile"], p["consumer_warps"]) == (rows, nt, cw)
    assert p["grid"] >= 1 and p["stages"] >= 2 and p["xbufs"] in (1, 2)
    # every row tile is either whole or split
    R = -(-N // rows)
    assert p["whole_row_tiles"] + p["split_row_tiles"] == R


@pytest.mark.parametrize("ks", [1, 2, 3, -2, -4])
def test_forced_split_is_honoured(dev, ks):
    N, K, D = 262144, 16384, 128
    p = km.kmassign_plan(N, K, D, ksplit=ks, rows_per_cta=256, centroids_per_tile=128,
                         consumer_warps=8)
    if ks > 0:
        assert p["ksplit"] == ks
        assert p["split_row_tiles"] == (0 if ks == 1 else 1024)
    else:
        # tail split: only the last, partial wave of row tiles is split
        assert p["ksplit"] in (1, -ks)
        assert p["split_row_tiles"] < 1024


def test_pair_plans_are_chosen_for_large_shapes(dev):
    # above D = 128 the pair; up to D = 128 the pair that folds the norms,
    # where enough tiles per unit amortise its fold operand
    for D in (256, 192, 128, 96, 64):
        p = km.kmassign_plan(262144, 16384, D)
        assert (p["rows_per_cta"], p["centroids_per_tile"]) == (256, 256), D
    # short centroid ranges at D = 64 stay on the single-block fold, longer
    # ones from ~2,048 centroids go to the pair
    for N, K in [(262144, 512), (262144, 1024), (65536, 512)]:
        p = km.kmassign_plan(N, K, 64)
        assert (p["rows_per_cta"], p["centroids_per_tile"]) == (256, 128), (N, K)
    p = km.kmassign_plan(262144, 4096, 64)
    assert (p["rows_per_cta"], p["centroids_per_tile"]) == (256, 256)
    # every shape can be forced at any D
    p = km.kmassign_plan(65536, 4096, 32, rows_per_cta=256, centroids_per_tile=256,
                         consumer_warps=8)
    assert (p["rows_per_cta"], p["centroids_per_tile"]) == (256, 256)


def test_plan_ex_rejects_bad_forcing(dev):
    for kw in [dict(ksplit=-1), dict(rows_per_cta=64), dict(centroids_per_tile=512),
               dict(consumer_warps=12)]:
        with pytest.raises(km.KmassignError):
            km.kmassign_plan(1000, 300, 64, **kw)


def test_plan_for_a_described_gb300_matches_the_device():
    """The host-only planner given this GPU's description plans what the
    device planner plans (GB300: 152 SMs, 232,448 bytes, 76 resident pairs)."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    props = torch.cuda.get_device_properties(0)
    if props.multi_processor_count != 152:
        pytest.skip("not a 152-SM GB300")
    for N, K, D in [(4096, 128, 64), (65536, 4096, 128), (262144, 16384, 256),
                    (1048576, 4096, 128), (65536, 16384, 64), (20000, 700, 64), (777, 300, 192)]:
        assert km.kmassign_plan_for(N, K, D) == km.kmassign_plan(N, K, D), (N, K, D)
