"""The planner on described devices, without a GPU (kmassign_plan_for).

Every plan must be one the kernels can run: a compiled tile shape, a grid
that fits the device (CTA pairs: an even grid within the resident pair
count), a ring of 2..16 stages, and a split that covers every row tile
exactly once."""

import itertools

import pytest

import means_nearest_centroid_gb300 as km
from means_nearest_centroid_gb300 import _build

GB300 = dict(sms=152, smem_per_block=232448, pair_clusters=76)
DEVICES = [GB300, dict(sms=148, smem_per_block=232448, pair_clusters=74),
           dict(sms=8, smem_per_block=232448, pair_clusters=4),
           dict(sms=152, smem_per_block=232448, pair_clusters=0),
           dict(sms=1, smem_per_block=232448, pair_clusters=0)]
SHAPES = [(1, 1, 16), (1, 1, 256), (3, 5, 48), (4096, 128, 64), (65536, 4096, 128),
          (262144, 16384, 256), (1048576, 4096, 128), (65536, 16384, 64), (20000, 700, 64),
          (330000, 524288, 128), (2**31 - 1, 1, 16), (1, 2**31 - 1, 256),
          (2**31 - 1, 2**31 - 1, 256), (777, 300, 192), (150000, 65536, 96)]
COMPILED = {(128, 128, 4), (256, 128, 8), (256, 128, 16), (128, 256, 8), (128, 256, 16),
            (256, 256, 8), (256, 256, 16)}


@pytest.fixture(scope="module", autouse=True)
def lib():
    _build.build()
    return km.library()


def _valid(p, N, K, D, dev):
    rows, nt, cw = p["rows_per_cta"], p["centroids_per_tile"], p["consumer_warps"]
    assert (rows, nt, cw) in COMPILED, p
    pair = (rows, nt) == (256, 256)
    assert 1 <= p["grid"] <= dev["sms"], p
    if pair:
        assert p["grid"] % 2 == 0 and p["grid"] // 2 <= min(dev["pair_clusters"], dev["sms"] // 2)
    assert 2 <= p["stages"] <= 16 and p["xbufs"] in (1, 2), p
    if pair and D <= 128:
        # a folding pair's ring holds whole tiles: a multiple of the tile's
        # k-blocks (one barrier pair each), at least two tiles
        kb = -(-D // 64)
        assert p["stages"] % kb == 0 and p["stages"] >= 2 * kb, p
    rowtiles = -(-max(N, 1) // rows)
    assert p["whole_row_tiles"] + p["split_row_tiles"] == rowtiles, p
    assert p["ksplit"] >= 1
    assert (p["ksplit"] > 1) == (p["split_row_tiles"] > 0), p
    assert p["ksplit"] <= -(-K // nt), p   # no empty centroid range


@pytest.mark.parametrize("dev", DEVICES, ids=lambda d: f"{d['sms']}sm-{d['pair_clusters']}p")
@pytest.mark.parametrize("N,K,D", SHAPES)
def test_automatic_plans_are_runnable(dev, N, K, D):
    _valid(km.kmassign_plan_for(N, K, D, **dev), N, K, D, dev)


@pytest.mark.parametrize("N,K,D", [(5000, 3000, 64), (262144, 16384, 256), (1, 1, 128)])
def test_every_forced_plan_is_runnable_or_refused(N, K, D):
    dev = GB300
    for ks, rows, nt, cw in itertools.product([0, 1, 2, 7, -2, -3], [0, 128, 256], [0, 128, 256],
                                              [0, 4, 8, 16]):
        try:
            p = km.kmassign_plan_for(N, K, D, ksplit=ks, rows_per_cta=rows, centroids_per_tile=nt,
                                     consumer_warps=cw, **dev)
        except km.KmassignError as e:
            assert e.code == km.STATUS["KMASSIGN_ERR_ARG"]
            continue
        _valid(p, N, K, D, dev)
        assert rows in (0, p["rows_per_cta"]) and nt in (0, p["centroids_per_tile"])
        assert cw in (0, p["consumer_warps"])
        if ks > 1:
            # ranges of whole tiles: ks ranges of ceil(tiles / ks) tiles each,
            # fewer when the last would be empty
            tiles = -(-K // p["centroids_per_tile"])
            chunk = -(-tiles // ks)
            assert p["ksplit"] == -(-tiles // chunk) or p["split_row_tiles"] == 0, p


def test_pairs_need_resident_pairs():
    for N, K, D in SHAPES[:10]:
        p = km.kmassign_plan_for(N, K, D, sms=152, smem_per_block=232448, pair_clusters=0)
        assert (p["rows_per_cta"], p["centroids_per_tile"]) != (256, 256)


def test_argument_errors():
    S = km.STATUS
    with pytest.raises(km.KmassignError) as e:
        km.kmassign_plan_for(10, 10, 64, sms=0)
    assert e.value.code == S["KMASSIGN_ERR_ARG"]
    with pytest.raises(km.KmassignError) as e:
        km.kmassign_plan_for(10, 10, 40)
    assert e.value.code == S["KMASSIGN_ERR_UNSUPPORTED_D"]
    with pytest.raises(km.KmassignError) as e:
        km.kmassign_plan_for(10, 0, 64)
    assert e.value.code == S["KMASSIGN_ERR_SHAPE"]
    with pytest.raises(km.KmassignError) as e:
        km.kmassign_plan_for(10, 10, 64, ksplit=-1)
    assert e.value.code == S["KMASSIGN_ERR_ARG"]
    # too little shared memory for any shape
    with pytest.raises(km.KmassignError) as e:
        km.kmassign_plan_for(10, 10, 64, smem_per_block=1024)
    assert e.value.code == S["KMASSIGN_ERR_ARG"]


def _shape(p):
    return (p["ksplit"], p["rows_per_cta"], p["centroids_per_tile"], p["consumer_warps"],
            p["whole_row_tiles"])


@pytest.mark.parametrize("N,K,D,plan", [
    # the five workloads: the reported figures were measured on these plans
    (4096, 128, 64, (1, 128, 128, 4, 32)),               # tiny_blobs
    (65536, 4096, 128, (2, 256, 256, 8, 228)),           # sampled_centroids: pair, tail split 2
    (262144, 16384, 256, (2, 256, 256, 8, 988)),         # iid_normal (the bench)
    (1048576, 4096, 128, (1, 256, 256, 8, 4096)),        # lognormal_clusters: pair, whole
    (65536, 16384, 64, (2, 256, 256, 8, 228)),           # adversarial_ties: pair, tail split 2
])
def test_workload_plans_on_a_gb300(N, K, D, plan):
    assert _shape(km.kmassign_plan_for(N, K, D)) == plan


@pytest.mark.parametrize("N,K,D,plan", [
    # a two-range split re-weighed within the chosen shape: whole pair row
    # tiles become a tail split in 2 (measured faster) ...
    (262144, 2048, 128, (2, 256, 256, 8, 988)),
    (65536, 1024, 256, (2, 256, 256, 8, 228)),
    # ... but it never tips the shape: this one stays on whole CTA-pair row
    # tiles, where single blocks with a tail split measured 18% slower
    (131072, 1024, 128, (1, 256, 256, 8, 512)),
])
def test_two_range_split_keeps_the_shape(N, K, D, plan):
    assert _shape(km.kmassign_plan_for(N, K, D)) == plan
