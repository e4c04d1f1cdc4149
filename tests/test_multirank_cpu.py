"""The multi-GPU host logic with two ranks on gloo (CPU only).

Points shard across GPUs with no exchange on the data path: each rank takes
the contiguous share given by shard_rows, assigns it (here with the oracle,
which stands in for the GPU call on a CPU-only machine) and the answers
concatenate in rank order.  The benchmark's timing reduction (max over ranks)
and its per-rank input sets are checked the same way.
"""

import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import means_nearest_centroid_gb300 as km


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out_dir):
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench
    import oracle
    import workloads
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        N, K, D = 1001, 37, 24
        X, C = workloads.blobs(N, K, D, seed=9)
        b, e = km.shard_rows(N, rank, world)
        idx, mins = oracle.assign(X[b:e], C)
        parts = [None] * world
        dist.all_gather_object(parts, (b, e, idx.tolist(), mins.tolist()))
        t = bench.max_over_ranks(float(rank + 1) * 1.5, dist, torch.device("cpu"))
        variants = [None] * world
        dist.all_gather_object(variants, bench.rank_variants(rank))
        if rank == 0:
            np.save(os.path.join(out_dir, "result.npy"),
                    np.array([parts, t, variants], dtype=object), allow_pickle=True)
    finally:
        dist.destroy_process_group()


def test_two_rank_shards_and_timing(tmp_path):
    world = 2
    port = _free_port()
    mp.start_processes(_worker, args=(world, port, str(tmp_path)), nprocs=world,
                       start_method="spawn", join=True)
    parts, t, variants = np.load(tmp_path / "result.npy", allow_pickle=True)
    import oracle
    import workloads
    X, C = workloads.blobs(1001, 37, 24, seed=9)
    full_idx, full_min = oracle.assign(X, C)
    got_idx = []
    got_min = []
    prev_end = 0
    for b, e, idx, mins in parts:
        assert b == prev_end
        prev_end = e
        got_idx += idx
        got_min += mins
    assert prev_end == 1001
    assert np.array_equal(np.array(got_idx), full_idx)
    assert np.array_equal(np.array(got_min), full_min)
    assert t == 3.0                      # max over ranks of 1.5 * (rank + 1)
    assert not set(variants[0]) & set(variants[1])


@pytest.mark.parametrize("N,world", [(0, 3), (5, 8), (1000, 7), (2**20 + 3, 4)])
def test_shard_rows_partition(N, world):
    bounds = [km.shard_rows(N, r, world) for r in range(world)]
    assert bounds[0][0] == 0 and bounds[-1][1] == N
    sizes = [e - b for b, e in bounds]
    assert max(sizes) - min(sizes) <= 1
    for (b0, e0), (b1, e1) in zip(bounds, bounds[1:]):
        assert e0 == b1


def test_shard_rows_rejects_bad_rank():
    with pytest.raises(ValueError):
        km.shard_rows(10, 2, 2)
