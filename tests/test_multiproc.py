"""The benchmark's multi-rank timing aggregation on world_size 2 over gloo (CPU only).

Replicas need no data-path collective: each rank runs its own problem, and the
job time is the maximum of the ranks' times while the work is their sum.
"""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench
    w, r, local = bench.dist_env()
    assert (w, r, local) == (world, rank, rank)
    dist = bench.init_dist(world, "gloo")
    bench.barrier(dist)
    elapsed = [0.25, 0.5][rank]
    units = [1e12, 3e12][rank]
    job_s, job_units = bench.aggregate(dist, elapsed, units)
    out[rank] = (job_s, job_units)
    dist.destroy_process_group()


def test_aggregate_takes_max_time_and_sum_of_work():
    world = 2
    port = _free_port()
    with mp.get_context("spawn").Manager() as mgr:  # no fork of a multi-threaded process
        out = mgr.dict()
        mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    assert res[0] == res[1] == (0.5, 4e12)


def test_single_rank_has_no_process_group():
    import bench
    assert bench.init_dist(1, "gloo") is None
    assert bench.aggregate(None, 1.5, 7.0) == (1.5, 7.0)


@pytest.mark.parametrize("name", ["resnet_56x56_c64", "proj_56_c256_1x1s2", "stem_224_c3_7x7s2"])
def test_algorithmic_counts(name):
    import bench
    import workloads
    wl = workloads.get(name)
    p, q = bench.shape_of(wl)
    assert bench.flops_per_step(wl) == 2.0 * wl.n * p * q * wl.k * wl.c * wl.r * wl.s
    nbytes = bench.algorithmic_bytes(wl)
    y_bytes = wl.n * p * q * wl.k * 4
    assert nbytes > y_bytes
    if name == "proj_56_c256_1x1s2":
        # a strided 1x1 touches every other row and column: a quarter of the input
        assert nbytes == wl.n * 28 * 28 * 256 * 2 + 512 * 256 * 2 + y_bytes
