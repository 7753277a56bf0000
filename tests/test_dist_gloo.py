"""The multi-rank path of bench.py on CPU: two gloo ranks, one process each.

The block shards by tokens with no data-path collective; the benchmark's only cross-rank steps
are the barrier and the max over ranks of the step time, and the whole-job rate counts every
rank's units against that slowest time.
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
    import torch
    import torch.distributed as dist

    import bench

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = [3.0, 5.0][rank]
        mx = bench.reduce_max(ms, world, torch.device("cpu"))
        dist.barrier()
        rate = bench.whole_job_rate(100.0, world, mx)
        out[rank] = (mx, rate)
    finally:
        dist.destroy_process_group()


def test_two_rank_max_and_whole_job_rate():
    world = 2
    port = _free_port()
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    assert res[0] == res[1] == (5.0, 2 * 100.0 / 5e-3)


def test_single_rank_needs_no_process_group():
    import bench
    assert bench.reduce_max(2.5, 1, None) == 2.5
    assert bench.whole_job_rate(10.0, 1, 2.0) == 5000.0
