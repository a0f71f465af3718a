"""The multi-GPU path is replicas only: each rank runs the same step on its
own device, with no collective on the data path; the job's time is the
slowest rank's and its throughput counts every rank's work.  This checks that
host logic with two gloo ranks on the CPU."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    local_ms = 10.0 * (rank + 1)             # rank 1 is the slow one
    ms, per_s = bench.aggregate_replicas(local_ms, 1e9, dist, torch.device("cpu"))
    out[rank] = (ms, per_s)
    dist.barrier()
    dist.destroy_process_group()


def test_replicas_take_the_slowest_rank_and_count_all_work():
    world, port = 2, _free_port()
    with mp.get_context("spawn").Manager() as m:  # no fork of a multi-threaded process
        out = m.dict()
        mp.spawn(_rank_main, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    for rank in range(world):
        ms, per_s = res[rank]
        assert ms == pytest.approx(20.0)
        assert per_s == pytest.approx(2 * 1e9 / 0.020)


def test_single_process_needs_no_process_group():
    import bench
    ms, per_s = bench.aggregate_replicas(5.0, 1e6)
    assert ms == 5.0 and per_s == pytest.approx(1e6 / 0.005)
