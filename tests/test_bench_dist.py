"""The benchmark's multi-rank bookkeeping on CPU with two gloo ranks: the step
time is the max over ranks and the value is the whole-job throughput."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    ms_local = [2.0, 5.0][rank]
    ms = bench.reduce_max(ms_local, dist, torch.device("cpu"))
    out[rank] = (ms, bench.job_gbs(1_000_000, ms, world))
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_max_and_job_value():
    world, port = 2, _free_port()
    out = mp.Manager().dict()
    mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
    for r in range(world):
        ms, gbs = out[r]
        assert ms == 5.0
        assert gbs == pytest.approx(2 * 1_000_000 / 5e-3 / 1e9)


def test_single_rank_identity():
    assert bench.reduce_max(3.0, None, None) == 3.0
    assert bench.job_gbs(35_651_584, 7.0e-3, 1) == pytest.approx(35_651_584 / 7e-6 / 1e9)
