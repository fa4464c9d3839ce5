"""The multi-GPU form of the benchmark runs one replica of the layer per rank
and reports the whole-job throughput over the slowest rank.  This checks that
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


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ws, r, _ = bench.dist_env()
        assert (ws, r) == (world, rank)
        rank_ms = [100.0, 250.0][rank]            # rank 1 is the slowest
        tps, slowest = bench.job_throughput(dist, ws, 8192, 10, rank_ms, torch.device("cpu"))
        bench.barrier(dist)
        out[rank] = (tps, slowest)
    finally:
        dist.destroy_process_group()


def test_two_rank_throughput_uses_slowest_rank():
    port = _free_port()
    with mp.get_context("spawn").Manager() as m:
        out = m.dict()
        mp.spawn(_rank, args=(2, port, out), nprocs=2, join=True)
        res = dict(out)
    for r in (0, 1):
        tps, slowest = res[r]
        assert slowest == pytest.approx(250.0)
        assert tps == pytest.approx(2 * 8192 * 10 / 0.25)


def test_single_process_throughput():
    import bench
    tps, slowest = bench.job_throughput(None, 1, 16, 20, 40.0, torch.device("cpu"))
    assert slowest == 40.0 and tps == pytest.approx(16 * 20 / 0.04)
