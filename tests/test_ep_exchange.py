"""The expert-parallel form of the layer (two ranks, each holding half of the
experts) and its one exchange step, on the CPU with two gloo ranks and the
float64 oracle: each rank computes the layer for its own experts, slots
routed to the other rank masked (expert id -1, the form the kernels take),
and a sum over ranks of those partial outputs (the all-reduce the pages' MoE
tail performs) gives the whole layer.  This pins the decomposition the
multi-GPU design relies on; the single-GPU part of it (a local expert slice
with masked slots) is the GPU test of the expert-parallel slice."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import workloads as W
from oracle import moe as O

WL = W.WORKLOADS["tiny"].with_(name="ep_exchange", T=24, H=128, I=128, E=8, k=3)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _local_routing(ids, rank, world, E):
    e_loc = E // world
    off = rank * e_loc
    local = (ids >= off) & (ids < off + e_loc)
    return np.where(local, ids - off, -1).astype(np.int32), off, e_loc


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        s = W.gen_small_inputs(WL)
        ids, wts, _ = O.route(s["logits"], s["bias"], WL.k)
        ids_loc, off, e_loc = _local_routing(ids, rank, world, WL.E)
        # this rank's experts are global experts off .. off + e_loc - 1
        local_w = W.gen_expert_weights_np(WL, list(range(off, off + e_loc)))
        part = O.forward(WL.with_(E=e_loc), s["x"], None, None, local_w, experts_host=list(range(e_loc)),
                         ids=ids_loc, topk_w=wts)["out"]
        t = torch.from_numpy(np.ascontiguousarray(part))
        dist.all_reduce(t, op=dist.ReduceOp.SUM)
        out[rank] = (t.numpy(), int((ids_loc >= 0).sum()))
    finally:
        dist.destroy_process_group()


def test_two_rank_expert_parallel_sum_equals_the_layer():
    port = _free_port()
    with mp.get_context("spawn").Manager() as m:
        out = m.dict()
        mp.spawn(_rank, args=(2, port, out), nprocs=2, join=True)
        res = dict(out)
    s = W.gen_small_inputs(WL)
    full = O.forward(WL, s["x"], s["logits"], s["bias"], W.gen_expert_weights_np(WL, range(WL.E)))["out"]
    # every routed slot is local to exactly one rank
    assert res[0][1] + res[1][1] == WL.T * WL.k
    for r in (0, 1):
        got = res[r][0]
        assert np.array_equal(res[0][0], got)  # both ranks hold the same reduced output
        assert np.allclose(got, full, rtol=1e-12, atol=1e-9 * np.abs(full).max())
