"""The multi-rank host logic on CPU: two gloo ranks, no GPU."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from deformable_convolution_03_b300.inputs import WORKLOADS, make_inputs
from deformable_convolution_03_b300.replicas import aggregate_gbs, max_over_ranks, rank_seed


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # rank r reports timings r+1, 10-r: the maximum over ranks wins
        got = max_over_ranks([rank + 1.0, 10.0 - rank], dist)
        w = WORKLOADS["v3_tiny_f32"]
        x = make_inputs(w, seed=rank_seed(w.seed, rank))["input"]
        gathered = [torch.zeros_like(x) for _ in range(world)]
        dist.all_gather(gathered, x)
        distinct = not torch.equal(gathered[0], gathered[1])
        out.put((rank, got, distinct))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_reduce_timings_and_shard_inputs():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, got, distinct in res:
        assert got == [2.0, 10.0], (rank, got)   # max over ranks of each entry
        assert distinct                           # each rank has its own batch


def test_single_process_helpers():
    assert max_over_ranks([3.0, 4.0]) == [3.0, 4.0]
    assert rank_seed(5, 0) == 5 and rank_seed(5, 1) != rank_seed(5, 0)
    assert aggregate_gbs(10**9, 4, 1000.0) == pytest.approx(4.0)
