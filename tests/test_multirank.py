"""The N > 1 path of bench.py on CPU: two gloo ranks, one replica each (data
parallel over requests, no collective in the data path). Checks the timing
reduction (slowest rank), the whole-job throughput and per-rank request seeds."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    elapsed = 1.0 + rank  # rank 1 is slower
    m = bench.reduce_max(elapsed, world)
    seeds = [None] * world
    dist.all_gather_object(seeds, bench.rank_seed(0, rank))
    out[rank] = (m, bench.weak_scaling_tokens_per_s(world, 8, 10, m), tuple(seeds))
    dist.destroy_process_group()


def test_two_rank_replicas_reduce_to_slowest_rank():
    world = 2
    port = _free_port()
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_worker, args=(world, port, out), nprocs=world, start_method="spawn", join=True)
    for r in range(world):
        m, v, seeds = out[r]
        assert m == 2.0                      # max over ranks
        assert v == world * 8 * 10 / 2.0     # tokens of every rank / slowest time
        assert len(set(seeds)) == world      # disjoint request streams


def test_single_rank_is_identity():
    assert bench.reduce_max(3.5, 1) == 3.5
    assert bench.weak_scaling_tokens_per_s(1, 8, 10, 2.0) == 40.0
