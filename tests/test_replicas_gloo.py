"""The multi-GPU path of bench.py is replicas: one process per GPU, each on
its own seeded problem, the step time the slowest rank's and the throughput
the units all ranks processed.  Checked here with two `gloo` ranks on CPU."""
import os
import socket

import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
from content_adaptive_block_02_b300 import synth


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        cpu = torch.device("cpu")
        ms = bench.max_over_ranks(10.0 + 5.0 * rank, cpu)     # rank 1 is slower
        flop = bench.sum_over_ranks(1e12 * (rank + 1), cpu)
        dist.barrier()
        out[rank] = (ms, flop)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time_and_the_total_work():
    world = 2
    out = mp.get_context("spawn").Manager().dict()
    mp.spawn(_rank_main, args=(world, _free_port(), out), nprocs=world, join=True)
    for r in range(world):
        assert out[r] == (15.0, 3e12)


def test_single_process_is_unchanged():
    cpu = torch.device("cpu")
    assert bench.max_over_ranks(7.5, cpu) == 7.5 and bench.sum_over_ranks(3.0, cpu) == 3.0


def test_replicas_get_independent_seeded_problems():
    w = synth.WORKLOADS["tiny"]
    a, b = bench.replica_workload(w, 0), bench.replica_workload(w, 1)
    assert a.seed_base != b.seed_base and a.with_(seed_base=0) == b.with_(seed_base=0)
    xa, xb = synth.generate(a, "cpu"), synth.generate(b, "cpu")
    assert not torch.equal(xa["Q"], xb["Q"])
