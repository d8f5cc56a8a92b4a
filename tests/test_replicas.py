"""The multi-GPU path is replicas only: each rank runs its own batch and the job
rate is all ranks' samples over the slowest rank's time.  These tests run the
host-side logic of that path (bench.py's helpers) on two gloo ranks on the CPU."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
from scale_deformable_attention_05_b300 import inputs as gen


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        step_ms = 2.0 + rank          # rank 1 is the slow one
        ms = bench.max_over_ranks(step_ms, dist)
        out[rank] = (ms, bench.job_rate(1000, world, ms))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_rank_time():
    world = 2
    with mp.get_context("spawn").Manager() as m:
        out = m.dict()
        mp.spawn(_rank_main, args=(world, _free_port(), out), nprocs=world, join=True)
        res = dict(out)
    assert res[0] == res[1] == (3.0, 1000 * world / 3e-3)


def test_each_rank_draws_its_own_batch():
    wl = gen.WORKLOADS["tiny"]
    a = gen.make_inputs(bench.rank_workload(wl, 0))
    b = gen.make_inputs(bench.rank_workload(wl, 1))
    assert a["value"].shape == b["value"].shape
    assert not (a["sampling_locations"] == b["sampling_locations"]).all()
    assert bench.max_over_ranks(4.5) == 4.5
