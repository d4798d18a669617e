"""Multi-process (N > 1) host logic of the benchmark, on CPU with the gloo backend.

The hot path shards over independent (sequence, value head) streams, so N GPUs run N replicas, each on
its own batch, and only the timing crosses ranks: a barrier and a max-reduction of each rank's time.
These tests run that host logic as two gloo ranks (no GPU, no data-path collective).
"""

import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
from gated_delta_rule_38_gb300.inputs import custom, make_inputs


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, out):
    dist.init_process_group("gloo", init_method="tcp://127.0.0.1:%d" % port, rank=rank, world_size=world)
    try:
        # each rank's own time; the job's time is the slowest one
        local = 1.0 + 2.0 * rank
        job = bench.max_over_ranks(local, dist, torch.device("cpu"))
        # each rank draws its own batch from its own seed
        w = custom(B=1, T=8, Hq=1, Hv=1)
        q = make_inputs(w, seed=bench.rank_seed(rank))["q"].float()
        qs = [torch.zeros_like(q) for _ in range(world)]
        dist.all_gather(qs, q)
        dist.barrier()
        out[rank] = (job, all(not torch.equal(qs[0], qs[i]) for i in range(1, world)))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_time_and_batches():
    world = 2
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_rank_main, args=(world, _free_port(), out), nprocs=world, start_method="spawn", join=True)
    assert sorted(out.keys()) == [0, 1]
    for r in range(world):
        job, distinct = out[r]
        assert job == pytest.approx(3.0)  # max over ranks of (1, 3)
        assert distinct  # the ranks' batches differ


def test_job_throughput_is_whole_job():
    # N ranks each process their own tokens in the slowest rank's time
    assert bench.job_throughput(8192, 4, 2.0) == pytest.approx(8192 * 4 / 2.0)
    assert bench.max_over_ranks(5.0, None, None) == 5.0
    assert bench.rank_seed(0) != bench.rank_seed(1)
