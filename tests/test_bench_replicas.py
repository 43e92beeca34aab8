"""The benchmark's multi-GPU host logic (replicas: every rank decodes its own
request, no data-path collective) on CPU with two gloo ranks: the job time is
the slowest rank's, the job throughput counts every rank's tokens, and the
reference arm runs on rank 0 only."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        own = 1.5 + rank                      # rank 1 is the slow one
        t_max = bench.max_over_ranks(own, dist, device="cpu")
        out[rank] = (t_max, bench.job_tokens_per_s(world, 256, t_max))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_slowest_time_and_the_job_throughput():
    world = 2
    port = _free_port()
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.start_processes(_rank_main, args=(world, port, out), nprocs=world, join=True, start_method="spawn")
        res = dict(out)
    assert res[0] == res[1]
    t_max, tok_s = res[0]
    assert t_max == 2.5
    assert tok_s == pytest.approx(2 * 256 / 2.5)


def test_single_process_needs_no_group():
    assert bench.max_over_ranks(0.75) == 0.75
    assert bench.job_tokens_per_s(1, 100, 0.5) == 200.0


def test_reference_arm_runs_on_rank_zero_only(monkeypatch):
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("LOCAL_RANK", "1")

    class Args:
        workload = "tiny"
        steps = 1
        warmup = 3
        gpus = 2

    assert bench.run_reference(Args()) is None     # returns before any work
