"""Host-side logic of bench.py's multi-rank (replica) path, run as world_size-2
gloo process groups on the CPU: the timed total is the slowest rank's, and the
job throughput counts every replica's tokens over that time."""
from __future__ import annotations

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


def _rank_main(rank: int, world: int, port: int, times, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        assert bench.dist_env() == (rank, world, rank)
        dist.barrier()
        t = bench.max_over_ranks(times[rank], dist, torch.device("cpu"))
        out[rank] = t
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_gloo():
    world = 2
    times = [12.5, 40.25]
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        out = m.dict()
        mp.start_processes(_rank_main, args=(world, _free_port(), times, out), nprocs=world,
                           join=True, start_method="spawn")
        got = dict(out)
    assert got == {0: 40.25, 1: 40.25}


def test_job_tokens_per_s():
    # 2 replicas x 64 tokens x 100 steps in 25 ms (the slowest rank's total)
    assert bench.job_tokens_per_s(2, 64, 100, 25.0) == pytest.approx(2 * 64 * 100 / 0.025)
    assert bench.job_tokens_per_s(1, 4096, 10, 5.0) == pytest.approx(4096 * 10 / 0.005)


def test_reference_arm_runs_on_rank0_only(monkeypatch, capsys):
    """Under torchrun the oracle arm runs on rank 0 alone; other ranks exit 0 without work."""
    import argparse
    from mixture_experts_ffn_03_gb300 import workloads as wl
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("LOCAL_RANK", "1")
    args = argparse.Namespace(steps=1, warmup=1, gpus=2, config="tiny")
    assert bench.run_reference(args, wl.CONFIGS["tiny"]) == 0
    assert capsys.readouterr().out == ""
