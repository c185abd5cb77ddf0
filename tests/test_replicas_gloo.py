"""The N > 1 bench path on CPU: two gloo ranks on 127.0.0.1 (no GPU).

The rollout layer runs as independent replicas (no data-path collective); the only cross-rank
steps are the bench's timing reductions: the job's time is the slowest replica's, and the job's
throughput counts every replica's bytes. The CPU reference arm runs on rank 0 only.
"""
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        local_ms = 10.0 + 5.0 * rank  # rank 1 is the slower replica
        ms = bench.max_over_ranks(local_ms, torch.device("cpu"), world, dist)
        value = bench.job_throughput(1e9, world, ms)
        with open(os.path.join(out_dir, f"rank{rank}.txt"), "w") as f:
            f.write(f"{ms!r} {value!r} {bench.reference_runs_here(rank, world)}\n")
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_slowest_time(tmp_path):
    world = 2
    mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True,
                       start_method="spawn")
    got = [open(tmp_path / f"rank{r}.txt").read().split() for r in range(world)]
    for r, (ms, value, ref) in enumerate(got):
        assert float(ms) == 15.0                        # the slowest replica's time, on every rank
        assert float(value) == pytest.approx(2 * 1e9 / 0.015 / 1e9)  # both replicas' bytes
        assert ref == ("True" if r == 0 else "False")   # the reference arm: rank 0 only


def test_single_rank_needs_no_collective():
    assert bench.max_over_ranks(12.5, torch.device("cpu"), 1, None) == 12.5
    assert bench.job_throughput(2e9, 1, 4.0) == pytest.approx(500.0)
    assert bench.reference_runs_here(0, 1) and bench.reference_runs_here(3, 1)
