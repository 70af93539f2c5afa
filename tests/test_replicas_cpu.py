"""Host logic of the multi-GPU path (replicas, one process per GPU), on CPU with gloo.

The layer shards by tokens with no exchange inside the step; bench.py times each replica's
steps, takes the slowest rank's time (all-reduce MAX) and reports all ranks' tokens over it.
These tests run that aggregation on two gloo ranks and check the reference arm's rank
handling; no GPU is needed."""
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, times, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        got = bench.slowest_rank(times[rank], world, device="cpu")
        out[rank] = got
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_slowest_rank_is_taken_on_every_rank():
    world = 2
    times = [[10.0, 3.0, 7.5], [9.0, 4.0, 8.25]]  # per rank: step, GEMM and graph timings
    with mp.get_context("spawn").Manager() as m:
        out = m.dict()
        mp.start_processes(_rank_main, args=(world, _free_port(), times, out), nprocs=world,
                           join=True, start_method="spawn")
        got = dict(out)
    want = [max(a, b) for a, b in zip(*times)]
    assert got[0] == want and got[1] == want


def test_job_throughput_is_weak_scaling_over_the_slowest_rank():
    # two replicas of 65536 tokens, slowest rank 50 ms per step -> 2.62 M tokens/s
    assert bench.job_tokens_per_s(2, 65536, 50.0) == pytest.approx(2 * 65536 / 0.05)
    assert bench.job_tokens_per_s(1, 512, 1.0) == pytest.approx(512_000)


def test_reference_arm_runs_on_rank_zero_only():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--config", "C0", "--steps", "1", "--warmup", "1"],
                       capture_output=True, text=True, env=env, timeout=300)
    assert r.returncode == 0
    assert r.stdout.strip() == ""
