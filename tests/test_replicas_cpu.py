"""Host logic of the benchmark on CPU: the multi-GPU path (replicas, one process per GPU)
with gloo, and the reference arm.

The layer shards by tokens with no exchange inside the step; bench.py times each replica's
steps, takes the slowest rank's time (all-reduce MAX) and reports all ranks' tokens over it.
These tests run that aggregation on two gloo ranks and check the reference arm's rank
handling; no GPU is needed."""
import json
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
from pretraining_sigmoid_softmax_gb300.configs import CONFIGS, MoEConfig  # noqa: E402
from pretraining_sigmoid_softmax_gb300.inputs import make_inputs  # noqa: E402


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


def test_reference_arm_prints_the_contract_line_on_rank_zero():
    env = dict(os.environ, RANK="0", WORLD_SIZE="1", LOCAL_RANK="0")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--config", "C0", "--steps", "2", "--warmup", "1"],
                       capture_output=True, text=True, env=env, timeout=300)
    assert r.returncode == 0, r.stderr
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["metric"] == bench.METRIC
    assert line["unit"] == "tokens/s" and line["higher_is_better"] is True
    assert line["steps"] == 2 and line["warmup"] == 1 and line["value"] > 0
    assert line["config"] == bench.workload_desc(CONFIGS["C0"])
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == line["value"]
    assert "forward" in cb["sample"]
    assert line["e2e"] == {"value": line["value"], "unit": "tokens/s", "h2d_bytes_per_step": 0,
                           "d2h_bytes_per_step": 0}


@pytest.mark.parametrize("kw", [dict(precision="fp8", f_shared=64),
                                dict(mode="softmax", z_coef=1e-3, aux_switch=1e-3, aux_seq=1e-3,
                                     seq_len=4096, bias_update=False)])
def test_cpu_baseline_times_the_workloads_own_layer(kw):
    """The timed oracle runs the workload's own precision and losses (FP8 operands, the
    balancing losses with a sample shorter than one sequence taken as one sequence)."""
    base = dict(name="t", T=64, d=128, E=8, k=2, f=128, f_shared=0, mode="sigmoid", seed=1,
                backward=True, bias_update=True)
    cfg = MoEConfig(**{**base, **kw})
    rate, cores, times = bench.cpu_oracle_rate(cfg, make_inputs(cfg), 32)
    assert rate > 0 and cores >= 1 and len(times) == 1
    desc = bench.oracle_pass_desc(cfg)
    assert ("FP8" in desc) == cfg.fp8
    assert ("balancing" in desc) == cfg.has_aux


def test_one_core_oracle_timing_runs_in_a_single_threaded_child():
    rate = bench.cpu_oracle_rate_one_core("C0", 32)
    assert rate > 0


def test_small_workloads_flush_l2_and_say_so():
    for name, cfg in CONFIGS.items():
        small = cfg.T * cfg.d * 2 < 128 * 2**20
        assert bench.needs_l2_flush(cfg) == small, name
        assert bench.workload_desc(cfg)["l2"].startswith("L2 flushed" if small else "inputs larger")


def test_host_cpu_description_reads_x86_and_arm_cpuinfo():
    assert isinstance(bench.host_cpu_desc(), str) and bench.host_cpu_desc()
    x86 = "processor\t: 0\nmodel name\t: Example CPU @ 2.0GHz\nflags\t: sse\n"
    assert bench.cpu_desc_from(x86, "x86_64") == "Example CPU @ 2.0GHz (x86_64)"
    arm = "processor\t: 0\nBogoMIPS\t: 2000.00\nCPU implementer\t: 0x41\nCPU part\t: 0xd4f\n"
    assert bench.cpu_desc_from(arm, "aarch64") == "aarch64, CPU implementer 0x41 part 0xd4f"
    assert bench.cpu_desc_from("", "aarch64") == "aarch64"
