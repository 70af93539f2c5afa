"""Benchmark of the MoE layer step (forward + backward + bias update) on GB300.

Default workload: the large fine-grained layer (T=65536 = 16 x 4096 tokens, d_model 4096,
64 experts, top-8, expert d_ff 1536, one shared expert of d_ff 3072, sigmoid router with
bias and bias update), synthetic inputs. Prints one JSON line (rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config C4] [--impl ours|reference]

Under torchrun every rank runs its own replica on its own batch (no collective on the data
path: the layer step does not exchange data); `value` is the tokens of all ranks divided
by the slowest rank's time.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MoE layer fwd+bwd tokens/s; grouped-GEMM TFLOP/s as % of GB300 BF16 peak"
# DRAM bytes (read + write) of one step's grouped-GEMM launches, summed from a stored ncu
# capture of the current kernels at that workload (not measured by this run; the line says
# so); workloads without a capture report null.
MEASURED_GEMM_TRAFFIC = {"C4": 144.04e9}
# Datasheet dense peaks of a GB300 (not from the source pages), reported beside the measured
# ones: bf16 2250 TFLOP/s (fp8 twice that), HBM3e about 8 TB/s.
NOMINAL_BF16_TFLOPS = 2250.0
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=20)
    p.add_argument("--warmup", type=int, default=3)
    p.add_argument("--config", default="C4")
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--cpu-sample-tokens", type=int, default=128)
    p.add_argument("--no-graph", action="store_true",
                   help="time eager per-call launches instead of one CUDA graph per step")
    return p.parse_args()


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as fh:
            pk = json.load(fh)
        return pk, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


L2_FLUSH_BYTES = 256 << 20  # about twice the 129 MB L2


def needs_l2_flush(cfg) -> bool:
    """Workloads whose input x is smaller than L2 flush it before every timed step."""
    return cfg.T * cfg.d * 2 < L2_FLUSH_BYTES // 2


def workload_desc(cfg):
    if needs_l2_flush(cfg):
        l2 = ("L2 flushed before every timed step (a %d MiB write outside the timed interval; "
              "x is %.1f MiB)" % (L2_FLUSH_BYTES >> 20, cfg.T * cfg.d * 2 / 2**20))
    else:
        l2 = ("inputs larger than L2 (x alone is %.0f MiB; permuted rows %.1f GiB)"
              % (cfg.T * cfg.d * 2 / 2**20, cfg.N * cfg.d * 2 / 2**30))
    return {"workload": cfg.name, "T": cfg.T, "d_model": cfg.d, "experts": cfg.E, "top_k": cfg.k,
            "d_ff": cfg.f, "shared_d_ff": cfg.f_shared, "router": cfg.mode,
            "bias_update": cfg.bias_update, "pass": "fwd+bwd" if cfg.backward else "fwd",
            "l2": l2, "parallelism": "replicas"}


class ClockSampler:
    """nvidia-smi samples of SM clock, power and throttle reasons while the timed region
    runs; ``mark(name)`` closes a phase, and the report gives each phase's medians too."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.proc = None
        self.phases = []  # (name, host start, host end)
        self._t = time.time()
        self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200", "-i", gpu_id], stdout=self.file, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def mark(self, name: str):
        """End the current phase (the caller has synchronised the device)."""
        now = time.time()
        self.phases.append((name, self._t, now))
        self._t = now

    @staticmethod
    def _stamp(text: str):
        import datetime
        try:
            return datetime.datetime.strptime(text.strip(), "%Y/%m/%d %H:%M:%S.%f").timestamp()
        except ValueError:
            return None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        self.proc.wait()
        self.file.flush()
        self.file.seek(0)
        rows = [r.split(",") for r in self.file.read().strip().splitlines() if r.strip()]
        os.unlink(self.file.name)
        samples, mx, reasons = [], 0.0, set()  # (time, sm MHz, power W)
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            try:
                pw = float(r[4]) if r[4].strip() not in ("", "[N/A]") else float("nan")
                samples.append((self._stamp(r[0]), float(r[2]), pw))
                mx = max(mx, float(r[3]))
                for name, v in zip(names, r[6:10]):
                    if v.strip().lower() == "active":
                        reasons.add(name)
            except (ValueError, IndexError):
                continue
        if not samples:
            return None
        out = {"sm_mhz": statistics.median(s[1] for s in samples), "sm_max_mhz": mx,
               "reasons": sorted(reasons), "samples": len(samples)}
        by_phase = {}
        for name, t0, t1 in self.phases:
            sel = [s for s in samples if s[0] is not None and t0 <= s[0] <= t1]
            if sel:
                pws = [s[2] for s in sel if s[2] == s[2]]
                by_phase[name] = {"sm_mhz": statistics.median(s[1] for s in sel),
                                  "power_w": statistics.median(pws) if pws else None,
                                  "samples": len(sel)}
        if by_phase:
            out["by_phase"] = by_phase
        return out


def slowest_rank(times_ms, world: int, device: str = "cuda"):
    """Replicas: every rank times its own steps; the job's step time is the slowest rank's.
    All-reduces (MAX) the list of timings over the default process group when world > 1
    and returns them as floats, identical on every rank."""
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(v) for v in times_ms], dtype=torch.float64, device=device)
    if world > 1:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t]


def job_tokens_per_s(world: int, tokens_per_rank: int, ms_per_step: float) -> float:
    """Weak scaling: each of `world` replicas processes its own batch of tokens per step; the
    job's throughput is all ranks' tokens over the slowest rank's step time."""
    return world * tokens_per_rank / (ms_per_step / 1e3)


def gpu_id_for(device_index: int) -> str:
    import torch
    try:
        return "GPU-" + str(torch.cuda.get_device_properties(device_index).uuid)
    except Exception:
        vis = os.environ.get("CUDA_VISIBLE_DEVICES")
        return vis.split(",")[device_index] if vis else str(device_index)


def oracle_aux(cfg, T_s: int):
    """Balancing-loss arguments of the oracle for a T_s-token sample: a sample shorter than
    one sequence is taken as one sequence."""
    if not cfg.has_aux:
        return None
    L = min(cfg.seq_len or T_s, T_s)
    return (L if T_s % L == 0 else T_s, cfg.aux_switch, cfg.aux_seq)


def oracle_pass_desc(cfg) -> str:
    """What one oracle step computes for this workload (as bench.py times it)."""
    parts = ["forward"]
    if cfg.backward:
        parts.append("backward")
    if cfg.bias_update:
        parts.append("bias update")
    desc = "fp64 " + "+".join(parts)
    if cfg.fp8:
        desc += ", FP8 (E4M3 rowwise) expert forward operands"
    if cfg.fp8_dgrad:
        desc += " and data-gradient operands"
    if cfg.has_aux:
        desc += ", both balancing losses (the sample as one sequence when shorter than one)"
    return desc


def cpu_oracle_rate(cfg, inp, T_s: int, steps: int = 1):
    """The fp64 oracle (forward + backward + bias update) on the first T_s tokens of the
    workload, all experts; returns (tokens/s, threads, seconds per step)."""
    from oracle import moe_oracle as O
    sub = dict(inp)
    sub["x"] = inp["x"][:T_s]
    i64 = {k: O.to64(v) for k, v in sub.items() if k != "dY"}
    dY = O.to64(inp["dY"][:T_s]) if cfg.backward else None
    aux = oracle_aux(cfg, T_s)
    times = []
    for _ in range(steps):
        t0 = time.perf_counter()
        fwd = O.layer_forward(i64, cfg.mode, cfg.k, cfg.z_coef, aux=aux,
                              fp8=cfg.fp8, fp8_dgrad=cfg.fp8_dgrad)
        if cfg.backward:
            O.layer_backward(i64, fwd, dY)
        if cfg.bias_update:
            rule = O.bias_update_proportional if cfg.bias_rule == "proportional" else O.bias_update
            rule(fwd["counts"], i64["b"].astype("float32"), T_s, cfg.k, cfg.gamma)
        times.append(time.perf_counter() - t0)
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    return T_s / statistics.median(times), cores, times


def cpu_desc_from(cpuinfo: str, machine: str) -> str:
    """The CPU model as a /proc/cpuinfo text names it (x86: model name; Arm: implementer and
    part numbers), with the machine type."""
    fields = {}
    for line in cpuinfo.splitlines():
        key, _, val = line.partition(":")
        fields.setdefault(key.strip(), val.strip())
    if fields.get("model name"):
        return f"{fields['model name']} ({machine})"
    if fields.get("CPU part"):
        return f"{machine}, CPU implementer {fields.get('CPU implementer', '?')} part {fields['CPU part']}"
    return machine


def host_cpu_desc() -> str:
    """This host's CPU model; the machine type alone when /proc/cpuinfo cannot be read."""
    import platform
    machine = platform.machine() or "unknown"
    try:
        with open("/proc/cpuinfo") as fh:
            return cpu_desc_from(fh.read(), machine)
    except OSError:
        return machine


def cpu_oracle_rate_one_core(config_name: str, T_s: int, steps: int = 1) -> float:
    """The same oracle timing on one host core: a child process whose numerical libraries
    are held to one thread. Returns tokens/s."""
    code = ("import json, sys, torch; torch.set_num_threads(1); sys.path.insert(0, %r); "
            "import bench; from pretraining_sigmoid_softmax_gb300.configs import CONFIGS; "
            "from pretraining_sigmoid_softmax_gb300.inputs import make_inputs; "
            "cfg = CONFIGS[%r]; r = bench.cpu_oracle_rate(cfg, make_inputs(cfg), %d, %d); "
            "print(json.dumps(r[0]))" % (ROOT, config_name, T_s, steps))
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1")
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, env=env,
                       timeout=600, check=True)
    return float(r.stdout.strip().splitlines()[-1])


def run_reference(args, cfg):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    from pretraining_sigmoid_softmax_gb300.inputs import make_inputs
    inp = make_inputs(cfg)
    T_s = max(8, min(args.cpu_sample_tokens // 4, cfg.T))
    _, cores, times = cpu_oracle_rate(cfg, inp, T_s, steps=args.warmup + args.steps)
    timed = times[args.warmup:] or times
    ms = 1e3 * sum(timed) / len(timed)
    value = T_s / (ms / 1e3)
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": workload_desc(cfg),
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                             "cpu": host_cpu_desc(),
                             "sample": f"first {T_s} tokens of the workload per step, all "
                                       f"{cfg.E} experts, {oracle_pass_desc(cfg)}"},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def main():
    args = parse()
    from pretraining_sigmoid_softmax_gb300.configs import CONFIGS
    cfg = CONFIGS[args.config]
    if args.impl == "reference":
        return run_reference(args, cfg)

    import torch
    import torch.distributed as dist
    from pretraining_sigmoid_softmax_gb300 import build, ops
    from pretraining_sigmoid_softmax_gb300.inputs import make_inputs
    from pretraining_sigmoid_softmax_gb300.layer import MoEPlan, MoEShape

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    if local == 0:
        build.build_library()
    if world > 1:
        dist.barrier()

    inp = make_inputs(cfg)
    dev = {k: v.cuda() for k, v in inp.items()}
    plan = MoEPlan(MoEShape.from_config(cfg), "cuda", backward=cfg.backward)
    # the end-to-end loop alternates two buffer sets; the second is made and warmed up here
    plan_b = None if args.no_e2e else MoEPlan(MoEShape.from_config(cfg), "cuda",
                                              backward=cfg.backward)
    b_work = dev["b"].clone()
    stream = torch.cuda.current_stream()

    def step(x, dY, p=plan):
        p.forward(x, dev["W_r"], b_work, dev["W_g"], dev["W_u"], dev["W_d"], dev.get("Ws_g"),
                  dev.get("Ws_u"), dev.get("Ws_d"))
        if cfg.backward:
            p.backward(dY)
            if cfg.bias_update:
                p.bias_update(b_work, cfg.gamma, cfg.bias_rule)

    def sync_all():
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()

    for _ in range(args.warmup):
        step(dev["x"], dev.get("dY"))
        if plan_b is not None:
            step(dev["x"], dev.get("dY"), plan_b)
    ops.moe_clear_device_status()
    sync_all()

    # ---------------------------------------------------------------- device-resident timing
    # Pass 1 (eager, the C-ABI calls issued one by one): CUDA events around every
    # grouped-GEMM call give the GEMM time of the roofline. Pass 2 (default): the same step
    # captured once as a CUDA graph and replayed, so host launch overhead is out of the
    # step; its time gives `value`.
    flush_buf = (torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device="cuda")
                 if needs_l2_flush(cfg) else None)

    def timed(run, n):
        sync_all()
        if flush_buf is None:  # the step's own data is far larger than L2
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            for _ in range(n):
                run()
            b.record(stream)
            sync_all()
            return a.elapsed_time(b)
        pairs = []  # small workloads: flush L2 before each step, time the steps alone
        for _ in range(n):
            flush_buf.fill_(0)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            run()
            b.record(stream)
            pairs.append((a, b))
        sync_all()
        return sum(a.elapsed_time(b) for a, b in pairs)

    plan.gemm_events = []
    sampler = ClockSampler(gpu_id_for(local))
    ms_eager = timed(lambda: step(dev["x"], dev.get("dY")), args.steps)
    gemm_ms = sum(a.elapsed_time(b) for a, b in plan.gemm_events)
    plan.gemm_events = None
    sampler.mark("device_eager")

    # ------------------------------------------------------------ end to end, host buffers
    # (between the two device-resident passes, under the same clock sampling)
    e2e = None
    if not args.no_e2e:
        # Pipelined like a training loop: step i+1's inputs are uploaded on a copy stream
        # while step i computes, and step i's out/dx are read back while step i+1 computes.
        # Two sets of activation buffers (plans) alternate so a readback never races the
        # next step's writes. Every step's copies are inside the timed region.
        plans = [plan, plan_b]
        hx = inp["x"].pin_memory()
        hdy = inp["dY"].pin_memory() if cfg.backward else None
        hout = [torch.empty_like(inp["x"]).pin_memory() for _ in range(2)]
        hdx = [torch.empty_like(inp["x"]).pin_memory() for _ in range(2)] if cfg.backward else None
        xd = [torch.empty_like(dev["x"]) for _ in range(2)]
        dyd = [torch.empty_like(dev["dY"]) for _ in range(2)] if cfg.backward else None
        up, down = torch.cuda.Stream(), torch.cuda.Stream()
        uploaded = [torch.cuda.Event() for _ in range(2)]
        computed = [torch.cuda.Event() for _ in range(2)]
        read_back = [torch.cuda.Event() for _ in range(2)]
        freed = [torch.cuda.Event() for _ in range(2)]  # inputs of a slot consumed

        def upload(i):
            j = i % 2
            up.wait_event(freed[j])
            with torch.cuda.stream(up):
                xd[j].copy_(hx, non_blocking=True)
                if cfg.backward:
                    dyd[j].copy_(hdy, non_blocking=True)
                uploaded[j].record(up)

        def run_steps(n):
            for j in range(2):  # nothing pending on either slot
                freed[j].record(stream)
                read_back[j].record(stream)
            upload(0)
            for i in range(n):
                j = i % 2
                if i + 1 < n:
                    upload(i + 1)
                stream.wait_event(uploaded[j])
                stream.wait_event(read_back[j])  # slot j's previous outputs are on the host
                p = plans[j]
                step(xd[j], dyd[j] if cfg.backward else None, p)
                freed[j].record(stream)
                computed[j].record(stream)
                down.wait_event(computed[j])
                with torch.cuda.stream(down):
                    hout[j].copy_(p.out, non_blocking=True)
                    if cfg.backward:
                        hdx[j].copy_(p.dx, non_blocking=True)
                    read_back[j].record(down)
            stream.wait_event(read_back[0])
            stream.wait_event(read_back[1])

        run_steps(args.warmup)
        sync_all()
        sampler.mark("e2e_warmup")
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        run_steps(args.steps)
        b.record(stream)
        sync_all()
        sampler.mark("e2e")
        ms_e2e = slowest_rank([a.elapsed_time(b)], world)[0] / args.steps
        nbytes = cfg.T * cfg.d * 2
        e2e = {"value": job_tokens_per_s(world, cfg.T, ms_e2e), "unit": "tokens/s",
               "h2d_bytes_per_step": nbytes * (2 if cfg.backward else 1),
               "d2h_bytes_per_step": nbytes * (2 if cfg.backward else 1),
               "ms_per_step": ms_e2e,
               "note": "pinned host buffers; uploads and readbacks overlap adjacent steps"}
        del plans, plan_b

    ms_graph = None
    if not args.no_graph:
        weights = {k: dev[k] for k in ("W_r", "W_g", "W_u", "W_d", "Ws_g", "Ws_u", "Ws_d") if k in dev}
        graph = plan.capture_step(dev["x"], weights, dev.get("dY") if cfg.backward else None,
                                  b_work, cfg.gamma, cfg.bias_rule, cfg.bias_update)
        graph.replay()
        torch.cuda.synchronize()
        sampler.mark("graph_capture")
        ms_graph = timed(graph.replay, args.steps)
        sampler.mark("device_graph")
    clocks = sampler.stop()
    code, site = ops.moe_device_status()
    if code != 0:
        raise RuntimeError(f"device status {code} ({ops.status_string(code)}) at site {site}")
    ms_eager, gemm_ms, ms_g = slowest_rank(
        [ms_eager, gemm_ms, ms_graph if ms_graph is not None else 0.0], world)
    ms_total = ms_g if ms_graph is not None else ms_eager
    ms_step = ms_total / args.steps
    value = job_tokens_per_s(world, cfg.T, ms_step)

    # ------------------------------------------------------------------------- report
    if rank != 0:
        if world > 1:
            dist.barrier()
            dist.destroy_process_group()
        return 0
    pk, kind = peaks()
    gemm_flops = cfg.gemm_flops()
    gemm_tflops = gemm_flops / (gemm_ms / args.steps / 1e3) / 1e12
    peak_t = float(pk.get("bf16_tflops_sustained", pk.get("bf16_tflops")))
    peak_kind = f"{kind} bf16 sustained"
    peak_nominal = NOMINAL_BF16_TFLOPS
    if cfg.fp8:
        # GEMMs on E4M3 have twice the dense bf16 rate (4.5 vs 2.25 PFLOP/s nominal): the
        # forward GEMMs are a third of the FLOPs with backward, and the data-gradient GEMMs
        # (fp8_dgrad) another third; the peak of the mix is the FLOP-weighted harmonic
        # combination of the measured bf16 peak and twice it
        f_fp8 = gemm_flops / (3.0 if cfg.backward else 1.0)
        if cfg.fp8_dgrad and cfg.backward:
            f_fp8 *= 2.0
        peak_t = gemm_flops / (f_fp8 / (2.0 * peak_t) + (gemm_flops - f_fp8) / peak_t)
        peak_nominal = gemm_flops / (f_fp8 / (2.0 * peak_nominal) +
                                     (gemm_flops - f_fp8) / peak_nominal)
        peak_kind = (f"{kind} bf16 sustained; fp8 forward"
                     f"{' and data-gradient' if cfg.fp8_dgrad else ''} GEMMs at 2x (nominal ratio)")
    line = {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic", "config": workload_desc(cfg),
            "gemm_tflops": gemm_tflops, "gemm_frac_of_peak": gemm_tflops / peak_t,
            "gemm_ms_per_step": gemm_ms / args.steps,
            "timing": {"value_from": "cuda_graph_replay" if not args.no_graph else "eager",
                       "eager_ms_per_step": ms_eager / args.steps,
                       "gemm_events_from": "eager pass, CUDA events around each grouped-GEMM call"},
            "roofline": {"bound": "tensor", "kernel": "grouped_gemm_kernel (all GEMM launches)",
                         "achieved": gemm_tflops, "peak": peak_t, "unit": "TFLOP/s",
                         "frac": gemm_tflops / peak_t, "peak_kind": peak_kind,
                         "peak_nominal": peak_nominal, "frac_of_nominal": gemm_tflops / peak_nominal,
                         "traffic": MEASURED_GEMM_TRAFFIC.get(args.config),
                         "traffic_unit": "bytes per step (all grouped-GEMM launches)",
                         "traffic_source": ("stored ncu capture (dram__bytes_read.sum + "
                                            "dram__bytes_write.sum) of these kernels at this "
                                            "workload, not measured in this run"
                                            if args.config in MEASURED_GEMM_TRAFFIC else None)},
            "gpu_launches": plan.launches_per_step(cfg.backward, cfg.bias_update) * args.steps,
            "gpu_launches_note": "kernels per timed pass (the graph pass replays the same kernels)",
            "clocks": clocks, "e2e": e2e}
    if clocks and clocks.get("sm_mhz"):
        # step time x median SM clock under load: comparable between runs at other clocks
        line["clock_normalised_ms_ghz"] = ms_step * clocks["sm_mhz"] / 1e3
    if world == 1 and not args.no_cpu_baseline:
        T_s = min(args.cpu_sample_tokens, cfg.T)
        rate, cores, _ = cpu_oracle_rate(cfg, inp, T_s)
        line["cpu_baseline"] = {"value": rate, "unit": "tokens/s", "cores": cores,
                                "kind": "oracle", "cpu": host_cpu_desc(),
                                "sample": f"first {T_s} tokens of the workload, all {cfg.E} "
                                          f"experts, {oracle_pass_desc(cfg)}"}
        if args.config == "C0":  # the tiny workload is also timed on one core
            line["cpu_baseline"]["one_core"] = cpu_oracle_rate_one_core("C0", T_s, steps=3)
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
