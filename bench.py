#!/usr/bin/env python3
"""Benchmark of the GB300 gradient allreduce.

Default workload (one line of JSON on stdout): the allreduce of one 25 MiB
fp32 DDP bucket across N = 8 virtual ranks held in one GPU's HBM
(8 x 6,553,600 fp32, N(0, 1e-3), op = avg), one fused ring-order pass per
step. Inputs are 200 MiB, larger than L2, so no flush between steps.

  metric: busbw GB/s = (M / t) * 2(N-1)/N, M = bytes per rank (the ring
          volume factor of the AllReduce glossary's algorithm table), and the
          fraction of the HBM roofline with bytes = 2*N*M per step.
  e2e:    the same metric with the host->device copy of the 8 inputs and the
          device->host copy of the 8 outputs (pinned host memory) inside the
          timed region, through the same C-ABI call.
  cpu_baseline: the CPU oracle (literal ring simulator, one thread) on the
          same workload, a bounded number of repetitions.

`--impl reference` times the oracle alone on this workload (rank 0 only).
Under torchrun each GPU runs its own full workload (weak scaling: the
virtual ranks already live on one device, so there is no exchange between
GPUs); a gloo process group supplies the barrier and the max over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import time
from pathlib import Path

ROOT = Path(__file__).resolve().parent
sys.path.insert(0, str(ROOT))

METRIC = "allreduce busbw GB/s and % of HBM roofline, N=8, 25 MB fp32 bucket, 1 GB300"
NRANKS = 8
COUNT = 6_553_600  # 25 MiB of fp32 per rank
SIGMA = 1e-3
OP = "avg"
FALLBACK_HBM_GBS = 6800.0


def busbw_gbs(bytes_per_rank: float, seconds: float, nranks: int = NRANKS) -> float:
    return bytes_per_rank / seconds * 2 * (nranks - 1) / nranks / 1e9


# ----------------------------------------------------------------- distributed plumbing


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def init_dist(world: int):
    if world <= 1:
        return None
    import torch.distributed as dist

    dist.init_process_group("gloo")
    return dist


def barrier(dist):
    if dist is not None:
        dist.barrier()


def max_over_ranks(dist, x: float) -> float:
    if dist is None:
        return x
    import torch

    t = torch.tensor([x], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(dist, x: float) -> float:
    if dist is None:
        return x
    import torch

    t = torch.tensor([x], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


# ----------------------------------------------------------------- clocks


class ClockSampler:
    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_id: str | None):
        self.device_id = device_id
        self.proc = None
        self.lines: list[str] = []

    def start(self):
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "50"]
        if self.device_id:
            cmd.insert(1, f"--id={self.device_id}")
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
        time.sleep(0.3)

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        time.sleep(0.15)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, smax, power, reasons = [], [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for line in out.splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
                power.append(float(f[3]))
            except ValueError:
                continue
            for name, val in zip(names, f[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        # samples under load: the upper half of the power readings
        pmid = statistics.median(power)
        loaded = [s for s, p in zip(sm, power) if p >= pmid] or sm
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm), "power_w_max": max(power)}


def device_uuid(dev: int) -> str | None:
    import torch

    try:
        u = torch.cuda.get_device_properties(dev).uuid
        s = str(u)
        return s if s.startswith("GPU-") else f"GPU-{s}"
    except Exception:
        return None


# ----------------------------------------------------------------- roofline inputs


def measured_peaks() -> dict:
    p = ROOT / "MEASURED_PEAKS.json"
    if p.exists():
        try:
            return json.loads(p.read_text())
        except ValueError:
            pass
    return {}


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    csrc = ROOT / "gradient_allreduce_collective_gb300" / "csrc"
    for p in sorted(csrc.iterdir()):
        if p.is_file():
            h.update(p.name.encode())
            h.update(p.read_bytes())
    return h.hexdigest()[:16]


def profiled_traffic(profile_name: str) -> float | None:
    """DRAM bytes per launch recorded from an ncu capture, if the kernel
    sources have not changed since (the summary records their hash)."""
    p = ROOT / "profiles" / profile_name
    if not p.exists():
        return None
    text = p.read_text(encoding="utf-8")
    m_hash = re.search(r"source_hash:\s*([0-9a-f]+)", text)
    m_bytes = re.search(r"dram_bytes_per_launch:\s*([0-9.eE+]+)", text)
    if not m_hash or not m_bytes or m_hash.group(1) != kernel_source_hash():
        return None
    return float(m_bytes.group(1))


# ----------------------------------------------------------------- CPU oracle timing


def oracle_baseline(budget_s: float, nranks: int = NRANKS, count: int = COUNT) -> dict:
    """Time the CPU oracle (the literal ring simulator, one thread) on a sample
    of the workload: the first `n` elements of every rank, n sized to fill
    about `budget_s` seconds, repeated at least twice."""
    import oracle
    import synthgen

    probe_n = 262_144
    send = synthgen.ranks_normal(nranks, count, SIGMA, base_seed=0)
    t0 = time.perf_counter()
    oracle.ring_allreduce([a[:probe_n] for a in send], "f32", OP)
    per_elem = (time.perf_counter() - t0) / probe_n
    n = int(min(count, max(probe_n, budget_s / 2 / per_elem)))
    sample = [a[:n] for a in send]
    reps, elapsed = 0, 0.0
    while reps < 2 or elapsed < budget_s * 0.5:
        t0 = time.perf_counter()
        oracle.ring_allreduce(sample, "f32", OP)
        elapsed += time.perf_counter() - t0
        reps += 1
        if elapsed > budget_s:
            break
    t = elapsed / reps
    return {"value": busbw_gbs(n * 4, t, nranks), "unit": "GB/s (busbw)", "cores": 1, "kind": "oracle",
            "sample": f"{nranks} ranks x first {n:,} of {count:,} fp32 (the full bucket when equal), op={OP}, "
                      f"{reps} repetitions, {t * 1e3:.1f} ms each, single-threaded C ring simulator",
            "ms_per_step": t * 1e3}


def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    import oracle
    import synthgen

    send = synthgen.ranks_normal(NRANKS, COUNT, SIGMA, base_seed=0)
    # size each step so that the whole run stays within about two minutes
    probe_n = 131_072
    t0 = time.perf_counter()
    oracle.ring_allreduce([a[:probe_n] for a in send], "f32", OP)
    per_elem = (time.perf_counter() - t0) / probe_n
    total_steps = max(1, args.steps + args.warmup)
    n = int(min(COUNT, max(4096, 90.0 / total_steps / per_elem)))
    n -= n % 64
    sample = [a[:n] for a in send]
    for _ in range(args.warmup):
        oracle.ring_allreduce(sample, "f32", OP)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.ring_allreduce(sample, "f32", OP)
    t = (time.perf_counter() - t0) / max(1, args.steps)
    value = busbw_gbs(n * 4, t)
    desc = (f"{NRANKS} ranks x first {n:,} of {COUNT:,} fp32 per step, op={OP}, single-threaded C ring "
            f"simulator (the CPU oracle)")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": t * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": workload_config("fused"),
        "cpu_baseline": {"value": value, "unit": "GB/s (busbw)", "cores": 1, "kind": "oracle", "sample": desc},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


# ----------------------------------------------------------------- GPU arm


def workload_config(algo: str) -> dict:
    return {
        "workload": f"allreduce of one 25 MiB fp32 DDP bucket: N={NRANKS} virtual ranks x {COUNT:,} fp32 "
                    f"in one GPU's HBM, op={OP}, {algo} ring-order pass",
        "nranks": NRANKS, "count_per_rank": COUNT, "bytes_per_rank": COUNT * 4, "op": OP, "algo": algo,
        "l2": "inputs 200 MiB and outputs 200 MiB exceed the 126 MiB L2; no flush between steps",
        "parallelism": "virtual ranks on one device; GPUs run independent buckets (weak scaling)",
    }


def time_steps(fn, steps: int, stream) -> float:
    import torch

    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    start.record(stream)
    for _ in range(steps):
        fn()
    end.record(stream)
    end.synchronize()
    return start.elapsed_time(end) / steps  # ms


def run_ours(args):
    import numpy as np
    import torch

    world, rank, local = dist_env()
    dist = init_dist(world)
    torch.cuda.set_device(local)
    import gradient_allreduce_collective_gb300 as gar
    import synthgen

    gar.build()
    gar.lib()
    stream = torch.cuda.current_stream()
    M = COUNT * 4
    send_np = synthgen.ranks_normal(NRANKS, COUNT, SIGMA, base_seed=0)
    send = [torch.from_numpy(a).cuda() for a in send_np]
    recv = [torch.empty_like(s) for s in send]

    def step_fused():
        gar.ar_allreduce(send, recv, OP, "fused", stream)

    for _ in range(args.warmup):
        step_fused()
    torch.cuda.synchronize()

    clocks = ClockSampler(device_uuid(local))
    clocks.start()
    barrier(dist)
    torch.cuda.synchronize()
    ms = time_steps(step_fused, args.steps, stream)
    torch.cuda.synchronize()
    barrier(dist)
    clk = clocks.stop()
    ms_max = max_over_ranks(dist, ms)

    # the same workload through the other two orders (not the headline)
    extra = {}
    for algo in ("ring", "tree"):
        def f(a=algo):
            gar.ar_allreduce(send, recv, OP, a, stream)
        for _ in range(max(3, args.warmup)):
            f()
        extra[algo] = time_steps(f, max(10, min(args.steps, 2000)), stream)

    # end to end: pinned host inputs -> device -> allreduce -> host outputs
    h_in = [torch.from_numpy(a).pin_memory() for a in send_np]
    h_out = [torch.empty(COUNT, dtype=torch.float32).pin_memory() for _ in range(NRANKS)]

    def step_e2e():
        for d, h in zip(send, h_in):
            d.copy_(h, non_blocking=True)
        gar.ar_allreduce(send, recv, OP, "fused", stream)
        for h, d in zip(h_out, recv):
            h.copy_(d, non_blocking=True)

    for _ in range(3):
        step_e2e()
    e2e_steps = max(5, min(args.steps, 200))
    barrier(dist)
    ms_e2e = max_over_ranks(dist, time_steps(step_e2e, e2e_steps, stream))
    torch.cuda.synchronize()
    ok = all(np.array_equal(h_out[r].numpy(), h_out[0].numpy()) for r in range(1, NRANKS))

    peaks = measured_peaks()
    peak = float(peaks.get("hbm_gbs", FALLBACK_HBM_GBS))
    peak_src = "measured (MEASURED_PEAKS.json hbm_gbs)" if "hbm_gbs" in peaks else "fallback"
    alg_bytes = 2 * NRANKS * M
    achieved = alg_bytes / (ms * 1e-3) / 1e9
    traffic = profiled_traffic("ar_fused_f32_avg_n8_25MiB.md")

    value = sum_over_ranks(dist, busbw_gbs(M, ms_max * 1e-3)) if dist else busbw_gbs(M, ms_max * 1e-3)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = oracle_baseline(args.cpu_budget)
        cpu.pop("ms_per_step", None)
    if rank != 0:
        return 0
    line = {
        "metric": METRIC,
        "value": value,
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms_max,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic (seeded SplitMix64 + Box-Muller N(0, 1e-3), rank r uses seed r)",
        "config": workload_config("fused"),
        "algbw_gbs": M / (ms_max * 1e-3) / 1e9,
        "hbm_gbs": achieved,
        "pct_hbm_roofline": 100.0 * achieved / peak,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "traffic": traffic, "kernel": "k_reduce<f32, avg, fused ring, N<=8>",
                     "algorithmic_bytes_per_launch": alg_bytes, "peak_source": peak_src},
        "e2e": {"value": (world if dist else 1) * busbw_gbs(M, ms_e2e * 1e-3), "unit": "GB/s",
                "ms_per_step": ms_e2e, "h2d_bytes_per_step": NRANKS * M, "d2h_bytes_per_step": NRANKS * M,
                "replicas_identical": ok},
        "gpu_launches": args.steps,
        "clocks": clk,
        "other_orders_ms_per_step": {"ring_rs_plus_ag": extra["ring"], "tree_recursive_halving": extra["tree"]},
        "cpu_baseline": cpu,
    }
    print(json.dumps(line))
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--cpu-budget", type=float, default=12.0, help="seconds of oracle time for cpu_baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
