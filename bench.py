#!/usr/bin/env python3
"""Benchmark of the GB300 gradient allreduce.

Default line (one JSON line on stdout): the allreduce of one 25 MiB fp32 DDP
bucket across N = 8 virtual ranks held in one GPU's HBM (8 x 6,553,600 fp32,
N(0, 1e-3), op = avg), one fused ring-order pass per step. Inputs are
200 MiB, larger than L2, so no flush between steps.

  metric: busbw GB/s = (M / t) * 2(N-1)/N, M = bytes per rank (the ring
          volume factor of the AllReduce glossary's algorithm table), and the
          fraction of the HBM roofline with bytes = 2*N*M per step.
  e2e:    the same metric with the host->device copy of the 8 inputs and the
          device->host copy of the 8 outputs (pinned host memory) inside the
          timed region, through the same C-ABI call; copies in and out run on
          their own streams with two device buffer sets, so one step's
          download overlaps the next step's upload.
  rows:   the other hot-path rows on their own workloads: the GPT-2-small
          DDP bucket sync (flatten -> allreduce -> unflatten, bf16, 8 ranks),
          the FP8-compressed allreduce (16 x 134,217,728 bf16) and Top-K
          sparsification with error feedback + the sparse allreduce (the
          bucket's 8 x 6,553,600 f32, k = 1%).
  cpu_baseline: the CPU oracle (literal ring simulator, one thread) on the
          same bucket, a bounded number of repetitions.

`--workload sweep` prints one line per message size (8 ranks, 4 KiB..1 GiB
per rank; fp32 uniform(-1,1) sum, or with `--sweep-dtype i32 --sweep-op
min|max` int32 uniform[-2^20, 2^20]; ring, tree, fused and the stepwise
executors; warm and cold L2).
`--workload fp8` and `--workload topk` print only that row; `--workload
strong` splits the bucket's elements over the GPUs (ar_allreduce_slice).
`--impl reference` times the oracle alone on the bucket (rank 0 only).
Under torchrun each GPU runs its own full workload (weak scaling: the
virtual ranks already live on one device, so there is no exchange between
GPUs); a gloo process group supplies the barrier and the max over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
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
CSRC = ROOT / "gradient_allreduce_collective_gb300" / "csrc"
FUSED_KERNEL_SOURCES = ("ar_internal.h", "ar_device.cuh", "ar_reduce_impl.cuh", "ar_reduce_f32.cu")


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

    if not dist.is_initialized():
        dist.init_process_group("gloo")
    return dist


def barrier(dist):
    if dist is not None:
        dist.barrier()


def reduce_over_ranks(dist, x: float, op: str) -> float:
    """max or sum of a host scalar over the ranks (identity without a group)."""
    if dist is None:
        return x
    import torch

    t = torch.tensor([x], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX if op == "max" else dist.ReduceOp.SUM)
    return float(t.item())


# ----------------------------------------------------------------- clocks


class ClockSampler:
    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_id: str | None):
        self.device_id = device_id
        self.proc = None

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
        pmid = statistics.median(power)  # samples under load: the upper half of the power readings
        loaded = [s for s, p in zip(sm, power) if p >= pmid] or sm
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm), "power_w_max": max(power)}


def device_uuid(dev: int) -> str | None:
    import torch

    try:
        s = str(torch.cuda.get_device_properties(dev).uuid)
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


def hbm_peak() -> tuple[float, str]:
    peaks = measured_peaks()
    if "hbm_gbs" in peaks:
        return float(peaks["hbm_gbs"]), "measured (MEASURED_PEAKS.json hbm_gbs)"
    return FALLBACK_HBM_GBS, "fallback"


def kernel_source_hash(files=FUSED_KERNEL_SOURCES) -> str:
    h = hashlib.sha256()
    for name in files:
        p = CSRC / name
        h.update(name.encode())
        h.update(p.read_bytes())
    return h.hexdigest()[:16]


def profiled_traffic(profile_name: str, files=FUSED_KERNEL_SOURCES) -> float | None:
    """DRAM bytes per launch recorded from an ncu capture, if the kernel's
    sources have not changed since (the summary records their hash)."""
    p = ROOT / "profiles" / profile_name
    if not p.exists():
        return None
    text = p.read_text(encoding="utf-8")
    m_hash = re.search(r"source_hash:\s*([0-9a-f]+)", text)
    m_bytes = re.search(r"dram_bytes_per_launch:\s*([0-9.eE+]+)", text)
    if not m_hash or not m_bytes or m_hash.group(1) != kernel_source_hash(files):
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
    out = {"value": busbw_gbs(n * 4, t, nranks), "unit": "GB/s (busbw)", "cores": 1, "kind": "oracle",
           "sample": f"{nranks} ranks x first {n:,} of {count:,} fp32 (the full bucket when equal), op={OP}, "
                     f"{reps} repetitions, {t * 1e3:.1f} ms each, single-threaded C ring simulator"}
    # the same per-element fold split over element ranges on every core this process may use
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)
    reps, elapsed = 0, 0.0
    while reps < 3 or elapsed < budget_s * 0.25:
        t0 = time.perf_counter()
        oracle.fold_allreduce_threads(sample, "f32", OP, cores)
        elapsed += time.perf_counter() - t0
        reps += 1
        if elapsed > budget_s * 0.5:
            break
    tm = elapsed / reps
    out["multicore"] = {"value": busbw_gbs(n * 4, tm, nranks), "unit": "GB/s (busbw)", "cores": cores,
                        "kind": "oracle",
                        "sample": f"same sample, per-element ring-order fold over {cores} element ranges on "
                                  f"{cores} threads, {reps} repetitions, {tm * 1e3:.1f} ms each"}
    return out


def workload_config(algo: str) -> dict:
    return {
        "workload": f"allreduce of one 25 MiB fp32 DDP bucket: N={NRANKS} virtual ranks x {COUNT:,} fp32 "
                    f"in one GPU's HBM, op={OP}, {algo} ring-order pass",
        "nranks": NRANKS, "count_per_rank": COUNT, "bytes_per_rank": COUNT * 4, "op": OP, "algo": algo,
        "l2": "inputs 200 MiB and outputs 200 MiB exceed the 126 MiB L2; no flush between steps",
        "parallelism": "virtual ranks on one device; GPUs run independent buckets (weak scaling)",
    }


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


# ----------------------------------------------------------------- GPU helpers


# About half a millisecond of SM cycles at the GB300's 2.07 GHz maximum clock.
HOLD_CYCLES = 1_000_000


def hold_stream(stream) -> None:
    """Keep `stream` busy for about 0.5 ms with PyTorch's spin kernel before a
    start event is recorded behind it. The host then has the first timed
    launches queued by the time the start event fires, so the timed region
    holds the device time of the steps and not the host's latency to issue
    the first one into an idle stream (the blocking-kernel idea of NVIDIA's
    NVBench). The steps themselves still run back to back as the host issues
    them; nothing of theirs is outside the region."""
    import torch

    with torch.cuda.stream(stream):
        torch.cuda._sleep(HOLD_CYCLES)


def time_steps(fn, steps: int, stream) -> float:
    """Average ms per call of fn() over `steps` calls, CUDA events on `stream`."""
    import torch

    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    hold_stream(stream)
    start.record(stream)
    for _ in range(steps):
        fn()
    end.record(stream)
    end.synchronize()
    return start.elapsed_time(end) / steps


def to_dev_bf16(a):
    import torch

    return torch.from_numpy(a).view(torch.int16).view(torch.bfloat16).cuda()


def oracle_row_timing(fn, max_n: int, budget_s: float = 6.0) -> dict:
    """Run `fn(n)` (the oracle on the first n elements of every rank, n <=
    max_n) on a sample sized to fill about budget_s / 4 seconds; returns
    seconds per element of one rank and the sample used."""
    n = min(16_384, max_n)
    while True:
        t0 = time.perf_counter()
        fn(n)
        t = time.perf_counter() - t0
        if t > budget_s / 4 or n >= max_n:
            break
        n = min(max_n, int(n * min(8.0, max(2.0, budget_s / 4 / max(t, 1e-6)))))
    return {"seconds_per_element_per_rank": t / n, "sample_elements_per_rank": n, "seconds": t}


def measure_ddp(gar, steps: int, warmup: int, with_oracle: bool = False) -> dict:
    """GPT-2-small DDP gradient sync on 8 ranks, two ways: (a) per bucket one
    flatten call for all ranks, one in-place fused allreduce (avg), one
    unflatten call; (b) per bucket one ar_bucket_allreduce straight from the
    gradient tensors (bit-identical results, no bucket copies). Then (b) on a
    communication stream overlapped with a synthetic backward pass (bf16 GEMMs
    on a compute stream), wall clock."""
    import torch
    import synthgen

    n = 8
    shapes = [s for _, s in synthgen.gpt2_small_param_shapes()]
    counts = [math.prod(s) for s in shapes]
    total = sum(counts)
    grads = [to_dev_bf16(g) for g in synthgen.ranks_normal(n, total, 1e-4, base_seed=0, dtype="bf16")]
    starts, pos = [], 0
    for c in counts:
        starts.append(pos)
        pos += c
    views = [[g[s:s + c] for s, c in zip(starts, counts)] for g in grads]
    bucket_of, offset_of, bcounts = gar.ar_bucket_plan(counts, torch.bfloat16, 25 * 1024 * 1024)
    plan, fused = [], []
    for b, bc in enumerate(bcounts):
        stride = (bc + 127) // 128 * 128  # 256-byte aligned rank slots
        flat = torch.empty(n * stride, dtype=torch.bfloat16, device="cuda")
        ids = [t for t in range(len(counts)) if bucket_of[t] == b]
        tens = [views[r][t] for r in range(n) for t in ids]
        offs = [r * stride + offset_of[t] for r in range(n) for t in ids]
        ranks = [flat[r * stride:r * stride + bc] for r in range(n)]
        plan.append((flat, tens, offs, ranks))
        fused.append(([[views[r][t] for t in ids] for r in range(n)], [offset_of[t] for t in ids], bc))
    stream = torch.cuda.current_stream()

    def three_step(st):
        for flat, tens, offs, ranks in plan:
            gar.ar_bucket_flatten(tens, offs, flat, st)
            gar.ar_allreduce(ranks, ranks, "avg", "fused", st)
            gar.ar_bucket_unflatten(flat, tens, offs, st)

    def direct(st):
        for tens, offs, bc in fused:
            gar.ar_bucket_allreduce(tens, tens, offs, bc, "avg", "fused", st)

    def graph_of(fn):
        g = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream()
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            g.capture_begin()
            fn(side)
            g.capture_end()
        stream.wait_stream(side)
        for _ in range(3):
            g.replay()
        return g

    res = {}
    for name, fn in (("three_step", three_step), ("direct", direct)):
        for _ in range(warmup):
            fn(stream)
        eager = time_steps(lambda: fn(stream), steps, stream)
        g = graph_of(fn)
        res[name] = (eager, time_steps(g.replay, steps, stream), g)
    peak, _ = hbm_peak()
    grad_bytes = total * 2

    # overlap: synthetic backward (bf16 GEMMs) on one stream, direct sync on another
    # (default priority, and a high-priority comm stream whose blocks the
    # scheduler starts first whenever an SM has room)
    comp, comm = torch.cuda.Stream(), torch.cuda.Stream()
    lo_pri, hi_pri = torch.cuda.Stream.priority_range() if hasattr(torch.cuda.Stream, "priority_range") else (0, -1)
    comm_hi = torch.cuda.Stream(priority=min(lo_pri, hi_pri))
    a = torch.randn(4096, 4096, device="cuda", dtype=torch.bfloat16)
    w = torch.randn(4096, 4096, device="cuda", dtype=torch.bfloat16)
    o = torch.empty_like(a)
    g_direct = res["direct"][2]

    def backward():
        for _ in range(8):
            torch.matmul(a, w, out=o)

    def timed(run):
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for _ in range(20):
            run()
        torch.cuda.synchronize()
        return (time.perf_counter() - t0) / 20 * 1e3

    def both_on(cs):
        def run():
            ev = torch.cuda.Event()
            ev.record(stream)
            comp.wait_event(ev)
            cs.wait_event(ev)
            with torch.cuda.stream(comp):
                backward()
            with torch.cuda.stream(cs):
                direct(cs)
            stream.wait_stream(comp)
            stream.wait_stream(cs)
        return run

    both, both_hi = both_on(comm), both_on(comm_hi)
    for _ in range(3):
        backward()
        both()
        both_hi()
    t_comp = timed(backward)
    t_comm = timed(lambda: direct(stream))
    t_both = timed(both)
    t_both_hi = timed(both_hi)
    out = {
        "workload": "DDP gradient sync: GPT-2-small shapes (148 tensors, 124,439,808 bf16 values) x 8 ranks, "
                    "N(0,1e-4), 9 buckets of <= 25 MiB, avg with binary32 accumulation",
        "buckets": len(bcounts),
    }
    for name, (eager, graph, _) in res.items():
        best = min(eager, graph)
        moved = (6 if name == "three_step" else 2) * n * grad_bytes
        out[name] = {"ms_per_step_eager": eager, "ms_per_step_cuda_graph": graph,
                     "launches_per_step": (3 if name == "three_step" else 1) * len(bcounts),
                     "busbw_gbs": busbw_gbs(grad_bytes, best * 1e-3, n),
                     "algorithmic_bytes_per_step": moved, "hbm_gbs": moved / (best * 1e-3) / 1e9,
                     "frac_hbm": moved / (best * 1e-3) / 1e9 / peak}
    out["three_step"]["what"] = "per bucket: flatten (all ranks) -> fused allreduce in place -> unflatten"
    out["direct"]["what"] = "per bucket: ar_bucket_allreduce from the tensors (no bucket copies)"
    if with_oracle:
        import oracle
        samp = synthgen.ranks_normal(n, 1 << 22, 1e-4, base_seed=0, dtype="bf16")
        o = oracle_row_timing(lambda k: oracle.ring_allreduce([a[:k] for a in samp], "bf16", "avg"), samp[0].size)
        t_all = o["seconds_per_element_per_rank"] * total
        out["cpu_oracle"] = {"kind": "oracle", "cores": 1,
                             "sample": f"ring allreduce (bf16, avg, 8 ranks) of the first "
                                       f"{o['sample_elements_per_rank']:,} values of a bucket, "
                                       f"{o['seconds']:.2f} s; scaled to all {total:,} values",
                             "ms_per_step_estimate": t_all * 1e3,
                             "busbw_gbs": busbw_gbs(grad_bytes, t_all, n)}
    out["overlap"] = {"backward_ms": t_comp, "sync_ms": t_comm, "both_ms": t_both,
                      "hidden_fraction_of_sync": max(0.0, (t_comp + t_comm - t_both) / t_comm),
                      "both_ms_high_priority_comm": t_both_hi,
                      "hidden_fraction_of_sync_high_priority_comm": max(0.0, (t_comp + t_comm - t_both_hi) / t_comm),
                      "what": "8 bf16 4096^3 GEMMs (torch.matmul) on a compute stream while the direct "
                              "sync (9 ar_bucket_allreduce launches) runs on a communication stream of default "
                              "or of the highest priority; wall clock, 20 reps"}
    return out


def measure_fp8(gar, steps: int, warmup: int, count: int = 134_217_728, with_oracle: bool = False) -> dict:
    """16 ranks x `count` bf16 with 0.1% outliers x100: quantise to E4M3
    blocks (workspace) then dequantise + fused ring-order reduce (sum) + 16
    bf16 replicas."""
    import torch
    import synthgen

    import numpy as np

    n = 16
    host = synthgen.ranks_normal(n, count, 1e-3, base_seed=0, dtype="bf16", outlier_p=1e-3, outlier_scale=100.0)
    send = [to_dev_bf16(a) for a in host]
    recv = [torch.empty_like(s) for s in send]
    ws = torch.empty(gar.ar_fp8_workspace_bytes(n, count), dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()

    def step():
        gar.ar_allreduce_fp8(send, recv, ws, "sum", "fused", stream)

    for _ in range(warmup):
        step()
    ms = time_steps(step, steps, stream)

    def step_fused():
        gar.ar_allreduce_fp8_fused(send, recv, "sum", "fused", stream)

    for _ in range(warmup):
        step_fused()
    ms_fused = time_steps(step_fused, steps, stream)
    # error against the fp64 sum on sampled elements, quantised once vs on every hop
    idx = np.sort(np.random.default_rng(0).choice(count, min(count, 1 << 20), replace=False))
    xs = np.stack([(a[idx].astype(np.uint32) << 16).view(np.float32).astype(np.float64) for a in host])
    ystar = xs.sum(axis=0)
    idx_t = torch.from_numpy(idx).cuda()

    def sampled_error(out):
        y = out[0].float()[idx_t].double().cpu().numpy()
        return float(np.linalg.norm(y - ystar) / np.linalg.norm(ystar))

    err_once = sampled_error(recv)

    def step_hops():
        gar.ar_allreduce_fp8_hops(send, recv, "sum", stream)

    for _ in range(warmup):
        step_hops()
    ms_hops = time_steps(step_hops, max(3, steps // 2), stream)
    torch.cuda.synchronize()
    err_hops = sampled_error(recv)
    M = count * 2
    wire = count + 4 * (count // 128)  # E4M3 codes + block scales per rank
    moved = n * M + n * wire + n * wire + n * M
    peak, _ = hbm_peak()
    del send, recv, ws
    torch.cuda.empty_cache()
    cpu = None
    if with_oracle:
        import oracle
        samp = synthgen.ranks_normal(n, 1 << 20, 1e-3, base_seed=0, dtype="bf16", outlier_p=1e-3,
                                     outlier_scale=100.0)
        o = oracle_row_timing(lambda k: oracle.fp8_ring_allreduce([a[:k] for a in samp], "bf16", "bf16", "sum"),
                              samp[0].size)
        t_all = o["seconds_per_element_per_rank"] * count
        cpu = {"kind": "oracle", "cores": 1,
               "sample": f"FP8 ring allreduce (16 ranks, bf16 in/out, sum) of the first "
                         f"{o['sample_elements_per_rank']:,} values per rank, {o['seconds']:.2f} s; "
                         f"scaled to {count:,}",
               "ms_per_step_estimate": t_all * 1e3, "busbw_gbs": busbw_gbs(count * 2, t_all, n)}
    return {
        "cpu_oracle": cpu,
        "workload": f"FP8-compressed allreduce: 16 ranks x {count:,} bf16, N(0,1e-3), 0.1% outliers "
                    "x100, E4M3 per-128 block scales, binary32 accumulation, sum, bf16 out, fused",
        "materialised": {"what": "quantise every rank into the workspace (the wire format), then dequantise + "
                                 "reduce + write 16 replicas",
                         "ms_per_step": ms, "busbw_gbs": busbw_gbs(M, ms * 1e-3, n),
                         "hbm_gbs": moved / (ms * 1e-3) / 1e9, "frac_hbm": moved / (ms * 1e-3) / 1e9 / peak,
                         "algorithmic_bytes_per_step": moved, "launches_per_step": 2},
        "fused_quantisation": {"what": "ar_allreduce_fp8_fused: quantise, dequantise and reduce in registers, "
                                       "same bits, no workspace",
                               "ms_per_step": ms_fused, "busbw_gbs": busbw_gbs(M, ms_fused * 1e-3, n),
                               "hbm_gbs": 2 * n * M / (ms_fused * 1e-3) / 1e9,
                               "frac_hbm": 2 * n * M / (ms_fused * 1e-3) / 1e9 / peak,
                               "algorithmic_bytes_per_step": 2 * n * M, "launches_per_step": 1,
                               "normwise_error_vs_fp64": err_once},
        "per_hop": {"what": "ar_allreduce_fp8_hops: the running partial re-quantised to FP8 on each of the 15 "
                            "ring hops, the finished chunk once more for the all-gather",
                    "ms_per_step": ms_hops, "busbw_gbs": busbw_gbs(M, ms_hops * 1e-3, n),
                    "hbm_gbs": 2 * n * M / (ms_hops * 1e-3) / 1e9,
                    "frac_hbm": 2 * n * M / (ms_hops * 1e-3) / 1e9 / peak,
                    "algorithmic_bytes_per_step": 2 * n * M, "launches_per_step": 1,
                    "normwise_error_vs_fp64": err_hops},
    }


SPEC_PROBES = 40  # untimed Top-K steps after the timed ones, each checked for the speculative path


def measure_topk(gar, steps: int, warmup: int, count: int = COUNT, frac: float = 0.01,
                 with_oracle: bool = False) -> dict:
    """Top-K sparsification with error feedback on 8 ranks x `count` f32
    (k = frac * count per rank, the residual carried from step to step), then
    the allreduce (avg) of the sparse vectors."""
    import torch
    import synthgen

    n = NRANKS
    k = int(count * frac)
    grads = [torch.from_numpy(a).cuda() for a in synthgen.ranks_normal(n, count, 1e-3, base_seed=0)]
    res = [torch.zeros(count, device="cuda") for _ in range(n)]
    idx = [torch.empty(k, dtype=torch.int32, device="cuda") for _ in range(n)]
    val = [torch.empty(k, dtype=torch.float32, device="cuda") for _ in range(n)]
    out = [torch.empty(count, device="cuda") for _ in range(n)]
    ws = torch.empty(gar.ar_topk_workspace_bytes(n, count, k), dtype=torch.uint8, device="cuda")
    sws = torch.empty(gar.ar_sparse_workspace_bytes(n, count), dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()

    def compress():
        gar.ar_topk_compress(grads, res, k, idx, val, ws, stream)

    def sparse_ar():
        gar.ar_sparse_allreduce(idx, val, [k] * n, out, "avg", "fused", sws, stream)

    def step():
        compress()
        sparse_ar()

    # at least 100 untimed steps: with the same gradients every step the
    # residual grows from call to call, and the threshold hint (and with it
    # the speculative first pass, which reads the data once) settles after
    # ~30 calls, T's leading 11 bits (which let pass 1 find the second digit
    # too) after ~100; a training run spends nearly all its steps past both
    for _ in range(max(warmup, 100)):
        step()
    # each loop times at least 100 calls: the first call of a back-to-back
    # run pays the pipeline fill, which a 20-call window spreads over few
    # calls (the sparse allreduce read 0.0365 ms over 20 calls, 0.0351 over 100)
    reps = max(steps, 100)
    ms = time_steps(step, reps, stream)
    ms_c = time_steps(compress, reps, stream)
    ms_s = time_steps(sparse_ar, reps, stream)
    # the same step as one CUDA graph (host launch cost removed)
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        g.capture_begin()
        gar.ar_topk_compress(grads, res, k, idx, val, ws, side)
        gar.ar_sparse_allreduce(idx, val, [k] * n, out, "avg", "fused", sws, side)
        g.capture_end()
    stream.wait_stream(side)
    for _ in range(3):
        g.replay()
    ms_graph = time_steps(g.replay, reps, stream)
    # how often pass 1's speculative candidate slots served the split pass
    # (one full pass over the data instead of two): rank 0's spec_ok word after
    # each of SPEC_PROBES further steps, untimed
    # and how often pass 1 also found the second digit (the previous call's
    # first digit held), so that the split pass returned at once
    spec_hits = pre2_hits = 0
    for _ in range(SPEC_PROBES):
        step()
        torch.cuda.synchronize()
        spec_hits += int(ws.view(torch.int32)[2048 + 10]) == 1
        pre2_hits += int(ws.view(torch.int32)[2048 + 14]) == 1
    spec = spec_hits / SPEC_PROBES
    M = count * 4
    min_c = n * 3 * M + n * k * 8          # read g and e, write e; the pairs
    struct_c = n * (3 * M + (1 - spec) * M) + 3 * n * k * 8  # + pass 2 over the data unless speculated
    sparse_b = n * M + n * k * 8  # the N outputs written once, the pairs read
    peak, _ = hbm_peak()
    del grads, res, idx, val, out, ws, sws, g
    torch.cuda.empty_cache()
    cpu = None
    if with_oracle:
        import numpy as np
        import oracle
        samp_g = synthgen.ranks_normal(n, 1 << 20, 1e-3, base_seed=0)
        zero = np.zeros(1 << 20, dtype=np.float32)

        def oracle_step(m):
            pairs = [oracle.topk_compress(g[:m], zero[:m], max(1, int(m * frac)))[:2] for g in samp_g]
            oracle.sparse_ring_allreduce([p[0] for p in pairs], [p[1] for p in pairs], m, "avg")

        o = oracle_row_timing(oracle_step, 1 << 20)
        t_all = o["seconds_per_element_per_rank"] * count
        cpu = {"kind": "oracle", "cores": 1,
               "sample": f"Top-K (1%) of 8 ranks then the ring allreduce of the sparse vectors, first "
                         f"{o['sample_elements_per_rank']:,} values per rank, {o['seconds']:.2f} s; scaled to "
                         f"{count:,}",
               "ms_per_step_estimate": t_all * 1e3}
    return {
        "cpu_oracle": cpu,
        "workload": f"Top-K sparsification with error feedback: {n} ranks x {count:,} f32 N(0,1e-3), "
                    f"k = {k:,} ({frac:.0%}) per rank, residual carried across steps; then the allreduce (avg, "
                    "fused ring order) of the sparse vectors",
        "ms_per_step": ms,
        "ms_per_step_graph": ms_graph,
        "timed_calls_per_loop": reps,
        "compress": {"ms": ms_c, "launches": 6, "min_bytes": min_c, "structure_bytes": struct_c,
                     "full_data_passes": round(2 - spec, 3), "speculative_share": spec,
                     "second_digit_in_pass1_share": pre2_hits / SPEC_PROBES,
                     "hbm_gbs_min_bytes": min_c / (ms_c * 1e-3) / 1e9,
                     "hbm_gbs_structure": struct_c / (ms_c * 1e-3) / 1e9,
                     "frac_hbm_structure": struct_c / (ms_c * 1e-3) / 1e9 / peak},
        "sparse_allreduce": {"ms": ms_s, "launches": 2, "bytes": sparse_b,
                             "hbm_gbs": sparse_b / (ms_s * 1e-3) / 1e9,
                             "frac_hbm": sparse_b / (ms_s * 1e-3) / 1e9 / peak},
        "wire_bytes_per_rank": {"dense_f32": M, "sparse_pairs": k * 8, "ratio": M / (k * 8)},
    }


# ----------------------------------------------------------------- GPU arm: headline


def rows_summary(rows: dict, other: dict, ms_headline: float, peak: float) -> dict:
    """Milliseconds per step and fraction of the measured HBM peak of every
    row, compact, so that they survive a truncated log next to the headline."""
    alg = 2 * NRANKS * COUNT * 4

    def ent(ms, moved):
        return {"ms": round(ms, 4), "frac": round(moved / (ms * 1e-3) / 1e9 / peak, 3)}

    out = {"fused_ring": ent(ms_headline, alg), "tree": ent(other["tree"], alg),
           "ring_rs_ag": ent(other["ring"], (2 * NRANKS + 1) * COUNT * 4)}  # reduce-scatter + all-gather bytes
    ddp = rows.get("ddp_bucket_sync")
    if ddp:
        for name in ("direct", "three_step"):
            r = ddp[name]
            best = min(r["ms_per_step_eager"], r["ms_per_step_cuda_graph"])
            out[f"ddp_{name}"] = {"ms": round(best, 4), "frac": round(r["frac_hbm"], 3)}
    fp8 = rows.get("fp8_allreduce")
    if fp8:
        for name in ("materialised", "fused_quantisation", "per_hop"):
            r = fp8[name]
            out[f"fp8_{name}"] = {"ms": round(r["ms_per_step"], 4), "frac": round(r["frac_hbm"], 3)}
    tk = rows.get("topk_sparse_allreduce")
    if tk:
        c = tk["compress"]
        out["topk_compress"] = {"ms": round(c["ms"], 4), "frac_min_bytes": round(c["hbm_gbs_min_bytes"] / peak, 3),
                                "frac_structure": round(c["frac_hbm_structure"], 3),
                                "speculative_share": c.get("speculative_share"),
                                "second_digit_in_pass1_share": c.get("second_digit_in_pass1_share")}
        sp = tk["sparse_allreduce"]
        out["sparse_allreduce"] = {"ms": round(sp["ms"], 4), "frac": round(sp["frac_hbm"], 3)}
    return out


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
    ms_max = reduce_over_ranks(dist, ms, "max")

    # per-call durations (the vasteelab metrics list: average, p95, p99 per call site)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(200)]
    for a, b in evs:
        a.record(stream)
        step_fused()
        b.record(stream)
    torch.cuda.synchronize()
    per_call = sorted(a.elapsed_time(b) * 1e3 for a, b in evs)
    pct = {"p50": per_call[len(per_call) // 2], "p95": per_call[int(len(per_call) * 0.95)],
           "p99": per_call[int(len(per_call) * 0.99)], "mean": sum(per_call) / len(per_call),
           "what": "200 fused calls, each between its own CUDA events (includes event overhead)"}

    # the same bucket through the other two orders (not the headline)
    other = {}
    for algo in ("ring", "tree"):
        def f(a=algo):
            gar.ar_allreduce(send, recv, OP, a, stream)
        for _ in range(max(3, args.warmup)):
            f()
        other[algo] = time_steps(f, max(10, min(args.steps, 2000)), stream)

    # end to end: pinned host inputs -> device -> allreduce -> pinned host outputs
    h_in = [torch.from_numpy(a).pin_memory() for a in send_np]
    h_out = [torch.empty(COUNT, dtype=torch.float32).pin_memory() for _ in range(NRANKS)]
    d_in = [[torch.empty(COUNT, device="cuda") for _ in range(NRANKS)] for _ in range(2)]
    d_out = [[torch.empty(COUNT, device="cuda") for _ in range(NRANKS)] for _ in range(2)]
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_red = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]
    k = [0]

    def step_e2e():
        j = k[0] & 1
        k[0] += 1
        with torch.cuda.stream(s_in):
            s_in.wait_event(ev_red[j])  # the previous reduction that read this input set is done
            for d, h in zip(d_in[j], h_in):
                d.copy_(h, non_blocking=True)
            ev_in[j].record(s_in)
        stream.wait_event(ev_in[j])
        stream.wait_event(ev_out[j])  # the previous download of this output set is done
        gar.ar_allreduce(d_in[j], d_out[j], OP, "fused", stream)
        ev_red[j].record(stream)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev_red[j])
            for h, d in zip(h_out, d_out[j]):
                h.copy_(d, non_blocking=True)
            ev_out[j].record(s_out)

    for e in ev_red + ev_out:
        e.record(stream)
    for _ in range(3):
        step_e2e()
    torch.cuda.synchronize()
    e2e_steps = max(5, min(args.steps, 200))
    barrier(dist)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    hold_stream(stream)
    start.record(stream)
    s_in.wait_stream(stream)  # the first upload starts after the start event, not during the hold
    for _ in range(e2e_steps):
        step_e2e()
    stream.wait_stream(s_out)
    end.record(stream)
    end.synchronize()
    ms_e2e = reduce_over_ranks(dist, start.elapsed_time(end) / e2e_steps, "max")
    gar.ar_allreduce(send, recv, OP, "fused", stream)  # recv last held the tree-order result
    want = recv[0].cpu().numpy()
    ok = all(np.array_equal(h.numpy(), want) for h in h_out)

    rows = {}
    if not args.headline_only:
        del d_in, d_out
        timed_cpu = rank == 0 and world == 1 and not args.no_cpu_baseline
        rows["ddp_bucket_sync"] = measure_ddp(gar, steps=max(5, min(args.steps, 50)), warmup=3,
                                              with_oracle=timed_cpu)
        rows["fp8_allreduce"] = measure_fp8(gar, steps=max(5, min(args.steps, 20)), warmup=3,
                                            with_oracle=timed_cpu)
        rows["topk_sparse_allreduce"] = measure_topk(gar, steps=max(5, min(args.steps, 50)), warmup=3,
                                                     with_oracle=timed_cpu)

    peak, peak_src = hbm_peak()
    alg_bytes = 2 * NRANKS * M
    achieved = alg_bytes / (ms * 1e-3) / 1e9
    traffic = profiled_traffic("ar_fused_f32_avg_n8_25MiB.md")
    value = reduce_over_ranks(dist, busbw_gbs(M, ms_max * 1e-3), "sum") if dist else busbw_gbs(M, ms_max * 1e-3)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = oracle_baseline(args.cpu_budget)
    if rank != 0:
        return 0
    summary = rows_summary(rows, other, ms_max, peak)
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
        "rows_summary": summary,
        "algbw_gbs": M / (ms_max * 1e-3) / 1e9,
        "hbm_gbs": achieved,
        "pct_hbm_roofline": 100.0 * achieved / peak,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "traffic": traffic, "kernel": "k_reduce<f32, avg, fused ring, N<=8>",
                     "algorithmic_bytes_per_launch": alg_bytes, "peak_source": peak_src},
        "e2e": {"value": (world if dist else 1) * busbw_gbs(M, ms_e2e * 1e-3), "unit": "GB/s",
                "ms_per_step": ms_e2e, "h2d_bytes_per_step": NRANKS * M, "d2h_bytes_per_step": NRANKS * M,
                "pipelined": "copy-in and copy-out streams, two device buffer sets", "replicas_identical": ok},
        "gpu_launches": args.steps,
        "clocks": clk,
        "per_call_us": pct,
        "other_orders_ms_per_step": {"ring_rs_plus_ag": other["ring"], "tree_recursive_halving": other["tree"]},
        "rows": rows,
        "cpu_baseline": cpu,
    }
    print(json.dumps(line))
    return 0


# ----------------------------------------------------------------- GPU arm: strong scaling


def run_strong(args):
    """The bucket shared by all GPUs: GPU g computes elements [g*count/G,
    (g+1)*count/G) of every rank with ar_allreduce_slice (the whole problem's
    chunk plan, no exchange between GPUs); value = the bucket's busbw at the
    slowest GPU's time."""
    import torch

    world, rank, local = dist_env()
    dist = init_dist(world)
    torch.cuda.set_device(local)
    import gradient_allreduce_collective_gb300 as gar
    import synthgen

    gar.build()
    gar.lib()
    stream = torch.cuda.current_stream()
    lo, hi = COUNT * rank // world, COUNT * (rank + 1) // world
    lo -= lo % 4
    hi = COUNT if rank == world - 1 else hi - hi % 4
    send_np = synthgen.ranks_normal(NRANKS, COUNT, SIGMA, base_seed=0)
    send = [torch.from_numpy(a[lo:hi].copy()).cuda() for a in send_np]
    recv = [torch.empty_like(x) for x in send]

    def step():
        gar.ar_allreduce_slice(send, recv, COUNT, lo, OP, "fused", stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    clocks = ClockSampler(device_uuid(local))
    clocks.start()
    barrier(dist)
    torch.cuda.synchronize()
    ms = time_steps(step, args.steps, stream)
    torch.cuda.synchronize()
    barrier(dist)
    clk = clocks.stop()
    ms_max = reduce_over_ranks(dist, ms, "max")
    if rank != 0:
        return 0
    M = COUNT * 4
    print(json.dumps({
        "metric": METRIC, "value": busbw_gbs(M, ms_max * 1e-3), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_max, "higher_is_better": True,
        "scaling": "strong", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": dict(workload_config("fused"), parallelism=f"the bucket's elements split over {world} GPU(s)"),
        "hbm_gbs_per_gpu": 2 * NRANKS * (hi - lo) * 4 / (ms * 1e-3) / 1e9, "clocks": clk,
        "gpu_launches": args.steps * (1 if lo % (-(-COUNT // NRANKS)) == 0 else 2)}))
    return 0


# ----------------------------------------------------------------- GPU arm: size sweep


def stepwise16_traffic(algo: str, n: int) -> float:
    """Bytes per call of the 16-bit stepwise orders, in units of M (bytes per
    rank, 2 per element): reduce-scatter steps read 2-byte inputs or 4-byte
    binary32 partials and write partials (the last step 2-byte results); the
    all-gather steps copy 2-byte values."""
    if algo == "step_ring":  # N-1 steps over every chunk: 8, 10, ..., 10, 8 bytes per element
        rs = 8 * 2 + 10 * (n - 3) if n >= 3 else 6
    else:  # level i combines N * count / 2^(i+1) elements: 8 (2+2+4), 12 (4+4+4), ..., 10 (4+4+2) bytes each
        levels = int(math.log2(n))
        rs = 0.0
        for i in range(levels):
            a = 2 if i == 0 else 4
            w = 2 if i == levels - 1 else 4
            rs += n / 2 ** (i + 1) * (2 * a + w)
    ag = 4 * (n - 1)  # N-1 copies of count elements of 2 bytes, read and written
    return (rs + ag) / 2


def run_sweep(args):
    import torch

    import gradient_allreduce_collective_gb300 as gar
    import synthgen

    torch.cuda.set_device(dist_env()[2])
    gar.build()
    gar.lib()
    n = 8
    max_bytes = args.sweep_max_bytes
    dtype, op = args.sweep_dtype, args.sweep_op
    es = 2 if dtype == "bf16" else 4
    nmax = max_bytes // es
    if dtype == "i32" and op not in ("min", "max"):
        raise SystemExit("the int32 leg of the sweep takes --sweep-op min or max")
    send = []
    for r in range(n):  # one rank at a time on the host: 1 GiB each at the largest size
        if dtype == "i32":
            t = torch.from_numpy(synthgen.uniform_i32(nmax, r, -(2**20), 2**20))
        elif dtype == "bf16":
            t = torch.from_numpy(synthgen.to_dtype(synthgen.uniform_f32(nmax, r, -1.0, 1.0), "bf16")).view(
                torch.int16).view(torch.bfloat16)
        else:
            t = torch.from_numpy(synthgen.uniform_f32(nmax, r, -1.0, 1.0))
        send.append(t.cuda())
        del t
    # binary32 partials of the 16-bit stepwise orders
    ws = (torch.empty(gar.ar_stepwise_workspace_bytes(n, nmax, dtype), dtype=torch.uint8, device="cuda")
          if es == 2 else None)
    recv = [torch.empty_like(s) for s in send]
    l2 = torch.cuda.get_device_properties(0).L2_cache_size
    flush = torch.empty(2 * l2 // 4 + 1024, dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream()
    peak, _ = hbm_peak()
    fits: dict[str, list] = {}
    size = 4096
    while size <= max_bytes:
        cnt = size // es
        s_v = [t[:cnt] for t in send]
        r_v = [t[:cnt] for t in recv]
        res = {}
        for algo in ("fused", "tree", "ring"):
            def f(a=algo):
                gar.ar_allreduce(s_v, r_v, op, a, stream)
            for _ in range(5):
                f()
            reps = max(5, min(2000, int(2e9 / (2 * n * size))))
            warm = time_steps(f, reps, stream)
            # cold: flush L2 before every call, time the call alone
            ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(20)]
            for a, b in ev:
                flush.fill_(1.0)
                a.record(stream)
                f()
                b.record(stream)
            torch.cuda.synchronize()
            cold = statistics.median(a.elapsed_time(b) for a, b in ev)
            res[algo] = {"warm_us": warm * 1e3, "cold_us": cold * 1e3,
                         "busbw_gbs_cold": busbw_gbs(size, cold * 1e-3, n),
                         "hbm_frac_cold": 2 * n * size / (cold * 1e-3) / 1e9 / peak}
        # per-call time inside a CUDA graph (launch overhead of the host gone), every order
        graph_us = {}
        reps = 100 if size <= (1 << 22) else 10
        for algo in ("fused", "tree", "ring", "step_ring", "step_tree"):
            g = torch.cuda.CUDAGraph()
            side = torch.cuda.Stream()
            side.wait_stream(stream)
            with torch.cuda.stream(side):
                g.capture_begin()
                for _ in range(reps):
                    if algo.startswith("step") and es == 2:
                        gar.ar_allreduce_stepwise(s_v, r_v, ws, op, algo, side)
                    else:
                        gar.ar_allreduce(s_v, r_v, op, algo, side)
                g.capture_end()
            stream.wait_stream(side)
            g.replay()
            graph_us[algo] = time_steps(g.replay, 3, stream) / reps * 1e3
            del g
        for algo, us in graph_us.items():
            fits.setdefault(algo, []).append((size, us))
        print(json.dumps({"workload": "size sweep", "nranks": n, "bytes_per_rank": size, "dtype": dtype, "op": op,
                          "in_l2": 2 * n * size <= l2, "graph_us": graph_us, **res}))
        sys.stdout.flush()
        size *= 2
    # alpha-beta model per order: t = alpha * launches + bytes / beta, least squares over the
    # sizes whose traffic exceeds L2 (bandwidth) and all sizes (latency)
    import numpy as np
    launches = {"fused": 1, "tree": 1, "ring": 2, "step_ring": 2 * (n - 1), "step_tree": 2 * int(math.log2(n))}
    traffic = {"fused": 2 * n, "tree": 2 * n, "ring": 2 * n + 1, "step_ring": 5 * (n - 1), "step_tree": 5 * (n - 1)}
    if es == 2:  # binary32 partials: bytes per call in units of M = 2 * count
        traffic["step_ring"] = stepwise16_traffic("step_ring", n)
        traffic["step_tree"] = stepwise16_traffic("step_tree", n)
    model = {}
    for algo, pts in fits.items():
        a = np.array([[launches[algo], traffic[algo] * m / 1e3] for m, _ in pts])  # us, (bytes/1e3) -> us at GB/s
        t = np.array([us for _, us in pts])
        (alpha, inv_beta), *_ = np.linalg.lstsq(a, t, rcond=None)
        model[algo] = {"alpha_us_per_launch": float(alpha), "beta_gbs": float(1.0 / inv_beta) if inv_beta > 0 else None,
                       "launches_per_call": launches[algo], "bytes_per_call": f"{traffic[algo]} x M"}
    best = {}
    for m in [1 << k for k in range(12, 31)]:
        pred = {al: v["alpha_us_per_launch"] * v["launches_per_call"] + traffic[al] * m / 1e3 / v["beta_gbs"]
                for al, v in model.items() if v["beta_gbs"]}
        best[m] = min(pred, key=pred.get)
    print(json.dumps({"workload": "alpha-beta fit", "nranks": n, "dtype": dtype, "op": op, "model": model,
                      "fastest_by_model": {str(k): v for k, v in best.items()}}))
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", choices=("bucket", "sweep", "fp8", "topk", "strong"), default="bucket")
    ap.add_argument("--fp8-count", type=int, default=134_217_728, help="elements per rank for --workload fp8")
    ap.add_argument("--sweep-max-bytes", type=int, default=1 << 30)
    ap.add_argument("--sweep-dtype", choices=("f32", "i32", "bf16"), default="f32",
                    help="f32 or bf16 uniform(-1,1), or int32 uniform[-2^20, 2^20] per rank")
    ap.add_argument("--sweep-op", choices=("sum", "min", "max"), default="sum")
    ap.add_argument("--cpu-budget", type=float, default=12.0, help="seconds of oracle time for cpu_baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--headline-only", action="store_true", help="skip the DDP, FP8 and Top-K rows")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)
    if args.workload == "sweep":
        return run_sweep(args)
    if args.workload == "strong":
        return run_strong(args)
    if args.workload == "fp8":
        import torch

        import gradient_allreduce_collective_gb300 as gar
        torch.cuda.set_device(dist_env()[2])
        gar.build()
        gar.lib()
        print(json.dumps(measure_fp8(gar, args.steps, args.warmup, args.fp8_count)))
        return 0
    if args.workload == "topk":
        import torch

        import gradient_allreduce_collective_gb300 as gar
        torch.cuda.set_device(dist_env()[2])
        gar.build()
        gar.lib()
        print(json.dumps(measure_topk(gar, args.steps, args.warmup, with_oracle=not args.no_cpu_baseline)))
        return 0
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
