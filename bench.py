"""Benchmark: one step = nbody_forces (a + p) + nbody_euler_step on N = 2^20
Plummer bodies (the headline workload), timed with CUDA events.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--config NAME] [--no-cpu-baseline] [--no-e2e] [--no-configs]

Prints one JSON line on rank 0.  `value` is interactions/s of the whole job
(N^2 pairs per step and GPU) with inputs resident in HBM; `e2e` is the same
metric through the C ABI with the step's inputs copied from pinned host
memory and its results copied back inside the timed region.  L2 is flushed
(a 256 MiB write) before every timed step, outside the step's events.

--impl reference times the oracle (fp64 CPU, all host cores) on a bounded
sample of the same workload: each step evaluates a fixed number of target
rows against all N sources.
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

METRIC = "interactions/s & GFLOP/s (20 flop/pair) at N=1M fp32, % of FP32/MUFU roofline"
FLOPS_PER_PAIR = 20           # the pages' pair count (bodyBodyInteraction annotation)
FP32_OPS_PER_PAIR = 13        # fp32 lane operations of the pair law for one ordered pair (a + p)
SYM_OPS_PER_PAIR = 18         # fp32 lane operations for one unordered pair, both bodies' a + p
FP32_LANES_PER_SM_CLK = 128
RECIPE_SM_MAX_MHZ = 2070.0    # fallback if no measured peaks file is present
PATH_CLUSTER = 2
PATH_SYMMETRIC = 3
PATH_ROWS = 4
PATH_NAMES = {1: "tiled", 2: "cluster", 3: "symmetric", 4: "rows"}
ACC_ONLY_WORKLOADS = {"disk4096"}   # configurations that check the acceleration only
PATH_IDS = {"auto": 0, "tiled": 1, "symmetric": 3}

# DRAM traffic (dram__bytes_read.sum + dram__bytes_write.sum) of the force
# kernel's launches in one force call at N = 2^20, from one ncu capture, keyed
# by a hash of the kernel's source files: a changed kernel reports null until
# it is re-measured.
KERNEL_SOURCES = {
    "tiled": ["all_pairs_gravitational_gb300/csrc/forces_tiled.cu",
              "all_pairs_gravitational_gb300/csrc/nbody_device.cuh"],
    "symmetric": ["all_pairs_gravitational_gb300/csrc/forces_sym.cu",
                  "all_pairs_gravitational_gb300/csrc/nbody_device.cuh"],
    "rows": ["all_pairs_gravitational_gb300/csrc/forces_rows.cu",
             "all_pairs_gravitational_gb300/csrc/nbody_device.cuh"],
    "cluster": ["all_pairs_gravitational_gb300/csrc/forces_cluster.cu",
                "all_pairs_gravitational_gb300/csrc/nbody_device.cuh"],
}
TRAFFIC_BY_SOURCE = {
    # one nbody_forces call = 7 passes of the symmetric kernel (default plan)
    "38e6a797d7d47b0e": {"bytes": 495.2e6 + 5738.4e6,
                         "profile": "profiles/forces_sym_plummer1048576_dram.md"},
}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", default="plummer1048576")
    ap.add_argument("--path", choices=["auto", "tiled", "symmetric"], default="auto",
                    help="force path of the timed step and e2e (auto: the library's choice)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-configs", "--no-small-n", dest="no_configs", action="store_true",
                    help="skip the per-workload table (every other configuration and the small-N "
                         "sweep, CUDA-graph-timed), the acceleration-only call and the Euler "
                         "HBM probe")
    ap.add_argument("--probe", choices=["euler", "configs"], default=None,
                    help="run one kernel probe alone and print its result (for profiling)")
    ap.add_argument("--cpu-seconds", type=float, default=10.0,
                    help="target seconds of oracle work for the CPU baseline sample")
    return ap.parse_args()


def kernel_source_hash(kind):
    """Hash of the kernel's source files with comments and blank space
    removed: a change of code changes it, a change of comments does not."""
    import hashlib
    import re
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES[kind]:
        with open(os.path.join(ROOT, rel)) as f:
            src = f.read()
        src = re.sub(r"/\*.*?\*/", " ", src, flags=re.S)
        src = re.sub(r"//[^\n]*", " ", src)
        h.update(" ".join(src.split()).encode())
    return h.hexdigest()[:16]


def euler_hbm_probe(apg, device, n=1 << 26, reps=5):
    """The Euler kernel at a size far beyond L2 (80 B per body, 5.4 GB per
    step at n = 2^26), L2 flushed before each timed launch: achieved HBM GB/s."""
    import torch
    pm = torch.rand((n, 4), device=device)
    vel = torch.rand((n, 4), device=device)
    acc = torch.rand((n, 4), device=device)
    flush = torch.empty(64 * 1024 * 1024, dtype=torch.float32, device=device)
    apg.nbody_euler_step(pm, vel, acc, 1e-6)
    ts = []
    for _ in range(reps):
        flush.zero_()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        apg.nbody_euler_step(pm, vel, acc, 1e-6)
        b.record()
        b.synchronize()
        ts.append(a.elapsed_time(b))
    ms = statistics.median(ts)
    del pm, vel, acc, flush
    torch.cuda.empty_cache()
    return {"n": n, "ms": ms, "bytes": 80 * n, "gbs": 80 * n / (ms / 1e3) / 1e9}


def force_roofline(plan, n, sm, sm_max_mhz, acc_only=False):
    """Arithmetic bound of the planned force kernel, in interactions/s.

    Ordered-pair kernels (tiled, cluster, row-split) execute 13 fp32 lane
    operations per interaction.  The symmetric kernel executes 18 per unordered pair, which
    serves two interactions, except on the nb diagonal blocks, which it
    evaluates one way (13 per ordered pair).  The bound is the FMA pipe's
    lane rate over the launch's lane operations, times its N^2 interactions."""
    lanes_per_s = sm * sm_max_mhz * 1e6 * FP32_LANES_PER_SM_CLK
    pairs = float(n) * float(n)
    ordered = FP32_OPS_PER_PAIR - (1 if acc_only else 0)
    unordered = SYM_OPS_PER_PAIR - (2 if acc_only else 0)
    if plan["path"] == PATH_SYMMETRIC:
        t = plan["threads"] * plan["i_per_thread"]
        nb = plan["num_iblocks"]
        last = n - (nb - 1) * t
        diag = float((nb - 1) * t * t + last * last)
        ops = unordered / 2.0 * (pairs - diag) + ordered * diag
        kind, kernel = "symmetric", "forces_sym_kernel (+ reduce_pass_kernel)"
    elif plan["path"] == PATH_ROWS:
        ops = ordered * pairs
        kind, kernel = "rows", "forces_rows_kernel"
    elif plan["path"] == PATH_CLUSTER:
        ops = ordered * pairs
        kind, kernel = "cluster", "forces_cluster_kernel"
    else:
        ops = ordered * pairs
        kind, kernel = "tiled", "forces_tiled_kernel (+ reduce_pass_kernel)"
    return {"peak": lanes_per_s * pairs / ops, "ops_per_interaction": ops / pairs,
            "kind": kind, "kernel": kernel,
            "ordered_pair_peak": lanes_per_s / ordered}


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return json.load(f), "MEASURED_PEAKS.json"
    return {}, "recipe fallback"


def cpu_model():
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True).stdout
        for line in out.splitlines():
            if line.startswith("Model name"):
                return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return "unknown"


def time_oracle(w, target_seconds, max_rows=None, threads=0):
    """Oracle interactions/s on a sample of target rows x all sources, sized to
    about target_seconds of work after a short calibration (threads = 0: all
    host cores)."""
    import oracle
    n = w.n
    cores = threads if threads > 0 else oracle.max_threads()
    probe = max(1, min(n, 8 * cores))
    oracle.forces(w.pos_mass, w.eps2, rows=range(min(n, cores)), threads=threads)   # wake the threads
    t0 = time.perf_counter()
    oracle.forces(w.pos_mass, w.eps2, rows=range(probe), threads=threads)
    dt = max(time.perf_counter() - t0, 1e-6)
    rows = int(max(probe, min(n, probe * target_seconds / dt)))
    if max_rows:
        rows = min(rows, max_rows)
    t0 = time.perf_counter()
    oracle.forces(w.pos_mass, w.eps2, rows=range(rows), threads=threads)
    el = time.perf_counter() - t0
    return {"value": rows * n / el, "unit": "interactions/s", "cores": cores,
            "kind": "oracle", "seconds": el,
            "sample": f"{rows} target rows x all {n} sources of {w.name} (fp64, OpenMP)",
            "cpu_model": cpu_model()}


class ClockSampler:
    """nvidia-smi samples (every 200 ms) while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu_index = gpu_index
        self.proc = None
        self.file = None

    def __enter__(self):
        try:
            self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu_index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=self.file, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if self.proc is None or self.file is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "note": "nvidia-smi unavailable"}
        self.file.flush()
        with open(self.file.name) as f:
            rows = [r.strip().split(", ") for r in f if r.strip()]
        os.unlink(self.file.name)
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        sm, smax, reasons = [], [], set()
        for r in rows:
            if len(r) < 9:
                continue
            try:
                sm.append(float(r[1]))
                smax.append(float(r[2]))
            except ValueError:
                continue
            for name, val in zip(names, r[5:9]):
                if val.strip().lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def physical_gpu_index(local):
    vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
    ids = [v.strip() for v in vis.split(",") if v.strip()]
    if local < len(ids) and ids[local].isdigit():
        return int(ids[local])
    return local


def dist_setup(args):
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        torch.cuda.set_device(0)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, world, device="cuda"):
    """The largest x over all ranks (the slowest rank's time)."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_value(total_pairs, step_ms):
    """Interactions/s of the whole job: the one N^2 problem the ranks share
    (each owns a range of targets) over the slowest rank's step."""
    return total_pairs / (step_ms / 1e3)


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    from all_pairs_gravitational_gb300 import workloads as W
    import oracle
    oracle.build()
    w = W.named(args.config)
    per_step = max(1.0, args.cpu_seconds / max(1, args.steps + args.warmup))
    # calibrate once, then every step evaluates the same row count
    cal = time_oracle(w, per_step)
    rows = int(cal["value"] * per_step / w.n) or 1
    rows = min(rows, w.n)
    for _ in range(args.warmup):
        oracle.forces(w.pos_mass, w.eps2, rows=range(rows))
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        oracle.forces(w.pos_mass, w.eps2, rows=range(rows))
        times.append(time.perf_counter() - t0)
    total = sum(times)
    value = rows * w.n * args.steps / total
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "interactions/s",
        "gflops_20": value * FLOPS_PER_PAIR / 1e9, "n_gpus": args.gpus, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps,
        "higher_is_better": True, "scaling": "strong", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": w.name, "n": w.n, "eps2": float(w.eps2),
                   "step": f"oracle forces for {rows} target rows x all {w.n} sources"},
        "cpu_baseline": {"value": value, "unit": "interactions/s", "cores": oracle.max_threads(),
                         "kind": "oracle",
                         "sample": f"{rows} target rows x all {w.n} sources per step",
                         "cpu_model": cpu_model()},
        "e2e": {"value": value, "unit": "interactions/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_ours(args):
    import numpy as np
    import torch

    import __graft_entry__
    __graft_entry__.build()
    import all_pairs_gravitational_gb300 as apg
    from all_pairs_gravitational_gb300 import workloads as W
    from all_pairs_gravitational_gb300.sharded import forces_sharded, shard_range

    world, rank, local = dist_setup(args)
    device = torch.device("cuda", local)
    props = torch.cuda.get_device_properties(device)
    w = W.named(args.config)
    n = w.n
    pairs = float(n) * float(n)
    path = PATH_IDS[args.path]
    plan = apg.nbody_plan_forces(n, props.multi_processor_count, path=path)
    # force launches (with a reduction after each when partials are used), then Euler
    launches_per_step = plan["passes"] * (2 if plan["scratch_bytes"] > 0 else 1) + 1

    # One GPU: the whole problem.  Several: rank r owns the targets
    # [lo, hi) and all-gathers every position each step (target sharding).
    lo, hi = shard_range(n, rank, world)
    pm = torch.from_numpy(w.pos_mass[lo:hi].copy()).to(device)
    vel = torch.from_numpy(w.vel[lo:hi].copy()).to(device)
    acc = torch.empty_like(pm)
    sources = torch.empty((n, 4), device=device) if world > 1 else None
    flush = torch.empty(64 * 1024 * 1024, dtype=torch.float32, device=device)   # 256 MiB > L2
    stream = torch.cuda.current_stream(device)
    eps2, dt = float(w.eps2), float(w.dt)
    if world > 1:
        # per rank: the ordered-pair tiled kernel on hi - lo targets x n sources
        plan = {"path": 1}
        launches_per_step = None

    def forces():
        if world > 1:
            forces_sharded(pm, n, eps2, acc, sources=sources)
        else:
            apg.nbody_forces_ex(pm, eps2, acc, path=path)

    def step():
        forces()
        apg.nbody_euler_step(pm, vel, acc, dt)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()

    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True),
           torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    sampler = ClockSampler(physical_gpu_index(local))
    barrier(world)
    torch.cuda.synchronize()
    with sampler:
        t_wall = time.perf_counter()
        for k in range(args.steps):
            flush.zero_()
            ev[k][0].record(stream)
            forces()
            ev[k][1].record(stream)
            apg.nbody_euler_step(pm, vel, acc, dt)
            ev[k][2].record(stream)
        torch.cuda.synchronize()
        t_wall = time.perf_counter() - t_wall
    barrier(world)
    forces_ms = [a.elapsed_time(b) for a, b, _ in ev]
    euler_ms = [b.elapsed_time(c) for _, b, c in ev]
    step_ms = sum(forces_ms + euler_ms) / args.steps
    step_ms = max_over_ranks(step_ms, world)
    clocks = sampler.summary()

    peaks, peaks_src = measured_peaks()
    sm_max = float(peaks.get("sm_max_mhz", RECIPE_SM_MAX_MHZ))
    roof = force_roofline(plan, n, props.multi_processor_count, sm_max)
    peak_pairs = roof["peak"]
    forces_s = statistics.mean(forces_ms) / 1e3
    achieved = float(hi - lo) * n / forces_s          # this rank's interactions
    euler_s = statistics.mean(euler_ms) / 1e3
    hbm = float(peaks.get("hbm_gbs", 6800.0))

    # interactions of the whole job over the slowest rank's step: every rank's
    # N^2 for independent replicas would be weak scaling; here the ranks
    # share one N^2 problem (strong scaling)
    value = whole_job_value(pairs, step_ms)

    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(apg, w, device, args.steps, world, path, (lo, hi))

    cpu = None
    if not args.no_cpu_baseline and rank == 0 and world == 1:
        cpu = time_oracle(w, args.cpu_seconds)
        # the whole evaluation on the host cores, extrapolated from the sample
        cpu["extrapolated_full_n_seconds"] = float(n) * n / cpu["value"]
        cpu["extrapolated_note"] = ("extrapolated: N^2 interactions at the sampled rate; "
                                    "the full oracle evaluation is not run by the benchmark")

    configs = acc_only = euler_hbm = None
    if not args.no_configs and world == 1:   # single-GPU figures; a scaling run skips them
        names = [c for c in W.CONFIG_NAMES if c != w.name] + [f"smallcube{k}" for k in W.SMALL_SWEEP]
        cpu_on = not args.no_cpu_baseline and rank == 0 and world == 1
        configs = configs_probe(apg, W, device, cpu_seconds=0.5 if cpu_on else 0,
                                cpu1_seconds=0.3 if cpu_on else 0, names=names)
        acc_only = acc_only_probe(apg, w, device, plan, props.multi_processor_count, sm_max)
        euler_hbm = euler_hbm_probe(apg, device)
    src_hash = kernel_source_hash(roof["kind"])
    traffic = TRAFFIC_BY_SOURCE.get(src_hash) if w.name == "plummer1048576" else None

    sm_at_clock = clocks.get("sm_mhz")
    line = {
        "metric": METRIC,
        "value": value,
        "unit": "interactions/s",
        "gflops_20": value * FLOPS_PER_PAIR / 1e9,
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": step_ms,
        "higher_is_better": True,
        "scaling": "strong",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": w.name, "n": n, "eps2": eps2, "dt": dt,
                   "step": "nbody_forces (a + p) then nbody_euler_step",
                   "path": args.path,
                   "l2": "flushed (256 MiB write) before each timed step, outside its events",
                   "parallelism": (f"target-sharded over {world} GPUs (all-gather of positions, "
                                   "nbody_forces_ts per rank)") if world > 1 else "single GPU",
                   "plan": {k: plan[k] for k in ("path", "variant", "i_per_thread", "threads",
                                                 "tile", "num_iblocks", "splits", "dists",
                                                 "groups", "passes", "grid", "scratch_bytes",
                                                 "fill")}},
        "roofline": {
            "bound": "alu",
            "achieved": achieved,
            "peak": peak_pairs,
            "unit": "interactions/s",
            "frac": achieved / peak_pairs,
            "traffic": traffic["bytes"] if traffic else None,
            "traffic_source": (traffic["profile"] if traffic else
                               f"not measured for kernel source {src_hash}"),
            "kernel": roof["kernel"],
            "peak_basis": (f"{props.multi_processor_count} SMs x {sm_max:.0f} MHz ({peaks_src}) x "
                           f"{FP32_LANES_PER_SM_CLK} fp32 lanes / "
                           f"{roof['ops_per_interaction']:.4f} fp32 ops per interaction"
                           + (f" ({SYM_OPS_PER_PAIR} per unordered pair for both bodies, "
                              f"{FP32_OPS_PER_PAIR} per ordered pair on the diagonal blocks)"
                              if roof["kind"] == "symmetric" else "")),
            "frac_of_ordered_pair_bound": achieved / roof["ordered_pair_peak"],
            "frac_at_sampled_clock": (achieved / (peak_pairs * sm_at_clock / sm_max)
                                      if sm_at_clock else None),
            "forces_ms": statistics.mean(forces_ms),
            "gflops_20": achieved * FLOPS_PER_PAIR / 1e9,
        },
        "euler": {"ms": statistics.mean(euler_ms), "bytes": 80 * n,
                  "gbs": 80 * n / euler_s / 1e9, "hbm_peak_gbs": hbm,
                  "note": "in-step figure; the 84 MB may be L2-resident at this size",
                  "hbm_probe": (dict(euler_hbm, hbm_peak_gbs=hbm, frac=euler_hbm["gbs"] / hbm,
                                     bound="hbm", peak_source=peaks_src)
                                if euler_hbm else None)},
        "cpu_baseline": cpu,
        "configs": configs,
        "acc_only": acc_only,
        "e2e": e2e,
        "gpu_launches": (launches_per_step * args.steps if launches_per_step is not None
                         else 3 * args.steps),
        "clocks": clocks,
        "wall_s_timed_loop": t_wall,
        "device": props.name,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def run_e2e(apg, w, device, steps, world, path=0, rows=None):
    """Same metric through the public API from host buffers: per step, copy
    this rank's bodies and velocities in from pinned memory, compute (on
    several GPUs: the target-sharded step with its all-gather), copy the new
    state and the accelerations/potentials back."""
    import torch
    from all_pairs_gravitational_gb300.sharded import forces_sharded
    n = w.n
    lo, hi = rows if rows is not None else (0, n)
    m = hi - lo
    h_pm = torch.from_numpy(w.pos_mass[lo:hi].copy()).pin_memory()
    h_vel = torch.from_numpy(w.vel[lo:hi].copy()).pin_memory()
    h_out = [torch.empty((m, 4), dtype=torch.float32).pin_memory() for _ in range(3)]
    d_pm = torch.empty((m, 4), device=device)
    d_vel = torch.empty_like(d_pm)
    d_acc = torch.empty_like(d_pm)
    sources = torch.empty((n, 4), device=device) if world > 1 else None
    stream = torch.cuda.current_stream(device)
    eps2, dt = float(w.eps2), float(w.dt)

    def one():
        d_pm.copy_(h_pm, non_blocking=True)
        d_vel.copy_(h_vel, non_blocking=True)
        if world > 1:
            forces_sharded(d_pm, n, eps2, d_acc, sources=sources)
        else:
            apg.nbody_forces_ex(d_pm, eps2, d_acc, path=path)
        apg.nbody_euler_step(d_pm, d_vel, d_acc, dt)
        h_out[0].copy_(d_pm, non_blocking=True)
        h_out[1].copy_(d_vel, non_blocking=True)
        h_out[2].copy_(d_acc, non_blocking=True)

    one()
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for _ in range(steps):
        one()
    end.record(stream)
    end.synchronize()
    ms = start.elapsed_time(end) / steps
    ms = max_over_ranks(ms, world)
    return {"value": float(n) * n / (ms / 1e3), "unit": "interactions/s",
            "h2d_bytes_per_step": 32 * m, "d2h_bytes_per_step": 48 * m, "ms_per_step": ms}


def graph_time_ms(fn, reps):
    """Per-call time of fn replayed `reps` times from one CUDA graph (best of 5)."""
    import torch
    fn()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for _ in range(reps):
            fn()
    g.replay()
    torch.cuda.synchronize()
    best = None
    for _ in range(5):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        g.replay()
        b.record()
        b.synchronize()
        t = a.elapsed_time(b) / reps
        best = t if best is None else min(best, t)
    return best


def configs_probe(apg, W, device, cpu_seconds=1.5, cpu1_seconds=0.5, names=None):
    """Every measured workload: the force call alone (replayed from a CUDA
    graph, so host launch overhead is excluded), one nbody_simulate step, the
    fraction of the planned kernel's fp32-pipe bound and of the ordered-pair
    bound, and the oracle on a sample of rows (all host cores, and one core
    for n <= 16384)."""
    import torch
    props = torch.cuda.get_device_properties(device)
    peaks, _ = measured_peaks()
    sm_max = float(peaks.get("sm_max_mhz", RECIPE_SM_MAX_MHZ))
    out = []
    if names is None:
        names = W.CONFIG_NAMES + [f"smallcube{n}" for n in W.SMALL_SWEEP]
    for name in names:
        w = W.named(name)
        n = w.n
        pm = torch.from_numpy(w.pos_mass).to(device)
        vel = torch.from_numpy(w.vel).to(device)
        acc = torch.empty_like(pm)
        eps2, dt = float(w.eps2), float(w.dt)
        reps = max(1, min(50, int(2e10 / (float(n) * n))))
        # the disk workload is evaluated for the acceleration only
        acc_only = name in ACC_ONLY_WORKLOADS
        call = apg.nbody_forces_acc if acc_only else apg.nbody_forces
        ms = graph_time_ms(lambda: call(pm, eps2, acc), reps)
        steps = max(1, min(100, int(1e11 / (float(n) * n))))
        apg.nbody_simulate(pm, vel, acc, eps2, dt, steps)
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        apg.nbody_simulate(pm, vel, acc, eps2, dt, steps)
        b.record()
        b.synchronize()
        step_ms = a.elapsed_time(b) / steps
        plan = apg.nbody_plan_forces(n, props.multi_processor_count)
        roof = force_roofline(plan, n, props.multi_processor_count, sm_max, acc_only=acc_only)
        rate = float(n) * n / (ms / 1e3)
        cpu = time_oracle(w, cpu_seconds) if cpu_seconds > 0 else None
        cpu1 = (time_oracle(w, cpu1_seconds, threads=1)
                if cpu1_seconds > 0 and n <= 16384 else None)
        out.append({"workload": name, "n": n, "call": call.__name__, "forces_ms": ms,
                    "interactions_per_s": rate,
                    "gflops_20": rate * FLOPS_PER_PAIR / 1e9, "frac_fp32_peak": rate / roof["peak"],
                    "frac_of_ordered_pair_bound": rate / roof["ordered_pair_peak"],
                    "simulate_step_ms": step_ms,
                    "path": PATH_NAMES[plan["path"]],
                    "splits": plan["splits"], "passes": plan["passes"],
                    "scratch_bytes": plan["scratch_bytes"],
                    "cpu_oracle_interactions_per_s": cpu["value"] if cpu else None,
                    "cpu_cores": cpu["cores"] if cpu else None,
                    "cpu_oracle_1thread_interactions_per_s": cpu1["value"] if cpu1 else None})
        del pm, vel, acc
    return out


def acc_only_probe(apg, w, device, plan, sm, sm_max, reps=2):
    """nbody_forces_acc on the headline workload: CUDA-event time of the
    call, against the acceleration-only bound (16 fp32 lane operations per
    unordered pair, 12 per ordered pair on the diagonal blocks)."""
    import torch
    pm = torch.from_numpy(w.pos_mass).to(device)
    acc = torch.empty_like(pm)
    apg.nbody_forces_acc(pm, float(w.eps2), acc)
    ts = []
    for _ in range(reps):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        apg.nbody_forces_acc(pm, float(w.eps2), acc)
        b.record()
        b.synchronize()
        ts.append(a.elapsed_time(b))
    ms = statistics.mean(ts)
    roof = force_roofline(plan, w.n, sm, sm_max, acc_only=True)
    rate = float(w.n) * w.n / (ms / 1e3)
    return {"call": "nbody_forces_acc", "forces_ms": ms, "interactions_per_s": rate,
            "peak": roof["peak"], "frac": rate / roof["peak"],
            "ops_per_interaction": roof["ops_per_interaction"], "runs": reps}


def run_probe(args):
    import torch

    import __graft_entry__
    __graft_entry__.build()
    import all_pairs_gravitational_gb300 as apg
    from all_pairs_gravitational_gb300 import workloads as W
    torch.cuda.set_device(0)
    device = torch.device("cuda", 0)
    peaks, src = measured_peaks()
    if args.probe == "euler":
        r = euler_hbm_probe(apg, device)
        r.update(probe="euler_kernel", hbm_peak_gbs=float(peaks.get("hbm_gbs", 6800.0)),
                 peak_source=src)
        r["frac"] = r["gbs"] / r["hbm_peak_gbs"]
        print(json.dumps(r), flush=True)
    else:
        for r in configs_probe(apg, W, device):
            print(json.dumps(r), flush=True)


def main():
    args = parse()
    if args.probe:
        run_probe(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
