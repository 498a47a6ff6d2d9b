#!/usr/bin/env python3
"""Benchmark of the fused ZeRO flat-parameter step on GB300.

One "step" is one pass of the whole hot path over one batch of gradients:
reduce_grads (registration of the N replica gradients) -> zero_step (the fused
rank-order fp32 reduce, Adam, bf16 cast) -> gather_weights (ZeRO-3 per-unit
copies; nothing to do for stages 0-2) -> post_step.

Default workload: Llama-style model, hidden 1024, intermediate 2048, 16/4
heads, 8 layers, vocab 1024 (73,417,728 params) flattened into one
FlatParameter, N = 8 simulated ranks, ZeRO-2, bf16 gradients ~N(0, 1e-3),
fp32 Adam.  Every step moves (2N + 26) B/param = 3.08 GB, well above the
129 MB L2, so no flush is needed between steps.

Prints ONE JSON line (rank 0).  ``--impl reference`` times the CPU oracle on
the host instead (a bounded sample of the same workload).
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "fused ZeRO step params/s and achieved HBM GB/s (% of GB300 peak), 1 GPU"
UNIT = "params/s"
FALLBACK_HBM_GBS = 6800.0


# ---------------------------------------------------------------------------
# Workloads.
# ---------------------------------------------------------------------------
def workload(name: str):
    import synth_inputs as si
    if name == "llama1024_zero2_n8":
        return dict(pl=si.llama_1024(), n=8, stage=2, grad_dtype="bf16", grad_std=1e-3, per_unit=False,
                    outliers=0.0)
    if name == "llama2048_zero3_n8":
        return dict(pl=si.llama_2048_units(), n=8, stage=3, grad_dtype="bf16", grad_std=1e-3, per_unit=True,
                    outliers=0.0)
    if name == "stage_buffer_zero1_fp32_n2":
        return dict(pl=si.llama_2048_stage_buffer(), n=2, stage=1, grad_dtype="fp32", grad_std=1e-3,
                    per_unit=False, outliers=0.0)
    if name == "toy_mlp_n4":
        return dict(pl=si.toy_mlp(), n=4, stage=2, grad_dtype="bf16", grad_std=1e-2, per_unit=True, outliers=0.0)
    if name.startswith("flat32:"):  # one flat buffer, fp32 replica gradients, ZeRO-1 (the stage-buffer case, any size)
        _, numel, n = name.split(":")
        return dict(pl=si.single_buffer(int(float(numel))), n=int(n), stage=1, grad_dtype="fp32", grad_std=1e-3,
                    per_unit=False, outliers=0.0)
    if name.startswith("units3:"):  # ZeRO-3 over equal units with per-unit gathers
        _, units, numel, n = name.split(":")
        return dict(pl=si.from_units([int(float(numel))] * int(units)), n=int(n), stage=3, grad_dtype="bf16",
                    grad_std=1e-3, per_unit=True, outliers=0.0)
    if name.startswith("flat:"):
        _, numel, n = name.split(":")
        return dict(pl=si.single_buffer(int(float(numel))), n=int(n), stage=2, grad_dtype="bf16", grad_std=1e-2,
                    per_unit=False, outliers=0.001)
    raise SystemExit(f"unknown workload {name}")


def bytes_per_param(n: int, grad_dtype: str) -> int:
    """Algorithmic bytes per (padded) element of one fused step: N replica
    gradient reads + master/m/v read (12) + master/m/v write (12) + bf16 write (2)."""
    return (2 if grad_dtype == "bf16" else 4) * n + 26


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def step_kernel_name(n: int, grad_dtype: str, clip_keep: bool, elems: int) -> str:
    """The step kernel the library launches for this workload: over >= 2^23
    elements the tile-staged one with 2,048-element tiles for N >= 11 bf16 or
    N = 8, 9 fp32 replicas and the one with 4 elements per thread for N = 7
    or N >= 10 fp32 or N = 1..4 bf16 replicas; the register-staged one
    otherwise (a kept
    fp32 reduced gradient is one fp32 replica)."""
    if clip_keep:
        n, grad_dtype = 1, "fp32"
    if elems < 2 ** 23:
        return "step_vec_kernel"
    if grad_dtype == "bf16":
        if n <= 4:
            return "step_tma4_kernel"
        return "step_tma_kernel" if n >= 11 else "step_vec_kernel"
    if n >= 10 or n == 7:
        return "step_tma4_kernel"
    return "step_tma_kernel" if n in (8, 9) else "step_vec_kernel"


def kernel_source_sha() -> str:
    """Hash of the step kernel's sources (the kernel whose traffic is recorded)."""
    h = hashlib.sha256()
    for rel in ("zero_sharded_mixed_flatparameter_gb300/csrc/zero_step_kernels.cu",
                "zero_sharded_mixed_flatparameter_gb300/csrc/zero_device.cuh",
                "zero_sharded_mixed_flatparameter_gb300/csrc/zero_internal.h"):
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(workload_name: str):
    """DRAM bytes per launch of the step kernel from the committed ncu summary,
    if it was taken on the current kernel source; else None."""
    path = os.path.join(ROOT, "profiles", "step_kernel_dram_traffic.txt")
    if not os.path.exists(path):
        return None
    sha = kernel_source_sha()
    for line in open(path):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        fields = dict(kv.split("=", 1) for kv in line.split() if "=" in kv)
        if fields.get("workload") == workload_name and fields.get("kernel_sha") == sha:
            return float(fields["dram_bytes_per_launch"])
    return None


# ---------------------------------------------------------------------------
# Clock sampling during the timed region.
# ---------------------------------------------------------------------------
class ClockSampler:
    """nvidia-smi samples (every 50 ms) of SM clock, power and throttle
    reasons; summary() keeps the samples taken inside the timed window."""
    QUERY = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.device_index = device_index
        self.proc = None
        self.file = None
        self.window = None

    def __enter__(self):
        try:
            self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.device_index), f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=self.file, stderr=subprocess.DEVNULL)
            time.sleep(0.5)
        except Exception:
            self.proc = None
        return self

    def mark(self, t_start: float, t_end: float):
        self.window = (t_start, t_end)

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.1)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        if self.proc is None or self.file is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        import datetime
        self.file.flush()
        rows = []
        with open(self.file.name) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    try:
                        ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                    except ValueError:
                        continue
                    rows.append([ts] + parts[1:])
        os.unlink(self.file.name)

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        inside = rows
        if self.window and rows:
            lo, hi = self.window
            inside = [r for r in rows if lo - 0.05 <= r[0] <= hi + 0.05]
        if not inside:
            # the timed region was shorter than the sampling interval: take the
            # sample nearest to its middle
            if not rows:
                return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
            mid = sum(self.window) / 2 if self.window else rows[-1][0]
            inside = [min(rows, key=lambda r: abs(r[0] - mid))]
        sm = [num(r[1]) for r in inside if num(r[1]) is not None]
        mx = [num(r[2]) for r in inside if num(r[2]) is not None]
        power = [num(r[3]) for r in inside if num(r[3]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[k] for r in inside for k in range(4) if str(r[5 + k]).lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "power_w_median": statistics.median(power) if power else None,
                "samples_in_timed_region": len(inside), "reasons": reasons}


# ---------------------------------------------------------------------------
# Distributed plumbing (replicas only: ranks run independent copies).
# ---------------------------------------------------------------------------
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def aggregate(values, op: str, world: int, device):
    """max / sum of a list of floats over ranks (identity at world 1)."""
    if world == 1:
        return list(values)
    import torch
    import torch.distributed as dist
    t = torch.tensor(values, dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX if op == "max" else dist.ReduceOp.SUM)
    return t.tolist()


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ---------------------------------------------------------------------------
# CPU baseline: the oracle on a bounded sample of the workload.
# ---------------------------------------------------------------------------
class OracleSample:
    """The oracle's literal per-rank ZeRO step on a contiguous window of the
    workload: one unit of ``sample_params`` elements with the workload's N,
    stage, gradient dtype and value distributions (inputs drawn once)."""

    def __init__(self, wl, sample_params: int, seed: int = 7):
        import oracle
        import synth_inputs as si
        self.oracle = oracle
        self.n, self.stage, gd = wl["n"], max(wl["stage"], 1), wl["grad_dtype"]
        self.sample_params = sample_params
        self.lay = oracle.layout([sample_params], [0], self.n, self.stage)
        init = si.normal_fp32(sample_params, 0.02, seed).numpy()
        self.state = oracle.make_master([sample_params], self.lay, [init])
        self.grads = [si.as_numpy_bits(t) for t in
                      si.replica_grads(self.n, self.lay.total_padded, wl["grad_std"], seed + 1, gd,
                                       outlier_fraction=wl["outliers"])]
        self.hyper = oracle.Hyper(n_ranks=self.n, grad_dtype=gd)
        self.t = 0

    def step(self):
        self.t += 1
        master, m, v, p16 = self.state
        self.oracle.zero_step(self.hyper, self.stage, self.t, self.lay, self.grads, master, m, v, p16)


def cpu_baseline(wl, sample_params: int = 4_000_000, min_seconds: float = 10.0):
    sample = OracleSample(wl, sample_params)
    steps, t0 = 0, time.perf_counter()
    while True:
        sample.step()
        steps += 1
        dt = time.perf_counter() - t0
        if dt >= min_seconds:
            break
    value = sample_params * steps / dt
    return {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
            "host_cores_total": os.cpu_count(),
            "sample": (f"{steps} literal per-rank oracle steps on a contiguous {sample_params:,}-param window "
                       f"of the workload (N={wl['n']}, {wl['grad_dtype']} grads), {dt:.1f} s single-threaded")}


def cpu_adam_baseline(sample_params: int = 16_000_000, min_seconds: float = 3.0):
    """The library's ZeRO-Offload CPU Adam (zero_cpu_adam) on host arrays, all
    host cores: the second, optimised CPU baseline."""
    import ctypes
    import numpy as np
    from zero_sharded_mixed_flatparameter_gb300 import binding as B
    rng = np.random.default_rng(7)
    g = rng.normal(0, 1e-3, sample_params).astype(np.float32)
    w = rng.normal(0, 0.02, sample_params).astype(np.float32)
    m, v = np.zeros_like(w), np.zeros_like(w)
    p16 = np.zeros(sample_params, np.uint16)
    ptr = [a.ctypes.data_as(ctypes.c_void_p).value for a in (g, w, m, v, p16)]
    cfg = B.make_config(2, 1, "fp32")
    threads = os.cpu_count() or 1
    B.zero_cpu_adam(cfg, 1, *ptr, sample_params, threads)  # first touch, warm-up
    steps, t0 = 0, time.perf_counter()
    while True:
        B.zero_cpu_adam(cfg, steps + 2, *ptr, sample_params, threads)
        steps += 1
        dt = time.perf_counter() - t0
        if dt >= min_seconds:
            break
    value = sample_params * steps / dt
    return {"value": value, "unit": UNIT, "cores": threads, "kind": "library host Adam (zero_cpu_adam)",
            "host_gbs": value * 30 / 1e9,
            "sample": (f"{steps} host Adam steps over {sample_params:,} params (fp32 grad, master, m, v; bf16 out: "
                       f"30 B/param of host memory traffic), {dt:.1f} s on {threads} threads")}


def host_copy_gbs(n: int = 128 * 1024 * 1024, reps: int = 5) -> float:
    """Host memory copy bandwidth (bytes read + written) with torch's CPU threads."""
    import torch
    a = torch.ones(n, dtype=torch.float32)
    b = torch.empty_like(a)
    b.copy_(a)
    best = 0.0
    for _ in range(reps):
        t0 = time.perf_counter()
        b.copy_(a)
        best = max(best, 8 * n / (time.perf_counter() - t0) / 1e9)
    return best


# ---------------------------------------------------------------------------
# Our arm.
# ---------------------------------------------------------------------------
def run_ours(args):
    import torch
    import synth_inputs as si
    from zero_sharded_mixed_flatparameter_gb300 import build_lib
    from zero_sharded_mixed_flatparameter_gb300.runner import FlatStep

    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    device = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(device)
    if rank == 0:
        build_lib.build()
    barrier(world)
    wl = workload(args.workload)
    pl, n = wl["pl"], wl["n"]

    init_flat = si.normal_fp32(pl.total, 0.02, 1 + rank, device=device)
    offs = [0]
    for k in pl.numel:
        offs.append(offs[-1] + k)
    init = [init_flat[offs[p]:offs[p + 1]] for p in range(len(pl.numel))]
    offload_kw = {}
    if args.offload:
        offload_kw = dict(offload=True, offload_chunk=args.offload_chunk, offload_threads=args.offload_threads)
    fs = FlatStep(pl.numel, pl.unit, stage=wl["stage"], n_ranks=n, grad_dtype=wl["grad_dtype"], init_params=init,
                  device=device, **offload_kw)
    del init, init_flat
    padded = fs.padded
    grads = si.replica_grads(n, padded, wl["grad_std"], 100 + rank, wl["grad_dtype"], device=device,
                             outlier_fraction=wl["outliers"])
    units = [fs.layout(i) for i in range(fs.n_units)]
    micro = []
    if args.accum > 0:
        if wl["grad_dtype"] != "fp32":
            raise SystemExit("--accum needs an fp32-gradient workload (the accumulators are the step's gradients)")
        micro = si.replica_grads(n, padded, wl["grad_std"], 200 + rank, "bf16", device=device)
    gather_bufs = []
    if wl["stage"] == 3:
        gather_bufs = [torch.empty(max(u[1], 1), dtype=torch.bfloat16, device=device) for u in units]
    stream = torch.cuda.current_stream(device)

    def one_step(ev_pair=None, clip_pair=None, accum_pair=None, gather_pair=None):
        launches = 0
        if micro:
            if accum_pair is not None:
                accum_pair[0].record(stream)
            for k in range(args.accum):
                fs.accumulate_grads(-1, micro, grads, first=(k == 0))
                launches += fs.last_launches()
            if accum_pair is not None:
                accum_pair[1].record(stream)
        if wl["per_unit"]:
            for i, (numel, pad, shard, base) in enumerate(units):
                fs.reduce_grads(i, [g[base:base + pad] for g in grads])
        else:
            fs.reduce_grads(-1, grads)
        if args.clip > 0:
            if clip_pair is not None:
                clip_pair[0].record(stream)
            fs.clip_grad_norm(args.clip, keep_reduced=args.clip_keep)
            if clip_pair is not None:
                clip_pair[1].record(stream)
            launches += fs.last_launches()
        if ev_pair is not None:
            ev_pair[0].record(stream)
        fs.step()
        if ev_pair is not None:
            ev_pair[1].record(stream)
        launches += fs.last_launches()
        if gather_pair is not None and gather_bufs:
            gather_pair[0].record(stream)
        for i, buf in enumerate(gather_bufs):
            fs.gather_weights(i, buf)
            launches += fs.last_launches()
        if gather_pair is not None and gather_bufs:
            gather_pair[1].record(stream)
        fs.post_step()
        return launches

    # Warm-up: W steps, extended until at least 0.3 s of device work has run so
    # that clocks have ramped before the timed region (the count is reported).
    warm_done, t_warm = 0, time.perf_counter()
    while warm_done < args.warmup or time.perf_counter() - t_warm < 0.3:
        one_step()
        warm_done += 1
        if warm_done % 16 == 0:
            torch.cuda.synchronize(device)
    torch.cuda.synchronize(device)

    # --graph: the step (registration, clip, step, gathers, post_step) is
    # captured once into a CUDA graph in the library's capturable mode and
    # the timed region replays it; one eager capturable step first caches
    # the launch shapes.
    graph, graph_launches = None, 0
    if args.graph:
        fs.enable_capturable(max_steps=warm_done + args.steps + 2)
        graph_launches = one_step()
        torch.cuda.synchronize(device)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            one_step()
        torch.cuda.synchronize(device)

    # ---- device-resident timed region ----
    pairs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    clip_pairs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                  for _ in range(args.steps)] if args.clip > 0 else [None] * args.steps
    accum_pairs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                   for _ in range(args.steps)] if args.accum > 0 else [None] * args.steps
    gather_pairs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                    for _ in range(args.steps)] if gather_bufs else [None] * args.steps
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    launches = 0
    with ClockSampler(device.index if device.index is not None else 0) as clocks:
        barrier(world)
        torch.cuda.synchronize(device)
        t_region0 = time.time()
        start.record(stream)
        for k in range(args.steps):
            if graph is not None:
                pairs[k][0].record(stream)
                graph.replay()
                pairs[k][1].record(stream)
                launches += graph_launches
            else:
                launches += one_step(pairs[k], clip_pairs[k], accum_pairs[k], gather_pairs[k])
        end.record(stream)
        torch.cuda.synchronize(device)
        t_region1 = time.time()
        barrier(world)
        clocks.mark(t_region0, t_region1)
    total_ms = start.elapsed_time(end)
    step_kernel_ms = [a.elapsed_time(b) for a, b in pairs]
    clip_ms = [a.elapsed_time(b) for a, b in clip_pairs] if args.clip > 0 and graph is None else None
    accum_ms = [a.elapsed_time(b) for a, b in accum_pairs] if args.accum > 0 and graph is None else None
    gather_ms = [a.elapsed_time(b) for a, b in gather_pairs] if gather_bufs and graph is None else None
    if graph is not None:
        fs.disable_capturable()  # the end-to-end leg below runs eagerly
        del graph
    clock = clocks.summary()

    total_ms_max, kern_ms_max = aggregate([total_ms, statistics.mean(step_kernel_ms)], "max", world, device)
    params_all = aggregate([float(pl.total * args.steps)], "sum", world, device)[0]
    value = params_all / (total_ms_max / 1e3)

    # with the kept reduced gradient the step reads one fp32 gradient (4 B)
    bpp = 4 + 26 if (args.clip > 0 and args.clip_keep) else bytes_per_param(n, wl["grad_dtype"])
    bytes_per_launch = bpp * padded
    achieved_gbs = bytes_per_launch / (kern_ms_max / 1e3) / 1e9
    peak, peak_kind = measured_peaks()
    traffic = recorded_traffic(args.workload)

    # ---- end to end through the public API with host buffers ----
    # Every step copies its N replica gradients from pinned host memory and
    # reads the updated bf16 parameters back.  The host link (not HBM) bounds
    # this, so the copies are pipelined: step k+1's gradients travel on a copy
    # stream into the second of two device buffer sets while step k runs and
    # its parameters are read back on the compute stream.
    e2e = None
    if not args.no_e2e and not args.offload:
        host_grads = [g.to("cpu").pin_memory() for g in grads]
        host_out = torch.empty(padded, dtype=torch.bfloat16).pin_memory()
        bufs = [grads, [torch.empty_like(g) for g in grads]]
        copy_stream = torch.cuda.Stream(device)
        h2d_done = [torch.cuda.Event(), torch.cuda.Event()]
        step_done = [torch.cuda.Event(), torch.cuda.Event()]

        def e2e_run(steps):
            with torch.cuda.stream(copy_stream):
                for hg, g in zip(host_grads, bufs[0]):
                    g.copy_(hg, non_blocking=True)
                h2d_done[0].record(copy_stream)
            for k in range(steps):
                cur, nxt = k % 2, (k + 1) % 2
                if k + 1 < steps:
                    with torch.cuda.stream(copy_stream):
                        if k >= 1:
                            copy_stream.wait_event(step_done[nxt])
                        for hg, g in zip(host_grads, bufs[nxt]):
                            g.copy_(hg, non_blocking=True)
                        h2d_done[nxt].record(copy_stream)
                stream.wait_event(h2d_done[cur])
                if wl["per_unit"]:
                    for i, (numel, pad, shard, base) in enumerate(units):
                        fs.reduce_grads(i, [g[base:base + pad] for g in bufs[cur]])
                else:
                    fs.reduce_grads(-1, bufs[cur])
                fs.step()
                for i, buf in enumerate(gather_bufs):
                    fs.gather_weights(i, buf)
                fs.post_step()
                step_done[cur].record(stream)
                host_out.copy_(fs.param16, non_blocking=True)

        e2e_run(min(args.warmup, 3) + 1)
        torch.cuda.synchronize(device)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier(world)
        torch.cuda.synchronize(device)
        e0.record(stream)
        e2e_run(args.steps)
        e1.record(stream)
        torch.cuda.synchronize(device)
        barrier(world)
        e2e_ms = aggregate([e0.elapsed_time(e1)], "max", world, device)[0]
        esz = 2 if wl["grad_dtype"] == "bf16" else 4
        e2e = {"value": params_all / (e2e_ms / 1e3), "unit": UNIT,
               "h2d_bytes_per_step": n * padded * esz, "d2h_bytes_per_step": padded * 2,
               "ms_per_step": e2e_ms / args.steps,
               "pipelining": "double-buffered: step k+1's H2D overlaps step k and its D2H"}
        del host_grads, host_out, bufs

    fs.close()
    del grads
    torch.cuda.empty_cache()

    cpu = cpu_adam = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(wl)
        cpu_adam = cpu_adam_baseline()

    roofline = {"bound": "hbm", "achieved": achieved_gbs, "peak": peak, "unit": "GB/s",
                "frac": achieved_gbs / peak, "peak_source": f"hbm_gbs {peak_kind}",
                "traffic": traffic, "algorithmic_bytes_per_launch": bytes_per_launch,
                "bytes_per_param": bpp, "kernel": step_kernel_name(n, wl["grad_dtype"], args.clip_keep, padded),
                "kernel_ms_mean": kern_ms_max, "kernel_ms_min": min(step_kernel_ms),
                "timed": "whole replayed step (CUDA graph)" if args.graph else "step kernel launch"}
    offload = None
    if args.offload:
        # The offloaded step is bound by host memory: the host Adam moves
        # 30 B/param (fp32 grad, master, m, v read; master, m, v, bf16 written)
        # and the copies another 6 (the fp32 gradient written by the D2H copy,
        # the bf16 parameters read by the H2D copy), against the host's own copy
        # bandwidth.  The link carries 4 B/param down and 2 B/param up.
        host_peak = host_copy_gbs()
        host_gbs = 36 * padded / (kern_ms_max / 1e3) / 1e9
        roofline = {"bound": "host", "achieved": host_gbs, "peak": host_peak, "unit": "GB/s",
                    "frac": host_gbs / host_peak, "peak_source": "host memory copy measured in this run (torch CPU copy)",
                    "traffic": None, "algorithmic_bytes_per_launch": 36 * padded, "bytes_per_param": 36,
                    "kernel": "zero_offload_step (host Adam; reduce_out_kernel on the GPU)",
                    "kernel_ms_mean": kern_ms_max, "kernel_ms_min": min(step_kernel_ms)}
        offload = {"chunk": args.offload_chunk, "threads": args.offload_threads or os.cpu_count(),
                   "d2h_bytes_per_step": 4 * padded, "h2d_bytes_per_step": 2 * padded,
                   "link_gbs": 6 * padded / (kern_ms_max / 1e3) / 1e9,
                   "note": "fp32 master/m/v in host memory; per chunk: GPU reduce -> D2H -> host Adam -> H2D, "
                           "3 chunks in flight"}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": warm_done, "ms_per_step": total_ms_max / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic (seeded; bf16/fp32 grads, fp32 state)",
            "config": {"workload": args.workload, "layout": pl.name, "params": pl.total, "padded_params": padded,
                       "units": fs.n_units, "n_ranks_simulated": n, "zero_stage": wl["stage"],
                       "grad_dtype": wl["grad_dtype"], "optimizer": "Adam fp32 (lr 1e-3, betas 0.9/0.999, eps 1e-8)",
                       "parallelism": f"{world} GPU replica(s); N={n} DP ranks simulated per GPU",
                       "l2": f"inputs larger than L2: {bytes_per_launch / 1e9:.2f} GB moved per step (L2 129 MB)",
                       "cuda_graph": bool(args.graph)},
            "hbm_gbs": None if args.offload else achieved_gbs,
            "hbm_frac_of_peak": None if args.offload else achieved_gbs / peak,
            "roofline": roofline,
            "offload": offload,
            "clip": None if clip_ms is None else {
                "max_norm": args.clip, "norm_pass_ms_mean": statistics.mean(clip_ms),
                "keep_reduced": args.clip_keep,
                "norm_pass_bytes": ((2 if wl["grad_dtype"] == "bf16" else 4) * n + (4 if args.clip_keep else 0)) * padded,
                "norm_pass_gbs": ((2 if wl["grad_dtype"] == "bf16" else 4) * n + (4 if args.clip_keep else 0)) * padded
                / (statistics.mean(clip_ms) / 1e3) / 1e9,
                "note": "the clipped step is the norm pass (grad_sq + finalize kernels) plus the step kernel"},
            "gather": None if gather_ms is None else {
                "units": len(gather_bufs), "gather_ms_mean": statistics.mean(gather_ms),
                "gather_bytes": 4 * padded, "gather_gbs": 4 * padded / (statistics.mean(gather_ms) / 1e3) / 1e9,
                "note": "ZeRO-3 per-unit gathers of the bf16 shards into unit buffers (2 B read + 2 B written)"},
            "accum": None if accum_ms is None else {
                "micro_steps": args.accum, "accumulate_ms_mean": statistics.mean(accum_ms),
                "accumulate_bytes": n * padded * (6 + 10 * (args.accum - 1)),
                "accumulate_gbs": n * padded * (6 + 10 * (args.accum - 1)) / (statistics.mean(accum_ms) / 1e3) / 1e9,
                "note": "K micro-steps of bf16 grads accumulated into the fp32 replica gradients, then the step"},
            "cpu_baseline": cpu,
            "cpu_adam": cpu_adam,
            "e2e": e2e,
            "gpu_launches": launches,
            "clocks": clock,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


# ---------------------------------------------------------------------------
# Roofline sweep: one flat fp32 buffer of 1M..1B params x N = 1..16.
# ---------------------------------------------------------------------------
L2_BYTES = 129 * 1024 * 1024


def run_sweep(args):
    import torch
    import synth_inputs as si
    from zero_sharded_mixed_flatparameter_gb300 import build_lib
    from zero_sharded_mixed_flatparameter_gb300.runner import FlatStep
    build_lib.build()
    device = torch.device("cuda", 0)
    stream = torch.cuda.current_stream(device)
    peak, peak_kind = measured_peaks()
    flush = torch.empty(512 * 1024 * 1024, dtype=torch.uint8, device=device)
    sizes = [int(float(x)) for x in args.sweep_sizes.split(",")]
    ranks = [int(x) for x in args.sweep_ranks.split(",")]
    for numel in sizes:
        for n in ranks:
            init = si.normal_fp32(numel, 0.02, 1, device=device)
            fs = FlatStep([numel], [0], stage=2, n_ranks=n, init_params=[init], device=device)
            del init
            # N replica buffers of the padded length (pads zero, as the hook pads them)
            grads = si.replica_grads(n, fs.padded, 1e-2, 2, "bf16", device=device, outlier_fraction=0.001,
                                     pad_from=numel)
            nbytes = bytes_per_param(n, "bf16") * fs.padded
            reps = max(5, min(50, int(2e10 // max(nbytes, 1))))

            def step():
                fs.reduce_grads(-1, grads)
                fs.step()
                fs.post_step()
            for _ in range(3):
                step()
            torch.cuda.synchronize(device)
            # Each timed step is queued behind ~0.1 ms of device work (a
            # bounded spin), so its events bracket the kernel, not the host's
            # launch latency.  "flushed": the 512 MB fill evicts the working
            # set from L2 first; "l2_resident": a warm step runs just before.
            flushed, warm = [], []
            for mode, out in (("flushed", flushed), ("warm", warm)):
                for _ in range(reps):
                    if mode == "flushed":
                        flush.fill_(1)
                    else:
                        step()
                    torch.cuda._sleep(200_000)
                    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    a.record(stream)
                    step()
                    b.record(stream)
                    torch.cuda.synchronize(device)
                    out.append(a.elapsed_time(b))
            mf, mw = statistics.median(flushed), statistics.median(warm)
            print(json.dumps({
                "sweep_point": f"flat:{numel}:{n}", "params": numel, "n_ranks_simulated": n,
                "kernel": step_kernel_name(n, "bf16", False, fs.padded),
                "algorithmic_bytes": nbytes, "bytes_per_param": bytes_per_param(n, "bf16"), "reps": reps,
                "kernel_ms_l2_flushed": mf, "gbs_l2_flushed": nbytes / mf / 1e6,
                "frac_l2_flushed": nbytes / mf / 1e6 / peak, "params_per_s_l2_flushed": numel / mf * 1e3,
                "kernel_ms_l2_resident": mw, "gbs_l2_resident": nbytes / mw / 1e6,
                "working_set_fits_l2": nbytes <= L2_BYTES, "peak_gbs": peak, "peak_source": peak_kind}), flush=True)
            fs.close()
            del grads
            torch.cuda.empty_cache()


# ---------------------------------------------------------------------------
# DRAM ceilings by read:write mix: torch's own elementwise kernels over
# 256 M-element fp32 tensors (1 GiB each), GB/s of bytes moved.  Context for
# the roofline: the copy (1 : 1) is the most write-heavy mix; the step at
# N = 8 bf16 is 2 : 1 and at N = 16 about 3 : 1.
# ---------------------------------------------------------------------------
def run_mix_ceilings(args):
    import torch
    n = 256 * 1024 * 1024
    t = [torch.randn(n, device="cuda") for _ in range(4)]

    def gbs(fn, nbytes, reps=30):
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        times = []
        for _ in range(reps):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            fn()
            b.record()
            torch.cuda.synchronize()
            times.append(a.elapsed_time(b))
        return nbytes / statistics.median(times) / 1e6
    print(json.dumps({
        "mix_ceilings_gbs": {
            "copy 1:1": gbs(lambda: t[1].copy_(t[0]), 8 * n),
            "add 2:1": gbs(lambda: torch.add(t[0], t[1], out=t[2]), 12 * n),
            "addcmul 3:1": gbs(lambda: torch.addcmul(t[0], t[1], t[2], out=t[3]), 16 * n),
            "fill 0:1": gbs(lambda: t[3].fill_(1.0), 4 * n)},
        "tensors": "4 x 256 M fp32 (1 GiB each)", "peak_measured_gbs": measured_peaks()[0]}), flush=True)


# ---------------------------------------------------------------------------
# Reference arm: the CPU oracle on the host cores.
# ---------------------------------------------------------------------------
def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return
    import oracle
    oracle.build()
    wl = workload(args.workload)
    # Each step is a bounded sample: sized so that the K timed steps take about
    # a minute on one core (at most 2M params per step).
    probe = OracleSample(wl, 262_144)
    t0 = time.perf_counter()
    probe.step()
    rate = 262_144 / max(time.perf_counter() - t0, 1e-6)
    sample_params = int(min(2_000_000, max(65_536, rate * 60.0 / max(args.steps, 1))))
    sample_params -= sample_params % 64
    sample = OracleSample(wl, sample_params)
    for _ in range(args.warmup):
        sample.step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        sample.step()
    dt = time.perf_counter() - t0
    value = sample_params * args.steps / dt
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3 / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": args.workload, "layout": wl["pl"].name, "params": wl["pl"].total,
                   "n_ranks_simulated": wl["n"], "zero_stage": wl["stage"], "grad_dtype": wl["grad_dtype"]},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
                         "sample": f"each step: one literal per-rank oracle step on a contiguous {sample_params:,}-param "
                                   f"window of the workload (N={wl['n']}, {wl['grad_dtype']} grads), single-threaded"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None, help="timed steps (default 2000; 50 with --offload)")
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="llama1024_zero2_n8")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--graph", action="store_true",
                    help="capture one step into a CUDA graph (capturable mode) and time its replays")
    ap.add_argument("--offload", action="store_true",
                    help="ZeRO-Offload: fp32 state in host memory, the step through zero_offload_step")
    ap.add_argument("--offload-chunk", type=int, default=1 << 23)
    ap.add_argument("--offload-threads", type=int, default=0)
    ap.add_argument("--accum", type=int, default=0,
                    help="fp32 gradient accumulation of this many bf16 micro-steps before every step (fp32 workloads)")
    ap.add_argument("--clip-keep", action="store_true",
                    help="with --clip: keep the reduced gradient for the step (fewer bytes for N > 4)")
    ap.add_argument("--mix-ceilings", action="store_true",
                    help="DRAM GB/s of torch copy / add / addcmul / fill (read:write mixes 1:1 .. 0:1)")
    ap.add_argument("--sweep", action="store_true",
                    help="roofline sweep of flat buffers (one JSON line per point instead of the bench line)")
    ap.add_argument("--sweep-sizes", default="1e6,16e6,128e6,512e6,1e9")
    ap.add_argument("--sweep-ranks", default="1,2,4,8,16")
    ap.add_argument("--clip", type=float, default=0.0,
                    help="global-norm clipping to this max norm before every step (0: off)")
    args = ap.parse_args()
    if args.steps is None:
        args.steps = 50 if args.offload else 2000
    if args.graph and args.offload:
        ap.error("--graph and --offload exclude each other (the offload step runs on host threads)")
    if args.warmup < 3 and args.impl == "ours":
        print("note: fewer than 3 warm-up steps", file=sys.stderr)
    if args.mix_ceilings:
        run_mix_ceilings(args)
    elif args.sweep:
        run_sweep(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
