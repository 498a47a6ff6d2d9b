#!/usr/bin/env python3
"""Benchmark of the fused ZeRO flat-parameter step on GB300.

One "step" is one pass of the whole hot path over one batch of gradients:
reduce_grads (registration of the N replica gradients) -> zero_step (the fused
rank-order fp32 reduce, Adam, bf16 cast) -> gather_weights (ZeRO-3 per-unit
copies; nothing to do for stages 0-2) -> post_step.

Default workload: the pipeline-stage-sized buffer of the Llama-style model
with hidden 2048, intermediate 8192, 32/8 heads, vocab 40960 — 32 decoder
layers plus the input embedding, 2,030,174,208 params in one FlatParameter —
with N = 2 simulated ranks, ZeRO-1, fp32 gradients ~N(0, 1e-3) and fp32 Adam:
(4N + 26) = 34 B/param, 69 GB per step, far above the 129 MB L2 (no flush
is needed between steps).  The same line carries a clipped leg on the same
buffers and, under ``also``, the Llama-1024 ZeRO-2 N = 8 and Llama-2048
ZeRO-3 N = 8 workloads timed the same way.

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

DEFAULT_WORKLOAD = "stage_buffer_zero1_fp32_n2"
ALSO_WORKLOADS = ("llama1024_zero2_n8", "llama2048_zero3_n8", "llama2048_zero3_n6", "llama2048_zero3_n6_unitbufs")
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
    if name.startswith("llama2048_zero3_n") and name[len("llama2048_zero3_n"):].split("_")[0].isdigit():
        # the same units at another N; "_unitbufs": every unit's gradients in
        # buffers of their own (at N = 3, 6, ... the unit bases are then not
        # multiples of 8 and the step takes the shifted-gradient kernel)
        rest = name[len("llama2048_zero3_n"):]
        n = int(rest.split("_")[0])
        if rest not in (str(n), f"{n}_unitbufs"):
            raise SystemExit(f"unknown workload {name}")
        return dict(pl=si.llama_2048_units(), n=n, stage=3, grad_dtype="bf16", grad_std=1e-3, per_unit=True,
                    outliers=0.0, unit_bufs=rest.endswith("_unitbufs"))
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
    """The step kernel the library launches for an aligned segment (base a
    multiple of 8, gradients 16-byte aligned; the others take the
    shifted-gradient kernel, see Workbench.kernel_name): over >= 2^23
    elements the barrier-free pipelined staged one for N = 7..12 bf16, the
    tile-staged one with 2,048-element tiles for N >= 13 bf16 or
    N = 8, 9 fp32 replicas and the one with 4 elements per thread for N = 7
    or N >= 10 fp32 or N = 1..4 bf16 replicas; the register-staged one
    otherwise (a kept fp32 reduced gradient is one fp32 replica)."""
    if clip_keep:
        n, grad_dtype = 1, "fp32"
    if elems < 2 ** 23:
        return "step_vec_kernel"
    if grad_dtype == "bf16":
        if n <= 4:
            return "step_tma4_kernel"
        if 7 <= n <= 12:
            return "step_pipe_kernel"
        return "step_tma_kernel" if n >= 13 else "step_vec_kernel"
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
# The workload's description, printed identically by both arms.
# ---------------------------------------------------------------------------
OPTIMIZER = "Adam fp32 (lr 1e-3, betas 0.9/0.999, eps 1e-8)"
L2_BYTES = 129 * 1024 * 1024


def config_for(name: str, wl, world: int, graph: bool = False) -> dict:
    """The line's ``config``: a function of the workload and the launch only,
    so that the GPU arm and the reference arm print the same dict."""
    pl, n = wl["pl"], wl["n"]
    moved = bytes_per_param(n, wl["grad_dtype"]) * pl.total
    if moved > L2_BYTES:
        l2 = f"inputs larger than L2: {moved / 1e9:.2f} GB moved per step (L2 129 MB)"
    else:
        l2 = f"working set fits L2: {moved / 1e6:.1f} MB moved per step (L2 129 MB), not flushed"
    return {"workload": name, "layout": pl.name, "params": pl.total, "units": pl.n_units,
            "n_ranks_simulated": n, "zero_stage": wl["stage"], "grad_dtype": wl["grad_dtype"],
            "optimizer": OPTIMIZER, "parallelism": f"{world} GPU replica(s); N={n} DP ranks simulated per GPU",
            "l2": l2, "cuda_graph": bool(graph)}


# ---------------------------------------------------------------------------
# Our arm.
# ---------------------------------------------------------------------------
class Workbench:
    """One workload resident on the device: the FlatStep context (master, m, v,
    bf16 parameters), the N replica gradients, the ZeRO-3 unit buffers and,
    with ``accum``, the bf16 micro-step gradients."""

    def __init__(self, name: str, device, rank: int, accum: int = 0, offload_kw=None):
        import torch
        import synth_inputs as si
        from zero_sharded_mixed_flatparameter_gb300.runner import FlatStep
        self.name, self.device, self.accum = name, device, accum
        self.wl = wl = workload(name)
        pl, n = wl["pl"], wl["n"]
        init_flat = si.normal_fp32(pl.total, 0.02, 1 + rank, device=device)
        offs = [0]
        for k in pl.numel:
            offs.append(offs[-1] + k)
        init = [init_flat[offs[p]:offs[p + 1]] for p in range(len(pl.numel))]
        self.fs = FlatStep(pl.numel, pl.unit, stage=wl["stage"], n_ranks=n, grad_dtype=wl["grad_dtype"],
                           init_params=init, device=device, **(offload_kw or {}))
        del init, init_flat
        self.padded = self.fs.padded
        self.units = [self.fs.layout(i) for i in range(self.fs.n_units)]
        self.unit_grads = None
        if wl.get("unit_bufs"):
            # one buffer per unit and replica, as a per-unit gradient hook hands them over
            self.grads = None
            self.unit_grads = [si.replica_grads(n, pad, wl["grad_std"], 100 + 31 * i + rank, wl["grad_dtype"],
                                                device=device, pad_from=numel)
                               for i, (numel, pad, shard, base) in enumerate(self.units)]
        else:
            self.grads = si.replica_grads(n, self.padded, wl["grad_std"], 100 + rank, wl["grad_dtype"],
                                          device=device, outlier_fraction=wl["outliers"])
        self.micro = []
        if accum > 0:
            if wl["grad_dtype"] != "fp32":
                raise SystemExit("--accum needs an fp32-gradient workload (the accumulators are the step's gradients)")
            self.micro = si.replica_grads(n, self.padded, wl["grad_std"], 200 + rank, "bf16", device=device)
        self.gather_bufs = []
        if wl["stage"] == 3:
            self.gather_bufs = [torch.empty(max(u[1], 1), dtype=torch.bfloat16, device=device) for u in self.units]
        self.stream = torch.cuda.current_stream(device)

    def one_step(self, ev=None, clip_ev=None, accum_ev=None, gather_ev=None, clip: float = 0.0,
                 clip_keep: bool = False, grads=None) -> int:
        """reduce_grads -> (clip) -> zero_step -> (gathers) -> post_step; the
        optional event pairs bracket the step kernel, the norm pass, the
        accumulation and the gathers.  Returns the kernels launched."""
        fs, s = self.fs, self.stream
        grads = self.grads if grads is None else grads
        launches = 0
        if self.micro:
            if accum_ev is not None:
                accum_ev[0].record(s)
            for k in range(self.accum):
                fs.accumulate_grads(-1, self.micro, grads, first=(k == 0))
                launches += fs.last_launches()
            if accum_ev is not None:
                accum_ev[1].record(s)
        if self.unit_grads is not None:
            for i, g in enumerate(self.unit_grads):
                fs.reduce_grads(i, g)
        elif self.wl["per_unit"]:
            for i, (numel, pad, shard, base) in enumerate(self.units):
                fs.reduce_grads(i, [g[base:base + pad] for g in grads])
        else:
            fs.reduce_grads(-1, grads)
        if clip > 0:
            if clip_ev is not None:
                clip_ev[0].record(s)
            fs.clip_grad_norm(clip, keep_reduced=clip_keep)
            if clip_ev is not None:
                clip_ev[1].record(s)
            launches += fs.last_launches()
        if ev is not None:
            ev[0].record(s)
        fs.step()
        if ev is not None:
            ev[1].record(s)
        launches += fs.last_launches()
        if gather_ev is not None and self.gather_bufs:
            gather_ev[0].record(s)
        for i, buf in enumerate(self.gather_bufs):
            fs.gather_weights(i, buf)
            launches += fs.last_launches()
        if gather_ev is not None and self.gather_bufs:
            gather_ev[1].record(s)
        fs.post_step()
        return launches

    def shifted_units(self) -> int:
        """Units whose step segment the shifted-gradient kernel takes (a unit
        base that is not a multiple of 8 with gradients in a buffer of its
        own); one flat buffer, or views of it, is one aligned segment."""
        if self.unit_grads is None:
            return 0
        return sum(1 for (numel, pad, shard, base) in self.units if base % 8 and pad)

    def kernel_name(self, clip_keep: bool = False) -> str:
        n, gd = self.wl["n"], self.wl["grad_dtype"]
        k = self.shifted_units()
        if k == 0 or clip_keep:
            return step_kernel_name(n, gd, clip_keep, self.padded)
        if k == len(self.units):
            return "step_shift_kernel"
        return f"step_shift_kernel ({k} units) + {step_kernel_name(n, gd, False, self.padded)}"

    def close(self):
        import torch
        self.fs.close()
        self.grads = self.unit_grads = self.micro = self.gather_bufs = None
        torch.cuda.empty_cache()


def _pairs(k: int, on: bool = True):
    import torch
    if not on:
        return [None] * k
    return [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(k)]


def _ms(pairs):
    if not pairs or pairs[0] is None:
        return None
    return [a.elapsed_time(b) for a, b in pairs]


def timed_steps(wb: Workbench, steps: int, world: int, clip: float = 0.0, clip_keep: bool = False,
                graph=None, graph_launches: int = 0) -> dict:
    """EXACTLY ``steps`` steps between a barrier + synchronize on both sides,
    bracketed by CUDA events on the launching stream; per-launch events give
    the step kernel's (and norm pass's, gathers', accumulation's) durations;
    nvidia-smi samples the clocks inside the window."""
    import torch
    device = wb.device
    ev = _pairs(steps)
    clip_ev = _pairs(steps, clip > 0 and graph is None)
    accum_ev = _pairs(steps, bool(wb.micro) and graph is None)
    gather_ev = _pairs(steps, bool(wb.gather_bufs) and graph is None)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    launches = 0
    with ClockSampler(device.index if device.index is not None else 0) as clocks:
        barrier(world)
        torch.cuda.synchronize(device)
        t0 = time.time()
        start.record(wb.stream)
        for k in range(steps):
            if graph is not None:
                ev[k][0].record(wb.stream)
                graph.replay()
                ev[k][1].record(wb.stream)
                launches += graph_launches
            else:
                launches += wb.one_step(ev[k], clip_ev[k], accum_ev[k], gather_ev[k], clip=clip, clip_keep=clip_keep)
        end.record(wb.stream)
        torch.cuda.synchronize(device)
        t1 = time.time()
        barrier(world)
        clocks.mark(t0, t1)
    return {"total_ms": start.elapsed_time(end), "step_ms": _ms(ev), "clip_ms": _ms(clip_ev),
            "accum_ms": _ms(accum_ev), "gather_ms": _ms(gather_ev), "launches": launches,
            "clocks": clocks.summary()}


def preroll(device, min_seconds: float = 0.3) -> dict:
    """Clock ramp before the warm-up: repeated fills of a 1 GiB scratch buffer
    (not a step, not counted as warm-up), reported in the line."""
    import torch
    buf = torch.empty(1 << 30, dtype=torch.uint8, device=device)
    fills, t0 = 0, time.perf_counter()
    while time.perf_counter() - t0 < min_seconds:
        for _ in range(8):
            buf.fill_(fills & 0xFF)
            fills += 1
        torch.cuda.synchronize(device)
    dt = time.perf_counter() - t0
    del buf
    torch.cuda.empty_cache()
    return {"what": "fills of a 1 GiB scratch buffer before the warm-up (clock ramp; not steps)",
            "fills": fills, "seconds": round(dt, 3)}


def kernel_stats(ms, bytes_per_launch: int, peak: float) -> dict:
    mean, med = statistics.mean(ms), statistics.median(ms)
    return {"kernel_ms_mean": mean, "kernel_ms_median": med, "kernel_ms_min": min(ms),
            "gbs_mean": bytes_per_launch / (mean / 1e3) / 1e9, "gbs_median": bytes_per_launch / (med / 1e3) / 1e9,
            "frac_mean": bytes_per_launch / (mean / 1e3) / 1e9 / peak}


def also_block(name: str, device, rank: int, args, peak: float) -> dict:
    """Another workload timed the same way (device-resident, exact warm-up,
    per-launch events), for the line's ``also`` map.  The timed step count is
    --steps, raised so that the window lasts at least 0.25 s (clock record)."""
    import torch
    wb = Workbench(name, device, rank)
    try:
        for _ in range(args.warmup):
            wb.one_step()
        torch.cuda.synchronize(device)
        wl, n = wb.wl, wb.wl["n"]
        bpp = bytes_per_param(n, wl["grad_dtype"])
        per_step_s = bpp * wb.padded / (0.9 * peak * 1e9)  # estimate, for the window length only
        steps = max(args.steps, int(0.25 / per_step_s) + 1)
        r = timed_steps(wb, steps, 1)
        out = {"config": config_for(name, wl, 1), "padded_params": wb.padded, "steps": steps,
               "warmup": args.warmup, "value": wl["pl"].total * steps / (r["total_ms"] / 1e3), "unit": UNIT,
               "ms_per_step": r["total_ms"] / steps, "bytes_per_param": bpp,
               "kernel": wb.kernel_name(),
               **kernel_stats(r["step_ms"], bpp * wb.padded, peak), "gpu_launches": r["launches"],
               "clocks": r["clocks"]}
        if r["gather_ms"]:
            g = statistics.mean(r["gather_ms"])
            out["gather"] = {"units": len(wb.gather_bufs), "gather_ms_mean": g,
                             "gather_ms_median": statistics.median(r["gather_ms"]), "gather_bytes": 4 * wb.padded,
                             "gather_gbs": 4 * wb.padded / (g / 1e3) / 1e9,
                             "gather_frac": 4 * wb.padded / (g / 1e3) / 1e9 / peak}
            out["gather_prefetch"] = prefetch_leg(wb, steps, peak)
        return out
    finally:
        wb.close()


def prefetch_leg(wb: Workbench, steps: int, peak: float) -> dict:
    """The same ZeRO-3 gathers issued as one zero_gather_units call for every
    unit (the prefetch form: one kernel per 32 units instead of one per unit),
    timed alone after the steps: 3 untimed calls, then ``steps`` calls, each
    bracketed by CUDA events on the launching stream."""
    import torch
    fs, s = wb.fs, wb.stream
    for _ in range(3):
        fs.gather_units(0, wb.gather_bufs, stream=s)
    ev = _pairs(steps)
    torch.cuda.synchronize(wb.device)
    for k in range(steps):
        ev[k][0].record(s)
        fs.gather_units(0, wb.gather_bufs, stream=s)
        ev[k][1].record(s)
    torch.cuda.synchronize(wb.device)
    ms = _ms(ev)
    g = statistics.mean(ms)
    return {"units": len(wb.gather_bufs), "launches_per_call": fs.last_launches(), "calls": steps,
            "gather_ms_mean": g, "gather_ms_median": statistics.median(ms), "gather_bytes": 4 * wb.padded,
            "gather_gbs": 4 * wb.padded / (g / 1e3) / 1e9, "gather_frac": 4 * wb.padded / (g / 1e3) / 1e9 / peak}


def e2e_leg(wb: Workbench, steps: int, warm: int, world: int) -> dict:
    """The same steps through the public API with HOST buffers: every step
    copies its N replica gradients from pinned host memory and reads the
    updated bf16 parameters back.  The host link (not HBM) bounds this, so the
    copies are pipelined on three streams: step k+1's gradients travel on a
    copy stream into the second of two device buffer sets while step k runs
    on the compute stream, which then copies the parameters into one of two
    device staging buffers (a device-to-device copy) that a third stream
    reads back to the host, so that a slow read-back holds up neither the
    next step nor the next gradients."""
    import torch
    device, stream, padded = wb.device, wb.stream, wb.padded
    host_grads = []
    for g in wb.grads:
        h = torch.empty(g.shape, dtype=g.dtype, pin_memory=True)
        h.copy_(g)
        host_grads.append(h)
    host_out = torch.empty(padded, dtype=torch.bfloat16, pin_memory=True)
    bufs = [wb.grads, [torch.empty_like(g) for g in wb.grads]]
    staging = [torch.empty_like(wb.fs.param16) for _ in range(2)]
    copy_stream = torch.cuda.Stream(device)
    d2h_stream = torch.cuda.Stream(device)
    h2d_done = [torch.cuda.Event(), torch.cuda.Event()]
    step_done = [torch.cuda.Event(), torch.cuda.Event()]
    staged = [torch.cuda.Event(), torch.cuda.Event()]
    d2h_done = [torch.cuda.Event(), torch.cuda.Event()]

    def run(k_steps):
        start = torch.cuda.Event()
        start.record(stream)
        with torch.cuda.stream(copy_stream):
            copy_stream.wait_event(start)  # after everything before the run on the compute stream
            for hg, g in zip(host_grads, bufs[0]):
                g.copy_(hg, non_blocking=True)
            h2d_done[0].record(copy_stream)
        for k in range(k_steps):
            cur, nxt = k % 2, (k + 1) % 2
            if k + 1 < k_steps:
                with torch.cuda.stream(copy_stream):
                    if k >= 1:
                        copy_stream.wait_event(step_done[nxt])
                    for hg, g in zip(host_grads, bufs[nxt]):
                        g.copy_(hg, non_blocking=True)
                    h2d_done[nxt].record(copy_stream)
            stream.wait_event(h2d_done[cur])
            wb.one_step(grads=bufs[cur])
            step_done[cur].record(stream)
            if k >= 2:
                stream.wait_event(d2h_done[cur])  # staging[cur]'s previous read-back
            with torch.cuda.stream(stream):
                staging[cur].copy_(wb.fs.param16, non_blocking=True)
            staged[cur].record(stream)
            with torch.cuda.stream(d2h_stream):
                d2h_stream.wait_event(staged[cur])
                host_out.copy_(staging[cur], non_blocking=True)
                d2h_done[cur].record(d2h_stream)
        stream.wait_event(d2h_done[(k_steps - 1) % 2])  # the last read-back ends the run

    run(warm)
    torch.cuda.synchronize(device)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize(device)
    e0.record(stream)
    run(steps)
    e1.record(stream)
    torch.cuda.synchronize(device)
    barrier(world)
    e2e_ms = aggregate([e0.elapsed_time(e1)], "max", world, device)[0]
    params_all = aggregate([float(wb.wl["pl"].total * steps)], "sum", world, device)[0]
    esz = 2 if wb.wl["grad_dtype"] == "bf16" else 4
    return {"value": params_all / (e2e_ms / 1e3), "unit": UNIT,
            "h2d_bytes_per_step": wb.wl["n"] * padded * esz, "d2h_bytes_per_step": padded * 2,
            "ms_per_step": e2e_ms / steps,
            "pipelining": "three streams: step k+1's H2D overlaps step k; each step's parameters are "
                          "copied on the device into one of two staging buffers and read back from there"}


def run_ours(args):
    import torch
    from zero_sharded_mixed_flatparameter_gb300 import binding as B
    from zero_sharded_mixed_flatparameter_gb300 import build_lib

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
    B.load()
    timeouts_before = B.zero_kernel_timeouts()
    peak, peak_kind = measured_peaks()
    pre = preroll(device)

    offload_kw = {}
    if args.offload:
        offload_kw = dict(offload=True, offload_chunk=args.offload_chunk, offload_threads=args.offload_threads)
    wb = Workbench(args.workload, device, rank, accum=args.accum, offload_kw=offload_kw)
    wl, fs, padded, n = wb.wl, wb.fs, wb.padded, wb.wl["n"]
    pl = wl["pl"]

    for _ in range(args.warmup):  # exactly --warmup steps
        wb.one_step(clip=args.clip, clip_keep=args.clip_keep)
    torch.cuda.synchronize(device)

    # --graph: the step (registration, clip, step, gathers, post_step) is
    # captured once into a CUDA graph in the library's capturable mode and
    # the timed region replays it; one eager capturable step first caches
    # the launch shapes.
    graph, graph_launches = None, 0
    if args.graph:
        fs.enable_capturable(max_steps=args.warmup + args.steps + 2)
        graph_launches = wb.one_step(clip=args.clip, clip_keep=args.clip_keep)
        torch.cuda.synchronize(device)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            wb.one_step(clip=args.clip, clip_keep=args.clip_keep)
        torch.cuda.synchronize(device)

    r = timed_steps(wb, args.steps, world, clip=args.clip, clip_keep=args.clip_keep, graph=graph,
                    graph_launches=graph_launches)
    if graph is not None:
        fs.disable_capturable()  # the legs below run eagerly
        del graph
    total_ms_max, kern_ms_max = aggregate([r["total_ms"], statistics.mean(r["step_ms"])], "max", world, device)
    params_all = aggregate([float(pl.total * args.steps)], "sum", world, device)[0]
    value = params_all / (total_ms_max / 1e3)

    # with the kept reduced gradient the step reads one fp32 gradient (4 B)
    bpp = 4 + 26 if (args.clip > 0 and args.clip_keep) else bytes_per_param(n, wl["grad_dtype"])
    bytes_per_launch = bpp * padded
    achieved_gbs = bytes_per_launch / (kern_ms_max / 1e3) / 1e9
    gbytes = (2 if wl["grad_dtype"] == "bf16" else 4) * n * padded  # replica gradient bytes (norm pass reads)

    # Clipped leg: unless the timed region already clipped, --steps more
    # steps with global-norm clipping to --clip-leg on the same buffers (after
    # --warmup clipped warm-up steps), timed the same way.
    clip_block = None
    if args.clip > 0 and r["clip_ms"]:
        c = statistics.mean(r["clip_ms"])
        nb = gbytes + (4 * padded if args.clip_keep else 0)
        clip_block = {"max_norm": args.clip, "keep_reduced": args.clip_keep, "leg": "the timed region itself",
                      "norm_pass_ms_mean": c, "norm_pass_ms_median": statistics.median(r["clip_ms"]),
                      "norm_pass_bytes": nb, "norm_pass_gbs": nb / (c / 1e3) / 1e9,
                      "note": "the clipped step is the norm pass (grad_sq + finalize kernels) plus the step kernel"}
    elif args.clip_leg > 0 and not args.offload and not args.graph:
        for _ in range(args.warmup):
            wb.one_step(clip=args.clip_leg)
        torch.cuda.synchronize(device)
        rc = timed_steps(wb, args.steps, world, clip=args.clip_leg)
        c = statistics.mean(rc["clip_ms"])
        clip_block = {"max_norm": args.clip_leg, "keep_reduced": False,
                      "leg": f"{args.steps} clipped steps after the timed region, same buffers, "
                             f"after {args.warmup} clipped warm-up steps",
                      "value": pl.total * args.steps / (rc["total_ms"] / 1e3), "unit": UNIT,
                      "ms_per_step": rc["total_ms"] / args.steps,
                      "norm_pass_ms_mean": c, "norm_pass_ms_median": statistics.median(rc["clip_ms"]),
                      "norm_pass_bytes": gbytes, "norm_pass_gbs": gbytes / (c / 1e3) / 1e9,
                      "norm_pass_frac": gbytes / (c / 1e3) / 1e9 / peak,
                      "step_kernel": kernel_stats(rc["step_ms"], bytes_per_launch, peak),
                      "gpu_launches": rc["launches"], "clocks": rc["clocks"],
                      "note": "the clipped step is the norm pass (grad_sq + finalize kernels) plus the step kernel"}

    e2e = None
    if not args.no_e2e and not args.offload and wb.grads is not None:
        e2e = e2e_leg(wb, args.steps, min(args.warmup, 3) + 1, world)
    kernel = wb.kernel_name(args.clip > 0 and args.clip_keep)
    wb.close()
    del wb, fs

    also = None
    if world == 1 and not args.offload and not args.graph and args.also:
        also = {name: also_block(name, device, rank, args, peak) for name in args.also.split(",") if name}
    timeouts = B.zero_kernel_timeouts() - timeouts_before

    cpu = cpu_adam = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(wl)
        cpu_adam = cpu_adam_baseline()

    roofline = {"bound": "hbm", "achieved": achieved_gbs, "peak": peak, "unit": "GB/s",
                "frac": achieved_gbs / peak, "peak_source": f"hbm_gbs {peak_kind}",
                "traffic": recorded_traffic(args.workload), "algorithmic_bytes_per_launch": bytes_per_launch,
                "bytes_per_param": bpp, "padded_params": padded,
                "kernel": kernel,
                "kernel_ms_mean": kern_ms_max, "kernel_ms_median": statistics.median(r["step_ms"]),
                "kernel_ms_min": min(r["step_ms"]),
                "gbs_at_median": bytes_per_launch / (statistics.median(r["step_ms"]) / 1e3) / 1e9,
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
                    "kernel_ms_mean": kern_ms_max, "kernel_ms_min": min(r["step_ms"])}
        offload = {"chunk": args.offload_chunk, "threads": args.offload_threads or os.cpu_count(),
                   "d2h_bytes_per_step": 4 * padded, "h2d_bytes_per_step": 2 * padded,
                   "link_gbs": 6 * padded / (kern_ms_max / 1e3) / 1e9,
                   "note": "fp32 master/m/v in host memory; per chunk: GPU reduce -> D2H -> host Adam -> H2D, "
                           "3 chunks in flight"}

    gather = None
    if r["gather_ms"]:
        g = statistics.mean(r["gather_ms"])
        gather = {"units": pl.n_units, "gather_ms_mean": g, "gather_bytes": 4 * padded,
                  "gather_gbs": 4 * padded / (g / 1e3) / 1e9,
                  "note": "ZeRO-3 per-unit gathers of the bf16 shards into unit buffers (2 B read + 2 B written)"}
    accum = None
    if r["accum_ms"]:
        a_ms = statistics.mean(r["accum_ms"])
        ab = n * padded * (6 + 10 * (args.accum - 1))
        accum = {"micro_steps": args.accum, "accumulate_ms_mean": a_ms, "accumulate_bytes": ab,
                 "accumulate_gbs": ab / (a_ms / 1e3) / 1e9,
                 "note": "K micro-steps of bf16 grads accumulated into the fp32 replica gradients, then the step"}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": total_ms_max / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic (seeded; bf16/fp32 grads, fp32 state)",
            "config": config_for(args.workload, wl, world, getattr(args, "graph", False)),
            "hbm_gbs": None if args.offload else achieved_gbs,
            "hbm_frac_of_peak": None if args.offload else achieved_gbs / peak,
            "roofline": roofline,
            "preroll": pre,
            "offload": offload,
            "clip": clip_block,
            "gather": gather,
            "accum": accum,
            "also": also,
            "cpu_baseline": cpu,
            "cpu_adam": cpu_adam,
            "e2e": e2e,
            "gpu_launches": r["launches"],
            "kernel_timeouts": timeouts,
            "clocks": r["clocks"],
        }
        if timeouts:
            line["error"] = (f"{timeouts} bounded wait(s) of a tile-staged kernel gave up during the run: "
                             "some steps were partial, the figures are not valid")
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    if timeouts:
        raise SystemExit(1)


# ---------------------------------------------------------------------------
# Roofline sweep: one flat fp32 buffer of 1M..1B params x N = 1..16.
# ---------------------------------------------------------------------------
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
        "config": config_for(args.workload, wl, world, getattr(args, "graph", False)),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
                         "sample": f"each step: one literal per-rank oracle step on a contiguous {sample_params:,}-param "
                                   f"window of the workload (N={wl['n']}, {wl['grad_dtype']} grads), single-threaded"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None, help="timed steps (default 100; 50 with --offload)")
    ap.add_argument("--warmup", type=int, default=5, help="untimed warm-up steps (exactly this many)")
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--also", default=",".join(ALSO_WORKLOADS),
                    help="comma-separated workloads timed after the main one (1 GPU), reported under 'also'")
    ap.add_argument("--clip-leg", type=float, default=1.0,
                    help="max norm of the clipped leg timed after the main region (0: no leg)")
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
        args.steps = 50 if args.offload else 100
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
