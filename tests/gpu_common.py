"""Helpers of the GPU parity tests: run the same seeded problem through the
CUDA library (C ABI) and through the oracle, and compare.

Tolerances (the acceptance bar of the method's GPU path):
  * layout (offsets, padding, shard lengths): exact;
  * fp32 master, m, v: max relative error <= 1e-6 (|got - want| <= 1e-6 |want|,
    so an expected 0 must be exactly 0);
  * bf16 parameters: within 1 bf16 ulp;
  * NaN where the oracle has NaN.
Both sides perform the same separately-rounded IEEE fp32 operations, so the
results are also expected to agree bit for bit; that stronger property is
checked separately (``assert_bit_exact``) so that a failure says which bar
was missed.
"""

from __future__ import annotations

from dataclasses import dataclass
from typing import List, Optional

import numpy as np
import torch

import oracle
import synth_inputs as si
from zero_sharded_mixed_flatparameter_gb300 import binding as B
from zero_sharded_mixed_flatparameter_gb300.runner import FlatStep

RTOL = 1e-6


def ensure_built():
    from zero_sharded_mixed_flatparameter_gb300 import build_lib
    build_lib.build()
    B.load()
    oracle.build()


def to_np(t: torch.Tensor) -> np.ndarray:
    return si.as_numpy_bits(t)


def assert_rel_close(got: np.ndarray, want: np.ndarray, what: str, rtol: float = RTOL):
    got = np.asarray(got, np.float32)
    want = np.asarray(want, np.float32)
    nan_w, nan_g = np.isnan(want), np.isnan(got)
    assert np.array_equal(nan_w, nan_g), f"{what}: NaN positions differ"
    ok = ~nan_w
    g64, w64 = got[ok].astype(np.float64), want[ok].astype(np.float64)
    with np.errstate(invalid="ignore"):
        err = np.abs(g64 - w64)
    # equal infinities have zero error
    err = np.where(g64 == w64, 0.0, err)
    bad = err > rtol * np.abs(w64)
    if bad.any():
        i = int(np.flatnonzero(bad)[0])
        rel = err / np.maximum(np.abs(w64), 1e-300)
        raise AssertionError(f"{what}: {int(bad.sum())} elements beyond rel {rtol}; first at {i}: "
                             f"got {g64[i]!r} want {w64[i]!r}; max rel {rel.max():.3e}")


def assert_bf16_1ulp(got_bits: np.ndarray, want_bits: np.ndarray, what: str):
    g = np.asarray(got_bits, np.uint16).astype(np.int32)
    w = np.asarray(want_bits, np.uint16).astype(np.int32)
    g_nan = ((g & 0x7F80) == 0x7F80) & ((g & 0x7F) != 0)
    w_nan = ((w & 0x7F80) == 0x7F80) & ((w & 0x7F) != 0)
    assert np.array_equal(g_nan, w_nan), f"{what}: NaN positions differ"
    ok = ~w_nan
    # map sign-magnitude bit patterns onto a monotonic integer line
    def ordered(x):
        return np.where(x & 0x8000, -(x & 0x7FFF), x & 0x7FFF)
    d = np.abs(ordered(g[ok]) - ordered(w[ok]))
    assert d.max(initial=0) <= 1, f"{what}: {int((d > 1).sum())} bf16 values beyond 1 ulp"


def assert_bit_exact(got: np.ndarray, want: np.ndarray, what: str):
    ga = np.ascontiguousarray(got).reshape(-1)
    wa = np.ascontiguousarray(want).reshape(-1)
    assert ga.dtype.itemsize == wa.dtype.itemsize and ga.size == wa.size, f"{what}: shape/dtype mismatch"
    ui = np.uint32 if ga.dtype.itemsize == 4 else np.uint16
    differ = ga.view(ui) != wa.view(ui)
    # NaN payloads are not fixed by IEEE arithmetic: a NaN matches any NaN
    if ga.dtype.itemsize == 4:
        both_nan = np.isnan(ga.view(np.float32)) & np.isnan(wa.view(np.float32))
    else:
        gi, wi = ga.view(np.uint16), wa.view(np.uint16)
        both_nan = (((gi & 0x7F80) == 0x7F80) & ((gi & 0x7F) != 0) & ((wi & 0x7F80) == 0x7F80) & ((wi & 0x7F) != 0))
    differ &= ~both_nan
    if differ.any():
        i = int(np.flatnonzero(differ)[0])
        raise AssertionError(f"{what}: {int(differ.sum())} elements differ bitwise; first at {i}: "
                             f"got {ga[i]!r} want {wa[i]!r}")


def compare_state(fs_or_arrays, ref, what: str, bit_exact: bool = True):
    """ref = (master, m, v, p16) numpy; fs_or_arrays a FlatStep or the same tuple."""
    if isinstance(fs_or_arrays, FlatStep):
        got = (to_np(fs_or_arrays.master), to_np(fs_or_arrays.exp_avg), to_np(fs_or_arrays.exp_avg_sq),
               to_np(fs_or_arrays.param16))
    else:
        got = fs_or_arrays
    for name, g, w in zip(("master", "m", "v"), got[:3], ref[:3]):
        assert_rel_close(g, w, f"{what} {name}")
    assert_bf16_1ulp(got[3], ref[3], f"{what} param16")
    if bit_exact:
        for name, g, w in zip(("master", "m", "v", "param16"), got, ref):
            assert_bit_exact(g, w, f"{what} {name} (bit-exact)")


@dataclass
class Problem:
    pl: si.ParamList
    n: int
    stage: int
    grad_dtype: str
    hyper: oracle.Hyper
    lay: oracle.OracleLayout
    init: List[np.ndarray]
    grads: List[List[np.ndarray]]     # [step][replica] flat padded buffers (host)
    max_norm: float = 0.0             # > 0: global-norm clipping before every step


def make_problem(pl: si.ParamList, n: int, stage: int, grad_dtype: str = "bf16", steps: int = 10,
                 seed: int = 0, lr: float = 1e-3, beta1: float = 0.9, beta2: float = 0.999, eps: float = 1e-8,
                 weight_decay: float = 0.0, adamw: bool = False, grad_std: float = 1e-2,
                 outlier_fraction: float = 0.0, max_norm: float = 0.0) -> Problem:
    hyper = oracle.Hyper(lr=lr, beta1=beta1, beta2=beta2, eps=eps, weight_decay=weight_decay, adamw=adamw,
                         n_ranks=n, grad_dtype=grad_dtype)
    lay = oracle.layout(pl.numel, pl.unit, n, stage) if pl.numel else None
    total = lay.total_padded if lay else 0
    init = [si.normal_fp32(k, 0.02, seed * 7919 + p).numpy() for p, k in enumerate(pl.numel)]
    gdt = np.uint16 if grad_dtype == "bf16" else np.float32
    grads = []
    for t in range(steps):
        reps = []
        for r in range(n):
            flat = np.zeros(total, dtype=gdt)
            for p, k in enumerate(pl.numel):
                g = si.replica_grads(1, k, grad_std, seed * 100003 + t * 1009 + p * 31 + r, grad_dtype,
                                     outlier_fraction=outlier_fraction)[0]
                off = int(lay.param_offset[p])
                flat[off:off + k] = to_np(g)
            reps.append(flat)
        grads.append(reps)
    return Problem(pl, n, stage, grad_dtype, hyper, lay, init, grads, max_norm)


def oracle_run(pb: Problem, steps: Optional[int] = None, every_step=None, norms: Optional[list] = None):
    """Runs the oracle over the problem; returns (master, m, v, p16).

    Stage 0 uses the unsharded data-parallel routine; stages 1-3 the literal
    per-rank ZeRO step.  ``every_step(t, state)`` is called after each step;
    with clipping the per-step norms are appended to ``norms``.
    """
    master, m, v, p16 = oracle.make_master(pb.pl.numel, pb.lay, pb.init)
    steps = len(pb.grads) if steps is None else steps
    for t in range(1, steps + 1):
        g = pb.grads[t - 1]
        if pb.stage == 0:
            nrm = oracle.dp_step(pb.hyper, t, g, master, m, v, p16, max_norm=pb.max_norm)
        else:
            nrm = oracle.zero_step(pb.hyper, pb.stage, t, pb.lay, g, master, m, v, p16, max_norm=pb.max_norm)
        if norms is not None:
            norms.append(nrm)
        if every_step:
            every_step(t, (master.copy(), m.copy(), v.copy(), p16.copy()))
    return master, m, v, p16


def gpu_flatstep(pb: Problem, guard: int = 64, device="cuda", offload: Optional[dict] = None) -> FlatStep:
    """offload: None, or dict(chunk=..., threads=...) for a ZeRO-Offload context."""
    init = [torch.from_numpy(a).to(device) for a in pb.init]
    h = pb.hyper
    extra = {}
    if offload is not None:
        extra = dict(offload=True, offload_chunk=offload.get("chunk", 1 << 23),
                     offload_threads=offload.get("threads", 0))
    return FlatStep(pb.pl.numel, pb.pl.unit, stage=pb.stage, n_ranks=pb.n, grad_dtype=pb.grad_dtype,
                    lr=h.lr, beta1=h.beta1, beta2=h.beta2, eps=h.eps, weight_decay=h.weight_decay,
                    adamw=h.adamw, init_params=init, device=device, guard=guard, **extra)


def upload_grads(pb: Problem, t: int, device="cuda") -> List[torch.Tensor]:
    dt = torch.bfloat16 if pb.grad_dtype == "bf16" else torch.float32
    out = []
    for flat in pb.grads[t - 1]:
        x = torch.from_numpy(flat.view(np.int16) if pb.grad_dtype == "bf16" else flat)
        out.append(x.to(device).view(dt))
    return out


def register(fs: FlatStep, pb: Problem, flats: List[torch.Tensor], mode: str, keep: list):
    """mode 'all': whole-buffer registration; 'units': per-unit views of the
    flat buffers; 'separate': per-unit copies in separately allocated buffers."""
    if mode == "all":
        fs.reduce_grads(-1, flats)
        return
    for i in range(fs.n_units):
        numel, padded, shard, base = fs.layout(i)
        if mode == "units":
            views = [f[base:base + padded] for f in flats]
        else:
            views = [f[base:base + padded].clone() for f in flats]
            keep.append(views)
        fs.reduce_grads(i, views)


def check_guards(fs: FlatStep, what: str):
    for gbuf in fs.guards():
        if gbuf.numel():
            assert torch.isnan(gbuf.float()).all().item(), f"{what}: a guard region was overwritten"


def run_gpu(pb: Problem, mode: str = "units", every_step=None, guard: int = 64,
            gather_check: bool = True, norms: Optional[list] = None, clip_keep: bool = False,
            offload: Optional[dict] = None) -> FlatStep:
    fs = gpu_flatstep(pb, guard=guard, offload=offload)
    try:
        for t in range(1, len(pb.grads) + 1):
            flats = upload_grads(pb, t)
            keep = []
            register(fs, pb, flats, mode, keep)
            if pb.max_norm > 0:
                fs.clip_grad_norm(pb.max_norm, keep_reduced=clip_keep)
                if norms is not None:
                    norms.append(fs.grad_norm())
            fs.step()
            if pb.stage == 3 and gather_check:
                for i in range(fs.n_units):
                    numel, padded, shard, base = fs.layout(i)
                    buf = torch.empty(max(padded, 1), dtype=torch.bfloat16, device="cuda")
                    fs.gather_weights(i, buf)
                    torch.cuda.synchronize()
                    assert torch.equal(buf[:padded].view(torch.int16), fs.param16[base:base + padded].view(torch.int16))
                # the same units in one call (the prefetch form), each buffer
                # one element past a 16-byte boundary on odd steps
                o = t % 2
                bufs = [torch.empty(int(fs.layout(i)[1]) + o, dtype=torch.bfloat16, device="cuda")[o:]
                        for i in range(fs.n_units)]
                fs.gather_units(0, bufs)
                torch.cuda.synchronize()
                for i, buf in enumerate(bufs):
                    numel, padded, shard, base = fs.layout(i)
                    assert torch.equal(buf.view(torch.int16), fs.param16[base:base + padded].view(torch.int16)), i
            fs.post_step()
            torch.cuda.synchronize()
            if every_step:
                every_step(t, fs)
        check_guards(fs, "run_gpu")
        return fs
    except Exception:
        fs.close()
        raise
