"""ctypes wrapper of the oracle library (test infrastructure only).

Builds ``zero_oracle.cpp`` with the host compiler (single-threaded, no
fast-math, no FMA contraction) and exposes its functions on numpy arrays.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "zero_oracle.cpp")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB = os.path.join(_BUILD_DIR, "libzero_oracle.so")
_lock = threading.Lock()
_lib = None


def library_path() -> str:
    return _LIB


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/_build/libzero_oracle.so``."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = [
        os.environ.get("CXX", "g++"), "-std=c++17", "-O2", "-ffp-contract=off",
        "-fno-fast-math", "-fPIC", "-shared", _SRC, "-o", tmp,
    ]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        build()
        lib = ctypes.CDLL(_LIB)
        i32, i64, f32, u16 = ctypes.c_int32, ctypes.c_int64, ctypes.c_float, ctypes.c_uint16
        vp, P = ctypes.c_void_p, ctypes.POINTER
        lib.oracle_bf16_round.argtypes = [f32]
        lib.oracle_bf16_round.restype = u16
        lib.oracle_bf16_widen.argtypes = [u16]
        lib.oracle_bf16_widen.restype = f32
        lib.oracle_bf16_round_array.argtypes = [i64, vp, vp]
        lib.oracle_bf16_round_array.restype = None
        lib.oracle_layout.argtypes = [i32, vp, vp, i32, i32, i32, vp, vp, vp, vp, vp, P(i64)]
        lib.oracle_layout.restype = ctypes.c_int
        lib.oracle_state_bytes.argtypes = [i32, vp, i32, i32, vp]
        lib.oracle_state_bytes.restype = None
        lib.oracle_zero3_backward_peak.argtypes = [i32, vp, i32, P(i32)]
        lib.oracle_zero3_backward_peak.restype = i64
        lib.oracle_make_master.argtypes = [i32, vp, vp, vp, i64, vp, vp, vp, vp]
        lib.oracle_make_master.restype = None
        lib.oracle_reduce.argtypes = [vp, vp, vp, i64]
        lib.oracle_reduce.restype = f32
        lib.oracle_step_scalars.argtypes = [vp, vp, i64, vp]
        lib.oracle_step_scalars.restype = None
        lib.oracle_zero_step.argtypes = [vp, vp, i32, i64, i32, vp, vp, vp, vp, vp, vp, vp, i32, i32, f32,
                                         P(ctypes.c_double)]
        lib.oracle_zero_step.restype = ctypes.c_int
        lib.oracle_dp_step.argtypes = [vp, vp, i64, i64, vp, vp, vp, vp, vp, f32, P(ctypes.c_double)]
        lib.oracle_dp_step.restype = None
        lib.oracle_step_window.argtypes = [vp, vp, i64, i64, vp, vp, vp, vp, vp, f32]
        lib.oracle_grad_norm.argtypes = [vp, vp, i64, vp]
        lib.oracle_grad_norm.restype = ctypes.c_double
        lib.oracle_clip_coef.argtypes = [ctypes.c_double, f32]
        lib.oracle_clip_coef.restype = f32
        lib.oracle_nonfinite_count.argtypes = [vp, vp, i64, vp]
        lib.oracle_nonfinite_count.restype = i64
        lib.oracle_step_window.restype = None
        lib.oracle_export.argtypes = [i32, vp, vp, vp, vp]
        lib.oracle_export.restype = None
        lib.oracle_import.argtypes = [i32, vp, vp, i64, vp, vp]
        lib.oracle_import.restype = None
        lib.oracle_accumulate.argtypes = [i32, i64, vp, vp, i32]
        lib.oracle_accumulate.restype = None
        lib.oracle_gather_unit.argtypes = [i64, i64, i32, vp, vp]
        lib.oracle_gather_unit.restype = None
        _lib = lib
        return lib


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be contiguous"
    return a.ctypes.data


@dataclass
class Hyper:
    """Optimizer hyper-parameters and the simulated DP degree N."""

    lr: float = 1e-3
    beta1: float = 0.9
    beta2: float = 0.999
    eps: float = 1e-8
    weight_decay: float = 0.0
    adamw: bool = False
    n_ranks: int = 1
    grad_dtype: str = "bf16"  # "bf16" or "fp32"

    def pack(self):
        f = np.array([self.lr, self.beta1, self.beta2, self.eps, self.weight_decay], dtype=np.float32)
        i = np.array([1 if self.adamw else 0, self.n_ranks, 0 if self.grad_dtype == "bf16" else 1],
                     dtype=np.int32)
        return f, i


@dataclass
class OracleLayout:
    unit_numel: np.ndarray
    unit_padded: np.ndarray
    unit_shard: np.ndarray
    unit_base: np.ndarray
    param_offset: np.ndarray
    total_padded: int


def bf16_round(x) -> np.ndarray:
    """fp32 -> bf16 bit patterns (uint16), round to nearest even."""
    lib = _load()
    x = np.ascontiguousarray(np.asarray(x, dtype=np.float32).reshape(-1))
    out = np.empty(x.shape, dtype=np.uint16)
    lib.oracle_bf16_round_array(x.size, _ptr(x), _ptr(out))
    return out


def bf16_widen(h) -> np.ndarray:
    """bf16 bit patterns -> fp32 (exact)."""
    lib = _load()
    h = np.asarray(h, dtype=np.uint16).reshape(-1)
    return np.array([lib.oracle_bf16_widen(int(b)) for b in h], dtype=np.float32)


def layout(param_numel, param_unit, n_ranks: int, stage: int) -> OracleLayout:
    lib = _load()
    numel = np.ascontiguousarray(np.asarray(param_numel, dtype=np.int64))
    unit = np.ascontiguousarray(np.asarray(param_unit, dtype=np.int32))
    n_units = int(unit.max()) + 1 if unit.size else 0
    un, up, us, ub = (np.zeros(max(n_units, 1), dtype=np.int64) for _ in range(4))
    po = np.zeros(max(numel.size, 1), dtype=np.int64)
    total = ctypes.c_int64(0)
    rc = lib.oracle_layout(numel.size, _ptr(numel), _ptr(unit), n_ranks, stage, n_units,
                           _ptr(un), _ptr(up), _ptr(us), _ptr(ub), _ptr(po), ctypes.byref(total))
    if rc != 0:
        raise ValueError("oracle_layout rejected the parameter list")
    return OracleLayout(un[:n_units], up[:n_units], us[:n_units], ub[:n_units],
                        po[:numel.size], int(total.value))


def state_bytes(unit_padded, n_ranks: int, stage: int) -> np.ndarray:
    lib = _load()
    up = np.ascontiguousarray(np.asarray(unit_padded, dtype=np.int64))
    out = np.zeros(n_ranks, dtype=np.int64)
    lib.oracle_state_bytes(up.size, _ptr(up), n_ranks, stage, _ptr(out))
    return out


def zero3_backward_peak(unit_padded, n_ranks: int):
    """Returns (peak_bytes, unit_index_of_peak) for one rank."""
    lib = _load()
    up = np.ascontiguousarray(np.asarray(unit_padded, dtype=np.int64))
    where = ctypes.c_int32(-1)
    peak = lib.oracle_zero3_backward_peak(up.size, _ptr(up), n_ranks, ctypes.byref(where))
    return int(peak), int(where.value)


def make_master(param_numel, lay: OracleLayout, init_params):
    """Returns (master, m, v, param16) for the flattened, padded layout."""
    lib = _load()
    numel = np.ascontiguousarray(np.asarray(param_numel, dtype=np.int64))
    srcs = [np.ascontiguousarray(np.asarray(p, dtype=np.float32).reshape(-1)) for p in init_params]
    ptrs = (ctypes.c_void_p * max(len(srcs), 1))(*[_ptr(s) for s in srcs])
    n = lay.total_padded
    master = np.empty(n, dtype=np.float32)
    m = np.empty(n, dtype=np.float32)
    v = np.empty(n, dtype=np.float32)
    p16 = np.empty(n, dtype=np.uint16)
    lib.oracle_make_master(numel.size, _ptr(numel), _ptr(lay.param_offset), ptrs, n,
                           _ptr(master), _ptr(m), _ptr(v), _ptr(p16))
    return master, m, v, p16


def _grad_ptrs(grads, hyper: Hyper):
    want = np.uint16 if hyper.grad_dtype == "bf16" else np.float32
    arrs = []
    for g in grads:
        a = np.asarray(g)
        if a.dtype != want:
            raise TypeError(f"replica grads must be {want.__name__} arrays (bf16 as uint16 bits)")
        arrs.append(np.ascontiguousarray(a.reshape(-1)))
    if len(arrs) != hyper.n_ranks:
        raise ValueError("need exactly N replica gradient buffers")
    return arrs, (ctypes.c_void_p * len(arrs))(*[_ptr(a) for a in arrs])


def reduce_element(hyper: Hyper, grads, j: int) -> float:
    lib = _load()
    f, i = hyper.pack()
    arrs, ptrs = _grad_ptrs(grads, hyper)
    return float(lib.oracle_reduce(_ptr(f), _ptr(i), ptrs, j))


def step_scalars(hyper: Hyper, t: int) -> dict:
    lib = _load()
    f, i = hyper.pack()
    out = np.zeros(6, dtype=np.float32)
    lib.oracle_step_scalars(_ptr(f), _ptr(i), t, _ptr(out))
    return dict(zip(["one_minus_beta1", "one_minus_beta2", "bc1", "bc2", "decay", "inv_n"], out))


def zero_step(hyper: Hyper, stage: int, t: int, lay: OracleLayout, grads, master, m, v,
              param16_copies, plant_skip_allgather: bool = False, max_norm: float = 0.0):
    """Literal per-rank ZeRO step in place.  ``param16_copies`` is (n_copies, P) uint16.

    ``max_norm`` > 0 clips the reduced gradient to that global L2 norm; the
    norm is returned (None without clipping)."""
    lib = _load()
    f, i = hyper.pack()
    arrs, ptrs = _grad_ptrs(grads, hyper)
    p16 = param16_copies
    n_copies = p16.shape[0] if p16.ndim == 2 else 1
    norm = ctypes.c_double(float("nan"))
    rc = lib.oracle_zero_step(_ptr(f), _ptr(i), stage, t, lay.unit_padded.size,
                              _ptr(lay.unit_padded), _ptr(lay.unit_base), ptrs,
                              _ptr(master), _ptr(m), _ptr(v), _ptr(p16), n_copies,
                              1 if plant_skip_allgather else 0, max_norm, ctypes.byref(norm))
    if rc != 0:
        raise ValueError("oracle_zero_step rejected its arguments")
    return norm.value if max_norm > 0 else None


def dp_step(hyper: Hyper, t: int, grads, master, m, v, param16, max_norm: float = 0.0):
    """Unsharded data-parallel step in place over the whole buffer (returns the norm when clipping)."""
    lib = _load()
    f, i = hyper.pack()
    arrs, ptrs = _grad_ptrs(grads, hyper)
    norm = ctypes.c_double(float("nan"))
    lib.oracle_dp_step(_ptr(f), _ptr(i), t, master.size, ptrs, _ptr(master), _ptr(m), _ptr(v),
                       _ptr(param16), max_norm, ctypes.byref(norm))
    return norm.value if max_norm > 0 else None


def step_window(hyper: Hyper, t: int, grads, master, m, v, param16, clip_coef: float = 1.0) -> None:
    """Step t on a window of consecutive elements, in place (optionally clipped by ``clip_coef``)."""
    lib = _load()
    f, i = hyper.pack()
    arrs, ptrs = _grad_ptrs(grads, hyper)
    lib.oracle_step_window(_ptr(f), _ptr(i), t, master.size, ptrs, _ptr(master), _ptr(m), _ptr(v),
                           _ptr(param16), clip_coef)


def grad_norm(hyper: Hyper, grads) -> float:
    """Global L2 norm of the reduced gradient (fp64 squares and sum, element order)."""
    lib = _load()
    f, i = hyper.pack()
    arrs, ptrs = _grad_ptrs(grads, hyper)
    return float(lib.oracle_grad_norm(_ptr(f), _ptr(i), arrs[0].size, ptrs))


def nonfinite_count(hyper: Hyper, grads) -> int:
    """Elements whose reduced gradient (rank-order fp32 sum x 1/N) is inf or NaN."""
    lib = _load()
    f, i = hyper.pack()
    arrs, ptrs = _grad_ptrs(grads, hyper)
    return int(lib.oracle_nonfinite_count(_ptr(f), _ptr(i), arrs[0].size, ptrs))


def clip_coef(norm: float, max_norm: float) -> float:
    """min(1, max_norm / (norm + 1e-6)) rounded to fp32."""
    return float(_load().oracle_clip_coef(norm, max_norm))


def export_state(lay: OracleLayout, padded) -> np.ndarray:
    """Real elements of every unit, back to back (pads dropped)."""
    lib = _load()
    src = np.ascontiguousarray(np.asarray(padded, dtype=np.float32))
    out = np.empty(int(lay.unit_numel.sum()), dtype=np.float32)
    lib.oracle_export(lay.unit_numel.size, _ptr(lay.unit_numel), _ptr(lay.unit_base), _ptr(src), _ptr(out))
    return out


def import_state(lay: OracleLayout, compact) -> np.ndarray:
    """Inverse of export_state into ``lay``'s padded layout (pads zero)."""
    lib = _load()
    src = np.ascontiguousarray(np.asarray(compact, dtype=np.float32))
    if src.size != int(lay.unit_numel.sum()):
        raise ValueError("compact state size does not match the layout")
    out = np.empty(lay.total_padded, dtype=np.float32)
    lib.oracle_import(lay.unit_numel.size, _ptr(lay.unit_numel), _ptr(lay.unit_base), lay.total_padded, _ptr(src),
                      _ptr(out))
    return out


def accumulate(micro, acc, first: bool) -> None:
    """One micro-step of fp32 gradient accumulation in place: acc[r] (+)= widen(micro[r])."""
    lib = _load()
    if len(micro) != len(acc):
        raise ValueError("one accumulator per replica")
    ms = [np.ascontiguousarray(np.asarray(x, dtype=np.uint16).reshape(-1)) for x in micro]
    for a in acc:
        if a.dtype != np.float32 or not a.flags["C_CONTIGUOUS"]:
            raise TypeError("accumulators must be contiguous float32 arrays (updated in place)")
    n = ms[0].size if ms else 0
    mp = (ctypes.c_void_p * max(len(ms), 1))(*[_ptr(x) for x in ms])
    ap = (ctypes.c_void_p * max(len(acc), 1))(*[_ptr(a) for a in acc])
    lib.oracle_accumulate(len(ms), n, mp, ap, 1 if first else 0)


def gather_unit(param16, unit_base: int, unit_padded: int, n_ranks: int) -> np.ndarray:
    lib = _load()
    p16 = np.ascontiguousarray(param16)
    out = np.empty(unit_padded, dtype=np.uint16)
    lib.oracle_gather_unit(unit_base, unit_padded, n_ranks, _ptr(p16), _ptr(out))
    return out
