"""ctypes binding of the C ABI in ``include/zero_flatstep.h`` (argument marshalling only).

Every function has the C name and takes plain integers for pointers and
streams (``tensor.data_ptr()``, ``stream.cuda_stream``).  A non-OK status
raises :class:`ZeroError` carrying the status and the library's error text.
There is no fallback: if the CUDA library has not been built, loading raises.
"""

from __future__ import annotations

import ctypes
import os
import threading
from typing import Sequence

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libzero_flatstep.so")

ZERO_OK, ZERO_EINVAL, ZERO_ENOMEM, ZERO_ECUDA, ZERO_ESTATE, ZERO_ENOTSUP = range(6)
STATUS_NAMES = {0: "ZERO_OK", 1: "ZERO_EINVAL", 2: "ZERO_ENOMEM", 3: "ZERO_ECUDA", 4: "ZERO_ESTATE",
                5: "ZERO_ENOTSUP"}
ZERO_GRAD_BF16, ZERO_GRAD_FP32 = 0, 1

# Every symbol the public header declares.
EXPORTED = (
    "zero_plan", "zero_make_master", "zero_num_units", "zero_padded_numel", "zero_layout",
    "zero_param_offset", "zero_state_bytes", "zero_stage3_peak_bytes", "zero_reduce_grads",
    "zero_step", "zero_gather_weights", "zero_post_step", "zero_step_count", "zero_last_launches", "zero_set_lr",
    "zero_destroy", "zero_last_error", "zero_status_string", "zero_clip_workspace_bytes", "zero_clip_grad_norm",
    "zero_grad_norm", "zero_clip_grad_norm_static", "zero_accumulate_grads", "zero_export_state",
    "zero_import_state", "zero_clip_workspace_bytes_ex", "zero_clip_grad_norm_ex", "zero_kernel_timeouts",
    "zero_make_master_offload", "zero_offload_workspace_bytes", "zero_offload_step", "zero_cpu_adam",
    "zero_debug_inject", "zero_debug_check_failures", "zero_capturable_workspace_bytes", "zero_enable_capturable",
    "zero_disable_capturable", "zero_count_nonfinite", "zero_read_nonfinite", "zero_gather_units",
)
ZERO_CLIP_KEEP_REDUCED = 1
ZERO_INJECT_MISSING_COPY = 1
ZERO_INJECT_SHORT_BOUNDS = 2


class zero_config(ctypes.Structure):
    _fields_ = [("stage", ctypes.c_int32), ("n_ranks", ctypes.c_int32), ("grad_dtype", ctypes.c_int32),
                ("adamw", ctypes.c_int32), ("lr", ctypes.c_float), ("beta1", ctypes.c_float),
                ("beta2", ctypes.c_float), ("eps", ctypes.c_float), ("weight_decay", ctypes.c_float)]


class zero_buffers(ctypes.Structure):
    _fields_ = [("master", ctypes.c_void_p), ("exp_avg", ctypes.c_void_p), ("exp_avg_sq", ctypes.c_void_p),
                ("param16", ctypes.c_void_p)]


class ZeroError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {message}")
        self.status = status


_lib = None
_lock = threading.Lock()


def load(path: str = LIB_PATH):
    """Load the CUDA library; raises if it is missing (no fallback exists)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(path):
            raise RuntimeError(
                f"CUDA library {path} is missing: build it with "
                "`python -c 'import __graft_entry__ as g; g.build()'`")
        lib = ctypes.CDLL(path)
        vp, i32, i64, f32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float
        P = ctypes.POINTER
        sig = {
            "zero_plan": [P(zero_config), vp, vp, i32, P(vp)],
            "zero_make_master": [P(zero_config), vp, vp, i32, vp, P(zero_buffers), vp, P(vp)],
            "zero_num_units": [vp, P(i32)],
            "zero_padded_numel": [vp, P(i64), P(i64)],
            "zero_layout": [vp, i32, P(i64), P(i64), P(i64), P(i64)],
            "zero_param_offset": [vp, i32, P(i64)],
            "zero_state_bytes": [vp, i32, vp],
            "zero_stage3_peak_bytes": [vp, P(i64), P(i32)],
            "zero_reduce_grads": [vp, i32, vp, vp],
            "zero_step": [vp, vp],
            "zero_gather_weights": [vp, i32, vp, vp],
            "zero_gather_units": [vp, i32, i32, P(vp), vp],
            "zero_post_step": [vp, vp],
            "zero_step_count": [vp, P(i64)],
            "zero_last_launches": [vp, P(i32)],
            "zero_set_lr": [vp, f32],
            "zero_destroy": [vp],
            "zero_clip_workspace_bytes": [vp, P(i64)],
            "zero_clip_grad_norm": [vp, f32, vp, i64, vp],
            "zero_grad_norm": [vp, P(ctypes.c_double), vp],
            "zero_clip_grad_norm_static": [vp, f32, vp],
            "zero_accumulate_grads": [vp, i32, vp, vp, i32, vp],
            "zero_export_state": [vp, vp, vp, vp, P(i64), vp],
            "zero_import_state": [vp, vp, vp, vp, i64, vp],
            "zero_clip_workspace_bytes_ex": [vp, i32, P(i64)],
            "zero_clip_grad_norm_ex": [vp, f32, i32, vp, i64, vp],
            "zero_kernel_timeouts": [vp, P(ctypes.c_uint32)],
            "zero_count_nonfinite": [vp, vp],
            "zero_read_nonfinite": [vp, P(ctypes.c_uint64), vp],
            "zero_make_master_offload": [P(zero_config), vp, vp, i32, vp, P(zero_buffers), vp, P(vp)],
            "zero_offload_workspace_bytes": [vp, i64, P(i64), P(i64)],
            "zero_offload_step": [vp, i64, vp, i64, vp, i64, i32, vp, vp],
            "zero_cpu_adam": [P(zero_config), i64, vp, vp, vp, vp, vp, i64, i32],
            "zero_debug_inject": [vp, i32],
            "zero_debug_check_failures": [P(ctypes.c_uint32)],
            "zero_capturable_workspace_bytes": [vp, i64, P(i64)],
            "zero_enable_capturable": [vp, vp, i64, i64, vp],
            "zero_disable_capturable": [vp, vp],
        }
        for name, args in sig.items():
            fn = getattr(lib, name)
            fn.argtypes = args
            fn.restype = ctypes.c_int
        lib.zero_last_error.argtypes = [vp]
        lib.zero_last_error.restype = ctypes.c_char_p
        lib.zero_status_string.argtypes = [ctypes.c_int]
        lib.zero_status_string.restype = ctypes.c_char_p
        _lib = lib
        return lib


def _check(status: int, ctx=None):
    if status != ZERO_OK:
        msg = load().zero_last_error(ctx)
        raise ZeroError(status, msg.decode() if msg else "")


def _i64(values: Sequence[int]):
    return (ctypes.c_int64 * max(len(values), 1))(*[int(v) for v in values])


def _i32(values: Sequence[int]):
    return (ctypes.c_int32 * max(len(values), 1))(*[int(v) for v in values])


def _ptrs(values: Sequence[int]):
    return (ctypes.c_void_p * max(len(values), 1))(*[int(v) if v else None for v in values])


def make_config(stage: int, n_ranks: int, grad_dtype: str = "bf16", lr: float = 1e-3, beta1: float = 0.9,
                beta2: float = 0.999, eps: float = 1e-8, weight_decay: float = 0.0,
                adamw: bool = False) -> zero_config:
    return zero_config(stage, n_ranks, ZERO_GRAD_BF16 if grad_dtype == "bf16" else ZERO_GRAD_FP32,
                       1 if adamw else 0, lr, beta1, beta2, eps, weight_decay)


# ---------------------------------------------------------------------------
# The C calls, one Python function each.  ``ctx`` is the opaque handle (int).
# ---------------------------------------------------------------------------
def zero_plan(cfg: zero_config, param_numel: Sequence[int], param_unit: Sequence[int]) -> int:
    lib = load()
    out = ctypes.c_void_p()
    _check(lib.zero_plan(ctypes.byref(cfg), _i64(param_numel), _i32(param_unit), len(param_numel),
                         ctypes.byref(out)))
    return out.value


def zero_make_master(cfg: zero_config, param_numel: Sequence[int], param_unit: Sequence[int],
                     init_params: Sequence[int], master: int, exp_avg: int, exp_avg_sq: int, param16: int,
                     stream: int = 0) -> int:
    lib = load()
    out = ctypes.c_void_p()
    bufs = zero_buffers(master, exp_avg, exp_avg_sq, param16)
    _check(lib.zero_make_master(ctypes.byref(cfg), _i64(param_numel), _i32(param_unit), len(param_numel),
                                _ptrs(init_params), ctypes.byref(bufs), stream or None, ctypes.byref(out)))
    return out.value


def zero_make_master_offload(cfg: zero_config, param_numel: Sequence[int], param_unit: Sequence[int],
                             init_params: Sequence[int], master: int, exp_avg: int, exp_avg_sq: int,
                             param16: int, stream: int = 0) -> int:
    """master / exp_avg / exp_avg_sq are host addresses, param16 a device one."""
    lib = load()
    out = ctypes.c_void_p()
    bufs = zero_buffers(master, exp_avg, exp_avg_sq, param16)
    _check(lib.zero_make_master_offload(ctypes.byref(cfg), _i64(param_numel), _i32(param_unit), len(param_numel),
                                        _ptrs(init_params), ctypes.byref(bufs), stream or None, ctypes.byref(out)))
    return out.value


def zero_offload_workspace_bytes(ctx: int, chunk: int):
    """(host bytes, device bytes) of zero_offload_step's workspaces."""
    h, d = ctypes.c_int64(), ctypes.c_int64()
    _check(load().zero_offload_workspace_bytes(ctx, chunk, ctypes.byref(h), ctypes.byref(d)), ctx)
    return h.value, d.value


def zero_offload_step(ctx: int, chunk: int, host_ws: int, host_bytes: int, dev_ws: int, dev_bytes: int,
                      n_threads: int = 0, stream: int = 0, copy_stream: int = 0) -> None:
    _check(load().zero_offload_step(ctx, chunk, host_ws, host_bytes, dev_ws, dev_bytes, n_threads, stream or None,
                                    copy_stream or None), ctx)


def zero_cpu_adam(cfg: zero_config, t: int, grad: int, master: int, exp_avg: int, exp_avg_sq: int, param16: int,
                  n: int, n_threads: int = 0) -> None:
    """Host Adam over host arrays (addresses of fp32 grad/master/m/v and uint16 param16)."""
    _check(load().zero_cpu_adam(ctypes.byref(cfg), t, grad, master, exp_avg, exp_avg_sq, param16, n, n_threads))


def zero_num_units(ctx: int) -> int:
    n = ctypes.c_int32()
    _check(load().zero_num_units(ctx, ctypes.byref(n)), ctx)
    return n.value


def zero_padded_numel(ctx: int):
    padded, numel = ctypes.c_int64(), ctypes.c_int64()
    _check(load().zero_padded_numel(ctx, ctypes.byref(padded), ctypes.byref(numel)), ctx)
    return padded.value, numel.value


def zero_layout(ctx: int, unit: int):
    """Returns (numel, padded, shard, base) of one unit."""
    vals = [ctypes.c_int64() for _ in range(4)]
    _check(load().zero_layout(ctx, unit, *[ctypes.byref(v) for v in vals]), ctx)
    return tuple(v.value for v in vals)


def zero_param_offset(ctx: int, param: int) -> int:
    off = ctypes.c_int64()
    _check(load().zero_param_offset(ctx, param, ctypes.byref(off)), ctx)
    return off.value


MAX_RANKS = 16  # the library's upper bound on n_ranks


def zero_state_bytes(ctx: int, stage: int, n_ranks: int):
    """Per-rank bytes of `stage` for the context's n_ranks ranks (n_ranks is
    the context's; the library writes that many entries, so the array has
    room for the largest n_ranks whatever the caller passes)."""
    out = (ctypes.c_int64 * MAX_RANKS)()
    _check(load().zero_state_bytes(ctx, stage, out), ctx)
    return list(out)[:n_ranks]


def zero_stage3_peak_bytes(ctx: int):
    peak, unit = ctypes.c_int64(), ctypes.c_int32()
    _check(load().zero_stage3_peak_bytes(ctx, ctypes.byref(peak), ctypes.byref(unit)), ctx)
    return peak.value, unit.value


def zero_reduce_grads(ctx: int, unit: int, replica_grads: Sequence[int], stream: int = 0) -> None:
    _check(load().zero_reduce_grads(ctx, unit, _ptrs(replica_grads), stream or None), ctx)


def zero_accumulate_grads(ctx: int, unit: int, micro_grads: Sequence[int], accumulators: Sequence[int],
                          first: bool, stream: int = 0) -> None:
    _check(load().zero_accumulate_grads(ctx, unit, _ptrs(micro_grads), _ptrs(accumulators), 1 if first else 0,
                                        stream or None), ctx)


def zero_step(ctx: int, stream: int = 0) -> None:
    _check(load().zero_step(ctx, stream or None), ctx)


def zero_gather_weights(ctx: int, unit: int, unit_buf: int, stream: int = 0) -> None:
    _check(load().zero_gather_weights(ctx, unit, unit_buf or None, stream or None), ctx)


def zero_gather_units(ctx: int, first_unit: int, unit_bufs, stream: int = 0) -> None:
    """Units first_unit .. first_unit + len(unit_bufs) - 1 into the device
    addresses unit_bufs (0 for an empty unit)."""
    arr = (ctypes.c_void_p * max(len(unit_bufs), 1))(*[b or None for b in unit_bufs])
    _check(load().zero_gather_units(ctx, first_unit, len(unit_bufs), arr, stream or None), ctx)


def zero_post_step(ctx: int, stream: int = 0) -> None:
    _check(load().zero_post_step(ctx, stream or None), ctx)


def zero_export_state(ctx: int, master_out: int, exp_avg_out: int, exp_avg_sq_out: int, stream: int = 0) -> int:
    """Enqueues the export; returns the step count t."""
    t = ctypes.c_int64()
    _check(load().zero_export_state(ctx, master_out or None, exp_avg_out or None, exp_avg_sq_out or None,
                                    ctypes.byref(t), stream or None), ctx)
    return t.value


def zero_import_state(ctx: int, master_in: int, exp_avg_in: int, exp_avg_sq_in: int, t: int,
                      stream: int = 0) -> None:
    _check(load().zero_import_state(ctx, master_in or None, exp_avg_in or None, exp_avg_sq_in or None, t,
                                    stream or None), ctx)


def zero_count_nonfinite(ctx: int, counter: int) -> None:
    _check(load().zero_count_nonfinite(ctx, counter or None), ctx)


def zero_read_nonfinite(ctx: int, stream: int = 0) -> int:
    n = ctypes.c_uint64()
    _check(load().zero_read_nonfinite(ctx, ctypes.byref(n), stream or None), ctx)
    return n.value


def zero_kernel_timeouts(ctx: int | None = None) -> int:
    n = ctypes.c_uint32()
    _check(load().zero_kernel_timeouts(ctx, ctypes.byref(n)), ctx)
    return n.value


def zero_debug_inject(ctx: int, what: int) -> None:
    _check(load().zero_debug_inject(ctx, what), ctx)


def zero_debug_check_failures() -> int:
    """Failed index checks of a debug build (raises ZERO_ENOTSUP on a release build)."""
    n = ctypes.c_uint32()
    _check(load().zero_debug_check_failures(ctypes.byref(n)))
    return n.value


def zero_capturable_workspace_bytes(ctx: int, max_steps: int) -> int:
    n = ctypes.c_int64()
    _check(load().zero_capturable_workspace_bytes(ctx, max_steps, ctypes.byref(n)), ctx)
    return n.value


def zero_enable_capturable(ctx: int, workspace: int, workspace_bytes: int, max_steps: int, stream: int = 0) -> None:
    _check(load().zero_enable_capturable(ctx, workspace, workspace_bytes, max_steps, stream or None), ctx)


def zero_disable_capturable(ctx: int, stream: int = 0) -> None:
    _check(load().zero_disable_capturable(ctx, stream or None), ctx)


def zero_step_count(ctx: int) -> int:
    t = ctypes.c_int64()
    _check(load().zero_step_count(ctx, ctypes.byref(t)), ctx)
    return t.value


def zero_last_launches(ctx: int) -> int:
    n = ctypes.c_int32()
    _check(load().zero_last_launches(ctx, ctypes.byref(n)), ctx)
    return n.value


def zero_set_lr(ctx: int, lr: float) -> None:
    _check(load().zero_set_lr(ctx, lr), ctx)


def zero_clip_workspace_bytes(ctx: int) -> int:
    n = ctypes.c_int64()
    _check(load().zero_clip_workspace_bytes(ctx, ctypes.byref(n)), ctx)
    return n.value


def zero_clip_grad_norm(ctx: int, max_norm: float, workspace: int, workspace_bytes: int, stream: int = 0) -> None:
    _check(load().zero_clip_grad_norm(ctx, max_norm, workspace or None, workspace_bytes, stream or None), ctx)


def zero_clip_workspace_bytes_ex(ctx: int, flags: int) -> int:
    n = ctypes.c_int64()
    _check(load().zero_clip_workspace_bytes_ex(ctx, flags, ctypes.byref(n)), ctx)
    return n.value


def zero_clip_grad_norm_ex(ctx: int, max_norm: float, flags: int, workspace: int, workspace_bytes: int,
                           stream: int = 0) -> None:
    _check(load().zero_clip_grad_norm_ex(ctx, max_norm, flags, workspace or None, workspace_bytes,
                                         stream or None), ctx)


def zero_clip_grad_norm_static(ctx: int, max_norm: float, stream: int = 0) -> None:
    """zero_clip_grad_norm without a workspace: for callers that cannot allocate."""
    _check(load().zero_clip_grad_norm_static(ctx, max_norm, stream or None), ctx)


def zero_grad_norm(ctx: int, stream: int = 0) -> float:
    out = ctypes.c_double()
    _check(load().zero_grad_norm(ctx, ctypes.byref(out), stream or None), ctx)
    return out.value


def zero_destroy(ctx: int) -> None:
    if ctx:
        _check(load().zero_destroy(ctx))


def zero_last_error(ctx: int | None = None) -> str:
    msg = load().zero_last_error(ctx)
    return msg.decode() if msg else ""


def zero_status_string(status: int) -> str:
    return load().zero_status_string(status).decode()
