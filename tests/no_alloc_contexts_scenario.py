"""Scenario run by tests/test_zz_no_alloc.py in a subprocess (not collected by
pytest): the library used from several CUDA contexts of one GPU — the
primary context, a second context made with the driver API, a third made
after the second was destroyed, and the primary again.  No torch: every
device buffer is allocated with the driver API in the context that uses it,
so nothing of one context is ever handed to another.

In every context:
  * the allocation-free clip (zero_clip_grad_norm_static) must give the norm
    and, after the step, the state that the clip with a caller workspace
    gives on the same inputs — its scratch must be the current context's own
    array, found by a lookup made in that context;
  * a step over 2^23 + 1,000 elements at N = 8 bf16 (a tile-staged kernel,
    whose raised shared-memory limit belongs to the context) must succeed and
    give the same state as in the primary context.
Exit status 0 on success."""

import ctypes
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(HERE))

from zero_sharded_mixed_flatparameter_gb300 import binding as B, build_lib  # noqa: E402

B.load(build_lib.build())
cu = ctypes.CDLL("libcuda.so.1")
VP, U64 = ctypes.c_void_p, ctypes.c_uint64


def ck(r, what):
    if r != 0:
        raise RuntimeError(f"{what}: CUresult {r}")


class Buffers:
    """Device allocations of the current context, freed together."""

    def __init__(self):
        self.ptrs = []

    def alloc(self, nbytes):
        p = U64()
        ck(cu.cuMemAlloc_v2(ctypes.byref(p), ctypes.c_size_t(max(nbytes, 16))), "cuMemAlloc")
        self.ptrs.append(p.value)
        return p.value

    def upload(self, host):
        host = np.ascontiguousarray(host)
        p = self.alloc(host.nbytes)
        ck(cu.cuMemcpyHtoD_v2(U64(p), host.ctypes.data_as(VP), ctypes.c_size_t(host.nbytes)), "cuMemcpyHtoD")
        return p

    def free(self):
        for p in self.ptrs:
            cu.cuMemFree_v2(U64(p))
        self.ptrs = []


def download(ptr, n, dtype):
    out = np.empty(n, dtype)
    ck(cu.cuMemcpyDtoH_v2(out.ctypes.data_as(VP), U64(ptr), ctypes.c_size_t(out.nbytes)), "cuMemcpyDtoH")
    return out


def bf16_bits(x):
    return (x.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)


def flat_problem(numel, n, seed):
    rng = np.random.default_rng(seed)
    cfg = B.make_config(2, n)
    plan = B.zero_plan(cfg, numel, list(range(len(numel))))
    padded, _ = B.zero_padded_numel(plan)
    offsets = [B.zero_param_offset(plan, p) for p in range(len(numel))]
    B.zero_destroy(plan)
    init = [rng.normal(0, 0.02, k).astype(np.float32) for k in numel]
    grads = []
    for _ in range(n):
        g = np.zeros(padded, np.uint16)
        for off, k in zip(offsets, numel):
            g[off:off + k] = bf16_bits(rng.normal(0, 1e-2, k))
        grads.append(g)
    return cfg, padded, init, grads


def make_ctx(bufs, cfg, numel, padded, init, grads):
    state = [bufs.alloc(4 * padded) for _ in range(3)] + [bufs.alloc(2 * padded)]
    ctx = B.zero_make_master(cfg, numel, list(range(len(numel))), [bufs.upload(p) for p in init], *state)
    return ctx, state, [bufs.upload(g) for g in grads]


def read_state(state, padded):
    return [download(p, padded, np.float32) for p in state[:3]] + [download(state[3], padded, np.uint16)]


def clip_twins(label):
    """Workspace clip and static-scratch clip on twin contexts, two steps."""
    numel = [40_000, 1552, 7]
    cfg, padded, init, grads = flat_problem(numel, 4, 5)
    bufs = Buffers()
    try:
        ctx_ws, st_ws, g_ws = make_ctx(bufs, cfg, numel, padded, init, grads)
        ctx_st, st_st, g_st = make_ctx(bufs, cfg, numel, padded, init, grads)
        ws_bytes = B.zero_clip_workspace_bytes(ctx_ws)
        ws = bufs.alloc(ws_bytes)
        for t in (1, 2):
            B.zero_reduce_grads(ctx_ws, -1, g_ws)
            B.zero_reduce_grads(ctx_st, -1, g_st)
            B.zero_clip_grad_norm(ctx_ws, 0.5, ws, ws_bytes)
            B.zero_clip_grad_norm_static(ctx_st, 0.5)
            n_ws, n_st = B.zero_grad_norm(ctx_ws), B.zero_grad_norm(ctx_st)
            assert n_ws > 0.5 and abs(n_st - n_ws) <= 1e-12 * n_ws, (label, t, n_ws, n_st)
            for c in (ctx_ws, ctx_st):
                B.zero_step(c)
                B.zero_post_step(c)
        a, b = read_state(st_ws, padded), read_state(st_st, padded)
        for x, y in zip(a, b):
            assert np.array_equal(x.view(np.uint8), y.view(np.uint8)), f"{label}: static-scratch clip state differs"
        for c in (ctx_ws, ctx_st):
            B.zero_destroy(c)
    finally:
        bufs.free()
    print("ok", label, "clip", flush=True)


def staged_step(label):
    numel = [2 ** 23 + 1000]
    cfg, padded, init, grads = flat_problem(numel, 8, 6)
    bufs = Buffers()
    try:
        ctx, state, g = make_ctx(bufs, cfg, numel, padded, init, grads)
        B.zero_reduce_grads(ctx, -1, g)
        B.zero_step(ctx)
        B.zero_post_step(ctx)
        out = read_state(state, padded)
        B.zero_destroy(ctx)
    finally:
        bufs.free()
    print("ok", label, "staged step", flush=True)
    return out


def main():
    ck(cu.cuInit(0), "cuInit")
    dev = ctypes.c_int()
    ck(cu.cuDeviceGet(ctypes.byref(dev), 0), "cuDeviceGet")
    primary = VP()
    ck(cu.cuDevicePrimaryCtxRetain(ctypes.byref(primary), dev), "cuDevicePrimaryCtxRetain")
    ck(cu.cuCtxPushCurrent_v2(primary), "push primary")
    clip_twins("primary context")
    ref = staged_step("primary context")
    popped = VP()
    ck(cu.cuCtxPopCurrent_v2(ctypes.byref(popped)), "pop primary")
    for label in ("second context", "third context (after the second was destroyed)"):
        c = VP()
        ck(cu.cuCtxCreate_v2(ctypes.byref(c), 0, dev), "cuCtxCreate")  # becomes current
        clip_twins(label)
        got = staged_step(label)
        for x, y in zip(ref, got):
            assert np.array_equal(x.view(np.uint8), y.view(np.uint8)), f"{label}: staged step differs"
        ck(cu.cuCtxDestroy_v2(c), "cuCtxDestroy")
    ck(cu.cuCtxPushCurrent_v2(primary), "push primary again")
    clip_twins("primary context again")
    ck(cu.cuCtxPopCurrent_v2(ctypes.byref(popped)), "pop primary")
    cu.cuDevicePrimaryCtxRelease_v2(dev)
    print("all contexts ok", flush=True)
    return 0


if __name__ == "__main__":
    sys.exit(main())
