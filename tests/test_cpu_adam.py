"""ZeRO-Offload's CPU Adam (``zero_cpu_adam``) against the oracle, on the host.

CMU 15-779 Lecture 13 notes §7.2: in ZeRO-Offload the fp32 state lives in
host memory and a SIMD + multi-threaded CPU Adam updates it.  The library's
host Adam must give exactly the device step's result, which the oracle's
window step defines for one fp32 replica (the reduced gradient itself: x 1/1
and x clip 1 are exact).  No CUDA call is made, so this runs without a GPU.
"""

from __future__ import annotations

import ctypes

import numpy as np
import pytest

import oracle
from gpu_common import assert_bit_exact


@pytest.fixture(scope="module")
def B():
    from zero_sharded_mixed_flatparameter_gb300 import binding, build_lib
    build_lib.build()
    binding.load()
    return binding


def _addr(a: np.ndarray) -> int:
    return a.ctypes.data_as(ctypes.c_void_p).value or 0


def _state(n, seed):
    rng = np.random.default_rng(seed)
    master = rng.normal(0.0, 0.02, n).astype(np.float32)
    return master, np.zeros(n, np.float32), np.zeros(n, np.float32), np.zeros(n, np.uint16)


def _run_both(B, hyper_kw, n, steps, threads, seed, grads=None):
    cfg = B.make_config(1, 1, "fp32", **hyper_kw)
    h = oracle.Hyper(n_ranks=1, grad_dtype="fp32", **hyper_kw)
    rng = np.random.default_rng(seed + 1)
    ours = _state(n, seed)
    ref = tuple(x.copy() for x in ours)
    for t in range(1, steps + 1):
        g = grads[t - 1] if grads is not None else rng.normal(0.0, 1e-2, n).astype(np.float32)
        B.zero_cpu_adam(cfg, t, _addr(g), *(_addr(x) for x in ours), n, threads)
        oracle.step_window(h, t, [g.copy()], *ref)
    return ours, ref


@pytest.mark.parametrize("n", [1, 7, 63, 64, 65, 1000, 100_003])
@pytest.mark.parametrize("threads", [1, 3, 8])
def test_matches_oracle_bit_exact(B, n, threads):
    ours, ref = _run_both(B, {}, n, 10, threads, seed=n + threads)
    for name, a, b in zip(("master", "m", "v", "param16"), ours, ref):
        assert_bit_exact(a, b, f"n={n} threads={threads} {name}")


@pytest.mark.parametrize("hyper", [dict(adamw=True, weight_decay=0.1, lr=3e-4),
                                   dict(beta1=0.8, beta2=0.95, eps=1e-6, lr=1e-2),
                                   dict(beta1=0.0, beta2=0.0, eps=0.0, lr=1.0)])
def test_hyperparameters(B, hyper):
    ours, ref = _run_both(B, hyper, 4099, 6, 4, seed=5)
    for name, a, b in zip(("master", "m", "v", "param16"), ours, ref):
        assert_bit_exact(a, b, f"{hyper} {name}")


def test_special_values(B):
    # zeros, signed zeros, tiny (subnormal squares), huge (overflowing
    # squares), inf and NaN gradients: every element still follows the oracle
    n = 64
    g = np.zeros(n, np.float32)
    g[1], g[2], g[3], g[4] = -0.0, 1e-30, -1e-40, 3e38
    g[5], g[6], g[7] = np.inf, -np.inf, np.nan
    g[8:] = np.linspace(-1, 1, n - 8, dtype=np.float32)
    ours, ref = _run_both(B, {}, n, 3, 2, seed=9, grads=[g, g[::-1].copy(), g])
    for name, a, b in zip(("master", "m", "v", "param16"), ours, ref):
        assert_bit_exact(a, b, f"special {name}")


def test_thread_count_does_not_change_results(B):
    cfg = B.make_config(1, 1, "fp32")
    outs = []
    for threads in (1, 2, 5, 16, 0):
        st = _state(50_001, 3)
        g = np.random.default_rng(4).normal(0, 1e-2, 50_001).astype(np.float32)
        B.zero_cpu_adam(cfg, 1, _addr(g), *(_addr(x) for x in st), 50_001, threads)
        outs.append(st)
    for st in outs[1:]:
        for a, b in zip(st, outs[0]):
            assert np.array_equal(a.view(np.uint32) if a.dtype == np.float32 else a,
                                  b.view(np.uint32) if b.dtype == np.float32 else b)


def test_errors(B):
    cfg = B.make_config(1, 1, "fp32")
    g, w, m, v, p = (np.zeros(8, np.float32),) * 4 + (np.zeros(8, np.uint16),)
    a = [_addr(x) for x in (g, w, m, v, p)]
    for bad in (dict(t=0), dict(n=-1), dict(threads=-1), dict(threads=5000)):
        kw = dict(t=1, n=8, threads=1)
        kw.update(bad)
        with pytest.raises(B.ZeroError) as e:
            B.zero_cpu_adam(cfg, kw["t"], *a, kw["n"], kw["threads"])
        assert e.value.status == B.ZERO_EINVAL
    with pytest.raises(B.ZeroError) as e:
        B.zero_cpu_adam(cfg, 1, 0, *a[1:], 8, 1)
    assert e.value.status == B.ZERO_EINVAL
    with pytest.raises(B.ZeroError) as e:
        B.zero_cpu_adam(cfg, 1, a[0] + 2, *a[1:], 4, 1)  # misaligned fp32 gradient
    assert e.value.status == B.ZERO_EINVAL
    bad_cfg = B.make_config(1, 1, "fp32", weight_decay=0.1)  # decay without adamw
    with pytest.raises(B.ZeroError):
        B.zero_cpu_adam(bad_cfg, 1, *a, 8, 1)
    B.zero_cpu_adam(cfg, 1, *a, 0, 1)  # n = 0 is a no-op
