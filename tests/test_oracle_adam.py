"""Pins for the oracle's reduce, Adam/AdamW and bf16 cast (not gpu).

Every expected value is a closed form derived from the update rule of the
lecture notes §2.1 (not a restatement of the recurrence), a hand-computed
special case, or an independent library routine (torch's bf16 conversion).
"""

import math

import numpy as np
import pytest
import torch

from oracle import Hyper


def bits(x):
    return np.float32(x).view(np.uint32)


def f32_from_bits(u):
    return np.uint32(u).view(np.float32)


def bf16_bits_of(values):
    """torch's own fp32 -> bf16 (round to nearest even) as uint16 bit patterns."""
    t = torch.tensor(np.asarray(values, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


# ---------------------------------------------------------------- bf16 cast --
def test_bf16_round_matches_torch_random(oracle_lib):
    rng = np.random.default_rng(0)
    raw = rng.integers(0, 2**32, size=200_000, dtype=np.uint64).astype(np.uint32)
    x = raw.view(np.float32)
    ours = oracle_lib.bf16_round(x)
    ref = bf16_bits_of(x)
    nan = np.isnan(x)
    assert np.array_equal(ours[~nan], ref[~nan])
    # NaN stays NaN
    back = ours[nan].astype(np.uint32) << 16
    assert np.all(np.isnan(back.view(np.float32)))


def test_bf16_round_special_cases(oracle_lib):
    cases = {
        0x3F808000: 0x3F80,  # 1 + 2^-8: exact tie, even neighbour below
        0x3F818000: 0x3F82,  # tie, odd below -> rounds up
        0x3F808001: 0x3F81,  # just above the tie
        0x3F807FFF: 0x3F80,  # just below the tie
        0x7F7FFFFF: 0x7F80,  # largest float rounds to +inf
        0xFF7FFFFF: 0xFF80,  # and to -inf
        0x7F800000: 0x7F80,  # +inf
        0x80000000: 0x8000,  # -0
        0x00000001: 0x0000,  # smallest denormal rounds to +0
        0x00008000: 0x0000,  # denormal tie -> even (0)
        0x00018000: 0x0002,  # denormal tie, odd below -> up
    }
    for src, want in cases.items():
        got = int(oracle_lib.bf16_round(f32_from_bits(src))[0])
        assert got == want, hex(src)
    nan_in = f32_from_bits(0x7F800001)
    got = int(oracle_lib.bf16_round(nan_in)[0])
    assert (got & 0x7F80) == 0x7F80 and (got & 0x7F) != 0


def test_bf16_widen_exact(oracle_lib):
    for h in [0x0000, 0x3F80, 0xBF80, 0x7F80, 0x0001, 0x4049]:
        assert bits(oracle_lib.bf16_widen([h])[0]) == h << 16


# ------------------------------------------------------------------ reduce --
def _bf(values):
    return bf16_bits_of(values)


def test_reduce_identical_replicas_is_exact(oracle_lib):
    rng = np.random.default_rng(1)
    x = _bf(rng.normal(0, 1e-2, 64))
    xf = (x.astype(np.uint32) << 16).view(np.float32)
    for n in (1, 2, 4, 8, 16):
        h = Hyper(n_ranks=n)
        for j in range(64):
            assert oracle_lib.reduce_element(h, [x] * n, j) == xf[j]


def test_reduce_rank_order(oracle_lib):
    # Replicas 2^24, 1, 1, 1 at N = 4.  In rank order each +1 is a tie that
    # rounds back to 2^24 (even), so the average is 2^22 exactly.  Summing in
    # reverse order would give 2^24 + 4 (-> 2^22 + 1); a pairwise tree
    # 2^24 + 2 (-> 2^22 + 0.5).
    g = [_bf([2.0 ** 24]), _bf([1.0]), _bf([1.0]), _bf([1.0])]
    h = Hyper(n_ranks=4)
    assert oracle_lib.reduce_element(h, g, 0) == 2.0 ** 22
    # The first operand is replica 0's value itself: with replica 0 at -0 and
    # N = 1 the sign of zero is kept.
    assert math.copysign(1.0, oracle_lib.reduce_element(Hyper(n_ranks=1), [_bf([-0.0])], 0)) == -1.0


def test_reduce_fp32_grads_and_scale(oracle_lib):
    h = Hyper(n_ranks=2, grad_dtype="fp32")
    g = [np.array([0.1], dtype=np.float32), np.array([0.3], dtype=np.float32)]
    want = (np.float32(0.1) + np.float32(0.3)) * np.float32(0.5)
    assert oracle_lib.reduce_element(h, g, 0) == want
    # N = 3: identical replicas give x within one ulp (1/3 is not exact in fp32)
    h3 = Hyper(n_ranks=3, grad_dtype="fp32")
    x = np.array([0.7], dtype=np.float32)
    got = np.float32(oracle_lib.reduce_element(h3, [x, x, x], 0))
    assert abs(int(bits(got)) - int(bits(x[0]))) <= 1


def test_step_scalars(oracle_lib):
    h = Hyper(lr=1e-3, beta1=0.9, beta2=0.999, weight_decay=0.1, adamw=True, n_ranks=8)
    s1 = oracle_lib.step_scalars(h, 1)
    # at t = 1 the bias corrections equal 1 - beta exactly
    assert s1["bc1"] == s1["one_minus_beta1"] == np.float32(1) - np.float32(0.9)
    assert s1["bc2"] == s1["one_minus_beta2"]
    assert s1["inv_n"] == np.float32(0.125)
    assert s1["decay"] == np.float32(1 - np.float64(np.float32(1e-3)) * np.float64(np.float32(0.1)))
    s10 = oracle_lib.step_scalars(h, 10)
    # 1 - beta^t of the fp32 betas, rounded once to fp32
    b1, b2 = float(np.float32(0.9)), float(np.float32(0.999))
    assert abs(s10["bc1"] - (1 - b1 ** 10)) <= 0.5 * np.spacing(np.float32(1 - b1 ** 10))
    assert abs(s10["bc2"] - (1 - b2 ** 10)) <= 0.5 * np.spacing(np.float32(1 - b2 ** 10))


# -------------------------------------------------------------------- Adam --
def _run(oracle_lib, h, w0, grads_per_step, m0=None, v0=None):
    """Runs the oracle window step over T steps on a tiny buffer; returns the w trace."""
    n = len(w0)
    w = np.array(w0, dtype=np.float32)
    m = np.zeros(n, np.float32) if m0 is None else np.array(m0, np.float32)
    v = np.zeros(n, np.float32) if v0 is None else np.array(v0, np.float32)
    p16 = np.zeros(n, np.uint16)
    trace = []
    for t, g in enumerate(grads_per_step, start=1):
        reps = [_bf(g)] * h.n_ranks if h.grad_dtype == "bf16" else [np.array(g, np.float32)] * h.n_ranks
        oracle_lib.step_window(h, t, reps, w, m, v, p16)
        trace.append((w.copy(), m.copy(), v.copy(), p16.copy()))
    return trace


def _ulp(x):
    return np.spacing(np.abs(np.float32(x))).astype(np.float64)


def f32(x):
    """The fp32 value the method runs on (hyper-parameters are fp32)."""
    return float(np.float32(x))


def test_adam_first_step_closed_form(oracle_lib):
    # m_1 = (1-b1) g, v_1 = (1-b2) g^2, so m_hat = g, v_hat = g^2 and
    # w_1 = w_0 - lr * g / (|g| + eps)   (close to w_0 - lr * sign g).
    g = [0.5, -0.25, 2.0, -3.0, 0.0078125, -1.0]
    w0 = [1.0, -2.0, 0.5, 0.25, 3.0, -0.125]
    h = Hyper(lr=1e-3, eps=1e-8, n_ranks=4)
    lr, eps, b1, b2 = f32(1e-3), f32(1e-8), f32(0.9), f32(0.999)
    (w, m, v, p16), = _run(oracle_lib, h, w0, [g])
    for k in range(len(g)):
        exact = w0[k] - lr * g[k] / (abs(g[k]) + eps)
        assert abs(w[k] - exact) <= 2 * _ulp(exact), k
        assert abs(m[k] - (1 - b1) * g[k]) <= _ulp((1 - b1) * g[k])
        assert abs(v[k] - (1 - b2) * g[k] ** 2) <= _ulp((1 - b2) * g[k] ** 2)
    assert np.array_equal(p16, bf16_bits_of(w))


def test_adam_constant_gradient_closed_form(oracle_lib):
    # With a constant g every step: m_t = (1 - b1^t) g and v_t = (1 - b2^t) g^2,
    # so the bias-corrected moments are g and g^2 at every t and each step
    # moves w by -lr g / (|g| + eps):  w_T = w_0 - T lr g / (|g| + eps).
    T = 10
    g = [0.5, -0.25, 0.0625, -2.0]
    w0 = [1.0, 1.0, -1.0, 0.5]
    h = Hyper(lr=1e-3, eps=1e-8, n_ranks=2)
    lr, eps, b1, b2 = f32(1e-3), f32(1e-8), f32(0.9), f32(0.999)
    trace = _run(oracle_lib, h, w0, [g] * T)
    for t, (w, m, v, _) in enumerate(trace, start=1):
        for k in range(len(g)):
            exact_w = w0[k] - t * lr * g[k] / (abs(g[k]) + eps)
            assert abs(w[k] - exact_w) <= (t + 1) * _ulp(exact_w), (t, k)
            exact_m = (1 - b1 ** t) * g[k]
            assert abs(m[k] - exact_m) <= 4 * t * _ulp(exact_m)
            exact_v = (1 - b2 ** t) * g[k] ** 2
            assert abs(v[k] - exact_v) <= 1e-6 * abs(exact_v) + 4 * t * _ulp(exact_v)


def test_adam_alternating_gradient_closed_form(oracle_lib):
    # g_t = g (-1)^(t-1).  Summing the geometric series:
    #   m_t = (1-b1) g (-1)^(t-1) (1 - (-b1)^t) / (1 + b1),  v_t = (1 - b2^t) g^2
    #   w_t = w_{t-1} - lr * [m_t / (1 - b1^t)] / (|g| + eps)
    T = 10
    g0 = [0.75, -0.375]
    w0 = [0.5, -0.5]
    h = Hyper(lr=1e-2, beta1=0.9, beta2=0.999, eps=1e-8, n_ranks=1)
    b1, b2, lr, eps = f32(0.9), f32(0.999), f32(1e-2), f32(1e-8)
    steps = [[x * (-1) ** (t - 1) for x in g0] for t in range(1, T + 1)]
    trace = _run(oracle_lib, h, w0, steps)
    w_exact = list(w0)
    for t, (w, m, v, _) in enumerate(trace, start=1):
        for k in range(len(g0)):
            m_t = (1 - b1) * g0[k] * (-1) ** (t - 1) * (1 - (-b1) ** t) / (1 + b1)
            assert abs(m[k] - m_t) <= 1e-6 * abs(m_t) + 4 * t * _ulp(m_t)
            v_t = (1 - b2 ** t) * g0[k] ** 2
            assert abs(v[k] - v_t) <= 1e-6 * abs(v_t)
            w_exact[k] -= lr * (m_t / (1 - b1 ** t)) / (abs(g0[k]) + eps)
            assert abs(w[k] - w_exact[k]) <= 1e-6 * abs(w_exact[k]) + (t + 1) * _ulp(w_exact[k]), (t, k)


def test_adam_single_impulse_closed_form(oracle_lib):
    # g at t = 1, then 0:  m_t = (1-b1) b1^(t-1) g,  v_t = (1-b2) b2^(t-1) g^2.
    T = 8
    g = [0.5, -1.5]
    w0 = [0.0, 0.0]
    h = Hyper(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, n_ranks=1)
    b1, b2, lr, eps = f32(0.9), f32(0.999), f32(1e-3), f32(1e-8)
    trace = _run(oracle_lib, h, w0, [g] + [[0.0, 0.0]] * (T - 1))
    w_exact = list(w0)
    for t, (w, m, v, _) in enumerate(trace, start=1):
        for k in range(2):
            m_t = (1 - b1) * b1 ** (t - 1) * g[k]
            v_t = (1 - b2) * b2 ** (t - 1) * g[k] ** 2
            assert abs(m[k] - m_t) <= 1e-6 * abs(m_t)
            assert abs(v[k] - v_t) <= 1e-6 * abs(v_t)
            m_hat, v_hat = m_t / (1 - b1 ** t), v_t / (1 - b2 ** t)
            w_exact[k] -= lr * m_hat / (math.sqrt(v_hat) + eps)
            assert abs(w[k] - w_exact[k]) <= 1e-5 * abs(w_exact[k]), (t, k)


def test_adam_epsilon_outside_sqrt(oracle_lib):
    # |g| = eps at t = 1: the step is lr * g / (|g| + eps) = lr / 2 exactly
    # (eps inside the sqrt would give lr / sqrt(1 + 1/eps) instead).
    eps = 2.0 ** -20
    h = Hyper(lr=2.0 ** -10, eps=eps, n_ranks=1)
    (w, _, _, _), = _run(oracle_lib, h, [1.0, -1.0], [[eps, -eps]])
    assert w[0] == np.float32(1.0 - 2.0 ** -11)
    assert w[1] == np.float32(-1.0 + 2.0 ** -11)


def test_adamw_decoupled_decay_closed_form(oracle_lib):
    # Zero gradient: the Adam part is 0 / (0 + eps) = 0, so only the decoupled
    # decay acts and w_T = w_0 (1 - lr wd)^T, rounded each step.  (An L2 decay
    # folded into g would instead move w by about lr per step.)
    lr, wd, T = 2.0 ** -4, 2.0 ** -2, 6   # 1 - lr*wd = 1 - 2^-6, exact in fp32
    h = Hyper(lr=lr, weight_decay=wd, adamw=True, n_ranks=2)
    trace = _run(oracle_lib, h, [1.0, -0.5], [[0.0, 0.0]] * T)
    d = 1 - lr * wd
    for t, (w, m, v, _) in enumerate(trace, start=1):
        assert abs(w[0] - d ** t) <= t * _ulp(d ** t)
        assert abs(w[1] + 0.5 * d ** t) <= t * _ulp(0.5 * d ** t)
        assert np.all(m == 0) and np.all(v == 0)


def test_adam_without_wd_ignores_decay(oracle_lib):
    h = Hyper(lr=0.1, weight_decay=0.5, adamw=False, n_ranks=1)
    (w, _, _, _), = _run(oracle_lib, h, [1.0], [[0.0]])
    assert w[0] == 1.0


def test_fp32_update_not_eaten(oracle_lib):
    # The reason for the fp32 master (notes §2.2): an update of 1e-6 on a
    # weight of 1.0 survives in fp32 (the bf16 copy does not move).
    h = Hyper(lr=1e-6, n_ranks=1)
    (w, _, _, p16), = _run(oracle_lib, h, [1.0], [[0.5]])
    assert w[0] < 1.0
    assert p16[0] == 0x3F80


def test_pads_stay_zero(oracle_lib):
    # zero master, zero grads, zero moments stay exactly zero, with AdamW too
    h = Hyper(lr=1e-2, weight_decay=0.1, adamw=True, n_ranks=3)
    trace = _run(oracle_lib, h, [0.0, 0.0], [[0.0, 0.0]] * 5)
    for w, m, v, p16 in trace:
        assert np.all(w == 0) and np.all(m == 0) and np.all(v == 0) and np.all(p16 == 0)
