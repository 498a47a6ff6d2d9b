"""Pins for the oracle's global-norm gradient clipping (not gpu).

ClipGradNorm runs on the fp32 (reduced) gradient before AdamW (Femtotron dev
logs #4/#5; the source guide's --clip-grad 1.0 / gradient_clipping 1.0).
Expected values are closed forms: Pythagorean norms, the clip coefficient's
definition at its edge cases, and Adam trajectories under a constant clip.
"""

import math

import numpy as np
import pytest
import torch

import synth_inputs as si
from oracle import Hyper


def _bf(values):
    t = torch.tensor(np.asarray(values, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def f32(x):
    return float(np.float32(x))


def test_norm_pythagorean(oracle_lib):
    h = Hyper(n_ranks=1)
    assert oracle_lib.grad_norm(h, [_bf([3.0, 4.0])]) == 5.0
    assert oracle_lib.grad_norm(h, [_bf([2.0, 3.0, 6.0])]) == 7.0  # 4 + 9 + 36 = 49
    # all-equal vector of 16: a * sqrt(16)
    assert oracle_lib.grad_norm(h, [_bf([0.375] * 16)]) == 1.5


def test_norm_is_of_the_reduced_gradient(oracle_lib):
    # replicas [6, 8] and [0, 0] average to [3, 4]: norm 5 (not the replicas' norms)
    h = Hyper(n_ranks=2)
    assert oracle_lib.grad_norm(h, [_bf([6.0, 8.0]), _bf([0.0, 0.0])]) == 5.0
    h4 = Hyper(n_ranks=4, grad_dtype="fp32")
    g = [np.array([12.0, 16.0], np.float32), np.zeros(2, np.float32), np.zeros(2, np.float32),
         np.zeros(2, np.float32)]
    assert oracle_lib.grad_norm(h4, g) == 5.0


def test_norm_permutation_invariant_on_exact_sums(oracle_lib):
    rng = np.random.default_rng(3)
    vals = rng.integers(-64, 64, 100).astype(np.float32)  # integer squares sum exactly in fp64
    h = Hyper(n_ranks=1)
    a = oracle_lib.grad_norm(h, [_bf(vals)])
    b = oracle_lib.grad_norm(h, [_bf(vals[::-1].copy())])
    assert a == b == math.sqrt(float(np.sum(vals.astype(np.float64) ** 2)))


def test_norm_sum_is_compensated(oracle_lib):
    # one square of 2^54 then a thousand squares of 1: a plain running fp64
    # sum stays at 2^54 (its ulp there is 4), the exact sum 2^54 + 1000 is
    # representable and is what the norm must be the square root of
    h = Hyper(n_ranks=1)
    g = _bf([2.0 ** 27] + [1.0] * 1000)
    assert oracle_lib.grad_norm(h, [g]) == math.sqrt(float(2 ** 54 + 1000))
    assert math.sqrt(float(2 ** 54 + 1000)) != 2.0 ** 27


def test_norm_of_non_finite_gradients(oracle_lib):
    # sqrt(sum g^2) under IEEE arithmetic: an infinite gradient makes the norm
    # +inf, a NaN makes it NaN (NaN wins over inf); the largest finite bf16
    # values square without overflow in fp64.
    h = Hyper(n_ranks=1)
    assert oracle_lib.grad_norm(h, [_bf([3.0, np.inf, 4.0])]) == math.inf
    assert oracle_lib.grad_norm(h, [_bf([-np.inf, 1.0])]) == math.inf
    assert math.isnan(oracle_lib.grad_norm(h, [_bf([3.0, np.nan, 4.0])]))
    assert math.isnan(oracle_lib.grad_norm(h, [_bf([np.inf, np.nan])]))
    top = np.array([0x7F7F], np.uint16)  # largest finite bf16, 3.3895e38
    top_f = float((top.astype(np.uint32) << 16).view(np.float32)[0])
    assert oracle_lib.grad_norm(h, [np.concatenate([top, top])]) == math.sqrt(2.0) * top_f
    # replicas whose fp32 sum overflows: the reduced gradient itself is inf
    h2 = Hyper(n_ranks=2)
    assert oracle_lib.grad_norm(h2, [top, top]) == math.inf
    # the coefficient: an infinite norm scales everything to 0, a NaN norm
    # gives a NaN coefficient (the cap at 1 passes NaN through)
    assert oracle_lib.clip_coef(math.inf, 1.0) == 0.0
    assert math.isnan(oracle_lib.clip_coef(math.nan, 1.0))


def test_non_finite_clip_follows_torch_clip_grad_norm(oracle_lib):
    # torch's own clip_grad_norm_ (the routine whose convention the clipping
    # follows) on the reduced gradient: a NaN anywhere makes every clipped
    # gradient NaN; an inf makes that element NaN (inf * 0) and every other 0.
    # The oracle's clipped first step must show the same pattern: a NaN
    # gradient turns the whole state NaN, an inf gradient that element only
    # (the others see g = 0: m = v = 0 and the weight keeps its value).
    h = Hyper(n_ranks=1, grad_dtype="fp32")
    for bad in (math.nan, math.inf):
        g = np.array([0.5, -0.25, bad, 2.0], np.float32)
        p = torch.nn.Parameter(torch.zeros(4))
        p.grad = torch.from_numpy(g.copy())
        torch.nn.utils.clip_grad_norm_([p], max_norm=1.0)
        clipped = p.grad.numpy()
        lay = oracle_lib.layout([4], [0], 1, 1)
        w0 = np.array([1.0, 2.0, 3.0, 4.0], np.float32)
        master, m, v, p16 = oracle_lib.make_master([4], lay, [w0])
        oracle_lib.zero_step(h, 1, 1, lay, [g], master, m, v, p16, max_norm=1.0)
        # the oracle's clipped gradient is m / (1 - beta1) after one step from m = 0
        assert np.array_equal(np.isnan(clipped), np.isnan(m)), (bad, clipped, m)
        finite = ~np.isnan(clipped)
        assert np.array_equal(clipped[finite] == 0.0, m[finite] == 0.0)
        assert np.array_equal(np.isnan(master), np.isnan(clipped))


def test_clip_coefficient(oracle_lib):
    assert oracle_lib.clip_coef(5.0, 1.0) == f32(1.0 / (5.0 + 1e-6))
    assert oracle_lib.clip_coef(0.5, 1.0) == 1.0          # below the threshold: untouched
    assert oracle_lib.clip_coef(0.0, 1.0) == 1.0          # zero gradient
    assert oracle_lib.clip_coef(1.0, 1.0) < 1.0           # norm == max_norm still scales (by 1/(1+1e-6))
    assert oracle_lib.clip_coef(1.0, 1.0) == f32(1.0 / (1.0 + 1e-6))


def _state(n):
    return (np.zeros(n, np.float32), np.zeros(n, np.float32), np.zeros(n, np.float32), np.zeros(n, np.uint16))


def test_clipped_first_step(oracle_lib):
    # g = [3, 4], max_norm 1: g' = g / (5 + 1e-6) (one fp32 multiply by the fp32
    # coefficient).  m1 = (1-b1) g', v1 = (1-b2) g'^2; the Adam step itself is
    # scale-invariant: w1 = w0 - lr g'/(|g'| + eps) ~ w0 - lr sign(g).
    pl = si.from_units([2])
    lay = oracle_lib.layout(pl.numel, pl.unit, 1, 1)
    h = Hyper(n_ranks=1)
    master, m, v, p16 = oracle_lib.make_master(pl.numel, lay, [np.array([1.0, -1.0], np.float32)])
    norm = oracle_lib.zero_step(h, 1, 1, lay, [_bf([3.0, 4.0])], master, m, v, p16, max_norm=1.0)
    assert norm == 5.0
    c = f32(1.0 / (5.0 + 1e-6))
    b1, b2, lr, eps = f32(0.9), f32(0.999), f32(1e-3), f32(1e-8)
    for k, g in enumerate([3.0, 4.0]):
        gp = f32(g * c)
        assert abs(m[k] - (1 - b1) * gp) <= np.spacing(np.float32((1 - b1) * gp))
        assert abs(v[k] - (1 - b2) * gp * gp) <= 2 * np.spacing(np.float32((1 - b2) * gp * gp))
        w0 = [1.0, -1.0][k]
        exact = w0 - lr * gp / (abs(gp) + eps)
        assert abs(master[k] - exact) <= 2 * np.spacing(np.abs(np.float32(exact)))


def test_unclipped_when_below_threshold(oracle_lib):
    pl = si.from_units([2])
    lay = oracle_lib.layout(pl.numel, pl.unit, 2, 2)
    h = Hyper(n_ranks=2)
    g = [_bf([0.25, 0.5]), _bf([0.25, 0.5])]
    a = oracle_lib.make_master(pl.numel, lay, [np.array([1.0, 2.0], np.float32)])
    b = tuple(x.copy() for x in a)
    norm = oracle_lib.zero_step(h, 2, 1, lay, g, *a, max_norm=10.0)
    assert abs(norm - math.sqrt(0.25 ** 2 + 0.5 ** 2)) < 1e-15
    oracle_lib.zero_step(h, 2, 1, lay, g, *b)
    for x, y in zip(a, b):
        assert np.array_equal(x, y)


def test_constant_clipped_gradient_trajectory(oracle_lib):
    # The same gradient every step, always clipped by the same c: m_t =
    # (1-b1^t) g', v_hat = g'^2, each step moves w by -lr g'/(|g'| + eps).
    pl = si.from_units([2])
    lay = oracle_lib.layout(pl.numel, pl.unit, 1, 3)
    h = Hyper(n_ranks=1)
    st = oracle_lib.make_master(pl.numel, lay, [np.array([0.5, 0.5], np.float32)])
    c = f32(2.0 / (5.0 + 1e-6))
    b1, lr, eps = f32(0.9), f32(1e-3), f32(1e-8)
    for t in range(1, 11):
        norm = oracle_lib.zero_step(h, 3, t, lay, [_bf([-3.0, 4.0])], *st, max_norm=2.0)
        assert norm == 5.0
        for k, g in enumerate([-3.0, 4.0]):
            gp = f32(g * c)
            assert abs(st[1][k] - (1 - b1 ** t) * gp) <= 4 * t * np.spacing(np.abs(np.float32(gp)))
            exact = 0.5 - t * lr * gp / (abs(gp) + eps)
            assert abs(st[0][k] - exact) <= (t + 1) * np.spacing(np.abs(np.float32(exact)))


def test_clipped_stages_bit_identical_to_dp(oracle_lib):
    # the norm runs over the flat element order; pads add exact zeros, so the
    # padded sharded layouts clip exactly like unpadded data parallelism
    pl = si.from_units([1552, 7, 33])
    n = 3
    rng = np.random.default_rng(9)
    init = [rng.normal(0, 0.02, k).astype(np.float32) for k in pl.numel]
    grads_per_param = [[_bf(rng.normal(0, 1.0, k)) for k in pl.numel] for _ in range(n)]
    results = {}
    for stage in (0, 1, 2, 3):
        lay = oracle_lib.layout(pl.numel, pl.unit, n, stage)
        flat = []
        for r in range(n):
            f = np.zeros(lay.total_padded, np.uint16)
            for p, k in enumerate(pl.numel):
                f[lay.param_offset[p]:lay.param_offset[p] + k] = grads_per_param[r][p]
            flat.append(f)
        st = oracle_lib.make_master(pl.numel, lay, init)
        h = Hyper(n_ranks=n)
        norms = []
        for t in range(1, 4):
            if stage == 0:
                norms.append(oracle_lib.dp_step(h, t, flat, *st, max_norm=1.0))
            else:
                norms.append(oracle_lib.zero_step(h, stage, t, lay, flat, *st, max_norm=1.0))
        real = [np.concatenate([a[lay.param_offset[p]:lay.param_offset[p] + k] for p, k in enumerate(pl.numel)])
                for a in st]
        results[stage] = (norms, real)
    for stage in (1, 2, 3):
        assert results[stage][0] == results[0][0]
        for a, b in zip(results[0][1], results[stage][1]):
            assert np.array_equal(a.view(np.uint8), b.view(np.uint8))
    assert results[0][0][0] > 1.0  # the clip was active
