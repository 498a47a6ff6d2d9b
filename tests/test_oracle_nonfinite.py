"""Pins of the oracle's count of non-finite reduced gradients (the overflow
check that DeepSpeed's ZeRO step makes before clipping and updating, source
guide §4.3): hand-made cases whose classification follows from IEEE
arithmetic alone, and planted non-finite values counted by position."""

import numpy as np

from oracle import Hyper

INF, NINF, NAN = np.uint16(0x7F80), np.uint16(0xFF80), np.uint16(0x7FC0)
MAX, NMAX = np.uint16(0x7F7F), np.uint16(0xFF7F)  # largest finite bf16 (3.39e38), negated
ONE, TWO, THREE, FOUR = np.uint16(0x3F80), np.uint16(0x4000), np.uint16(0x4040), np.uint16(0x4080)
ZERO = np.uint16(0)


def test_hand_made_bf16_cases(oracle_lib):
    r0 = np.array([ONE, INF, TWO, NAN, MAX, NMAX, THREE, INF, ZERO], np.uint16)
    r1 = np.array([ONE, ONE, NINF, ONE, MAX, MAX, FOUR, NINF, ZERO], np.uint16)
    # 1+1 finite; inf+1 inf; 2-inf -inf; NaN+1 NaN; max+max overflows to inf;
    # -max+max = 0; 3+4 finite; inf-inf NaN; 0+0 finite  -> 5 non-finite
    assert oracle_lib.nonfinite_count(Hyper(n_ranks=2), [r0, r1]) == 5


def test_rank_order_decides_an_overflow(oracle_lib):
    # (max + max) overflows before -max is added: inf in rank order 0, 1, 2;
    # -max first would have kept the sum finite
    h = Hyper(n_ranks=3)
    assert oracle_lib.nonfinite_count(h, [np.array([MAX]), np.array([MAX]), np.array([NMAX])]) == 1
    assert oracle_lib.nonfinite_count(h, [np.array([MAX]), np.array([NMAX]), np.array([MAX])]) == 0
    # the fp32 sum overflows although the average would fit: it is counted
    half_max = np.uint16(0x7EFF)  # 1.69e38
    assert oracle_lib.nonfinite_count(h, [np.array([MAX]), np.array([half_max]), np.array([ZERO])]) == 1


def test_fp32_replicas(oracle_lib):
    h = Hyper(n_ranks=2, grad_dtype="fp32")
    r0 = np.array([3.0e38, 1.0, np.inf, np.nan, -3.0e38], np.float32)
    r1 = np.array([3.0e38, 2.0, -1.0, 0.0, 3.0e38], np.float32)
    assert oracle_lib.nonfinite_count(h, [r0, r1]) == 3
    # N = 1: the reduced gradient is the gradient
    assert oracle_lib.nonfinite_count(Hyper(n_ranks=1, grad_dtype="fp32"), [r0]) == 2


def test_planted_positions(oracle_lib):
    rng = np.random.default_rng(5)
    n, N = 100_000, 4
    reps = [rng.normal(0, 1e-2, n).astype(np.float32) for _ in range(N)]
    h = Hyper(n_ranks=N, grad_dtype="fp32")
    assert oracle_lib.nonfinite_count(h, reps) == 0
    pos = rng.choice(n, 37, replace=False)
    for k, p in enumerate(pos):
        reps[k % N][p] = (np.inf, -np.inf, np.nan)[k % 3]
    # two planted values may share no position (replace=False), so 37 positions
    assert oracle_lib.nonfinite_count(h, reps) == 37
