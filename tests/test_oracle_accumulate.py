"""Pins for the oracle's fp32 gradient accumulation over micro-steps (not gpu).

Femtotron dev log #5 (no_sync micro-steps accumulate before the one reduce)
and the source guide's Megatron main_grad (fp32 accumulation).  Expected
values are exact sums and hand-worked rounding cases."""

import numpy as np
import torch

import synth_inputs as si
from oracle import Hyper


def _bf(values):
    t = torch.tensor(np.asarray(values, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def test_first_micro_step_discards_old_contents(oracle_lib):
    acc = [np.full(4, np.nan, np.float32), np.full(4, 7.0, np.float32)]
    oracle_lib.accumulate([_bf([1, 2, 3, 4]), _bf([-1, -0.5, 0.25, 8])], acc, first=True)
    assert np.array_equal(acc[0], [1, 2, 3, 4]) and np.array_equal(acc[1], [-1, -0.5, 0.25, 8])


def test_exact_sums(oracle_lib):
    # k micro-steps of j/256 (exact in bf16 and their sums exact in fp32)
    acc = [np.zeros(8, np.float32)]
    vals = np.arange(8, dtype=np.float32) / 256
    for k in range(100):
        oracle_lib.accumulate([_bf(vals)], acc, first=(k == 0))
    assert np.array_equal(acc[0], vals * 100)


def test_fp32_keeps_what_bf16_would_lose(oracle_lib):
    # 1 + 256 micro-steps of 2^-9: in fp32 the total 1.5 is exact; a bf16
    # accumulator (8 significant bits) would stay at 1.0
    acc = [np.zeros(1, np.float32)]
    oracle_lib.accumulate([_bf([1.0])], acc, first=True)
    for _ in range(256):
        oracle_lib.accumulate([_bf([2.0 ** -9])], acc, first=False)
    assert acc[0][0] == 1.5


def test_micro_step_order(oracle_lib):
    # 2^24, then 1, then 1: each +1 is a tie that rounds back to 2^24 (even);
    # summing the ones first would give 2^24 + 2
    acc = [np.zeros(1, np.float32)]
    for k, v in enumerate([2.0 ** 24, 1.0, 1.0]):
        oracle_lib.accumulate([_bf([v])], acc, first=(k == 0))
    assert acc[0][0] == 2.0 ** 24


def test_accumulated_step_equals_fp32_grad_step(oracle_lib):
    # accumulating K micro-steps and stepping on the fp32 sums is the fp32-gradient step
    pl = si.from_units([40, 9])
    n, K = 3, 4
    lay = oracle_lib.layout(pl.numel, pl.unit, n, 2)
    rng = np.random.default_rng(1)
    micro = [[_bf(np.concatenate([rng.normal(0, 1e-2, lay.total_padded - 2), [0, 0]]).astype(np.float32))
              for _ in range(n)] for _ in range(K)]
    acc = [np.zeros(lay.total_padded, np.float32) for _ in range(n)]
    for k in range(K):
        oracle_lib.accumulate(micro[k], acc, first=(k == 0))
    manual = [np.zeros(lay.total_padded, np.float32) for _ in range(n)]
    for r in range(n):
        for k in range(K):
            x = (micro[k][r].astype(np.uint32) << 16).view(np.float32)
            manual[r] = x.copy() if k == 0 else (manual[r] + x).astype(np.float32)
    for a, b in zip(acc, manual):
        assert np.array_equal(a, b)
    init = [rng.normal(0, 0.02, k).astype(np.float32) for k in pl.numel]
    st = oracle_lib.make_master(pl.numel, lay, init)
    oracle_lib.zero_step(Hyper(n_ranks=n, grad_dtype="fp32"), 2, 1, lay, acc, *st)
    assert np.all(np.isfinite(st[0]))
