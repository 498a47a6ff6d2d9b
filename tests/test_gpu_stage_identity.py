"""ZeRO-1/2/3 GPU runs are bit-identical to the unsharded (stage 0) GPU run
on every real parameter element, pads included in the sharded layouts
(CMU 15-779 Lecture 13 notes §3.4: ZeRO computes exactly what data
parallelism computes when the summation order is fixed)."""

import numpy as np
import pytest
import torch

import synth_inputs as si
from gpu_common import ensure_built, make_problem, run_gpu, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


def _per_param(fs, pl):
    arrays = [to_np(fs.master), to_np(fs.exp_avg), to_np(fs.exp_avg_sq), to_np(fs.param16)]
    out = []
    for a in arrays:
        out.append(np.concatenate([a[fs.param_offset(p):fs.param_offset(p) + k] for p, k in enumerate(pl.numel)]))
    return out


CASES = [
    ("toy_mlp_n4", si.toy_mlp(), 4, "bf16"),
    ("lecture_mlp_n3", si.lecture_mlp(), 3, "bf16"),
    ("odd_n16", si.from_units([1, 7, 15, 17, 33, 4099]), 16, "bf16"),
    ("fp32_n5", si.from_units([11, 1, 2049]), 5, "fp32"),
]


@pytest.mark.parametrize("name,pl,n,gd", CASES, ids=[c[0] for c in CASES])
def test_sharded_equals_unsharded(name, pl, n, gd):
    results = {}
    for stage in (0, 1, 2, 3):
        pb = make_problem(pl, n, stage, grad_dtype=gd, steps=10, seed=21)
        fs = run_gpu(pb, mode="units")
        results[stage] = _per_param(fs, pl)
        # pads of the sharded layouts stay exactly zero
        for i in range(fs.n_units):
            numel, padded, shard, base = fs.layout(i)
            for buf in (fs.master, fs.exp_avg, fs.exp_avg_sq, fs.param16):
                assert not torch.any(buf[base + numel:base + padded].float() != 0).item()
        fs.close()
    for stage in (1, 2, 3):
        for a, b in zip(results[0], results[stage]):
            assert np.array_equal(a.view(np.uint8), b.view(np.uint8)), (name, stage)
