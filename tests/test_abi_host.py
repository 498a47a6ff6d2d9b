"""The C-ABI library on the host (not gpu): it builds, loads, exports every
symbol the public header declares, and its host logic — FlatParameter layout,
ledger, config validation and the state machine of a plan-only context —
matches the oracle.  No device work is requested."""

import ctypes
import glob
import os
import re

import numpy as np
import pytest

import synth_inputs as si
from conftest import ROOT


@pytest.fixture(scope="session")
def B():
    from zero_sharded_mixed_flatparameter_gb300 import binding, build_lib
    build_lib.build()
    binding.load()
    return binding


def _declared_functions():
    names = []
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names += re.findall(r"\b(zero_[a-z0-9_]+)\s*\(", text)
    return sorted(set(names))


def test_exports_every_declared_symbol(B):
    declared = _declared_functions()
    assert len(declared) >= 15
    lib = ctypes.CDLL(B.LIB_PATH)
    for name in declared:
        assert hasattr(lib, name), name
    assert set(declared) == set(B.EXPORTED)


def test_status_strings(B):
    assert B.zero_status_string(0) == "ZERO_OK"
    assert B.zero_status_string(4) == "ZERO_ESTATE"


LAYOUTS = [
    (si.toy_mlp(), 4, 1), (si.lecture_mlp(), 3, 2), (si.lecture_mlp(), 4, 3),
    (si.from_units([1, 7, 15, 17, 0, 33]), 16, 3), (si.from_units([15]), 16, 1),
    (si.llama_2048_units(), 8, 3), (si.from_units([1552, 9]), 3, 0),
    (si.ParamList("mixed", [3, 2, 5, 0, 2], [0, 0, 2, 2, 3], list("abcde")), 4, 2),
]


@pytest.mark.parametrize("pl,n,stage", LAYOUTS)
def test_layout_matches_oracle(B, oracle_lib, pl, n, stage):
    cfg = B.make_config(stage, n)
    ctx = B.zero_plan(cfg, pl.numel, pl.unit)
    try:
        lay = oracle_lib.layout(pl.numel, pl.unit, n, stage)
        assert B.zero_num_units(ctx) == len(lay.unit_numel)
        padded, numel = B.zero_padded_numel(ctx)
        assert padded == lay.total_padded and numel == sum(pl.numel)
        for i in range(len(lay.unit_numel)):
            assert B.zero_layout(ctx, i) == (lay.unit_numel[i], lay.unit_padded[i], lay.unit_shard[i],
                                             lay.unit_base[i])
        for p in range(len(pl.numel)):
            assert B.zero_param_offset(ctx, p) == lay.param_offset[p]
        for s in range(4):
            # the ledger of stage s is that of the layout as stage s pads it
            lay_s = oracle_lib.layout(pl.numel, pl.unit, n, s)
            assert B.zero_state_bytes(ctx, s, n) == list(oracle_lib.state_bytes(lay_s.unit_padded, n, s))
        lay3 = oracle_lib.layout(pl.numel, pl.unit, n, 3)
        assert B.zero_stage3_peak_bytes(ctx) == oracle_lib.zero3_backward_peak(lay3.unit_padded, n)
    finally:
        B.zero_destroy(ctx)


def test_layout_random_vs_oracle(B, oracle_lib):
    rng = np.random.default_rng(17)
    for _ in range(200):
        k = int(rng.integers(0, 10))
        numel = rng.integers(0, 5000, k).tolist()
        unit = np.sort(rng.integers(0, 5, k)).tolist()
        if k:
            unit = [u - unit[0] for u in unit]
        n, stage = int(rng.integers(1, 17)), int(rng.integers(0, 4))
        ctx = B.zero_plan(B.make_config(stage, n), numel, unit)
        try:
            lay = oracle_lib.layout(numel, unit, n, stage) if k else None
            padded, _ = B.zero_padded_numel(ctx)
            assert padded == (lay.total_padded if lay else 0)
            for p in range(k):
                assert B.zero_param_offset(ctx, p) == lay.param_offset[p]
        finally:
            B.zero_destroy(ctx)


def test_zero3_peak_lecture_mlp(B):
    # CMU 15-779 Lecture 13 notes §11 Exercise 5: peak 161,632 B at unit 1,
    # steady 130,624 B for the zero.py MLP at N = 4.
    pl = si.lecture_mlp()
    ctx = B.zero_plan(B.make_config(3, 4), pl.numel, pl.unit)
    try:
        assert B.zero_stage3_peak_bytes(ctx) == (161_632, 1)
        assert B.zero_state_bytes(ctx, 3, 4) == [130_624] * 4
    finally:
        B.zero_destroy(ctx)


@pytest.mark.parametrize("ctx_stage", [0, 1, 2, 3])
def test_ledger_independent_of_the_context_stage(B, oracle_lib, ctx_stage):
    # Units whose sizes are not multiples of N: a stage-0 context does not pad
    # (F = 1), yet its stage-1..3 ledger must count the shards those stages
    # pad to a multiple of N (ceil(psi / N) per rank), exactly as a context of
    # that stage reports it.
    numel, unit, n = [1552, 7, 33, 1], [0, 1, 1, 2], 3
    ctx = B.zero_plan(B.make_config(ctx_stage, n), numel, unit)
    try:
        for s in range(4):
            lay_s = oracle_lib.layout(numel, unit, n, s)
            assert B.zero_state_bytes(ctx, s, n) == list(oracle_lib.state_bytes(lay_s.unit_padded, n, s))
        # by hand: stage 3 holds 16 B per element of ceil(psi / N) per unit
        assert B.zero_state_bytes(ctx, 3, n)[0] == 16 * (518 + 14 + 1)
        assert B.zero_state_bytes(ctx, 0, n)[0] == 16 * (1552 + 7 + 33 + 1)
        lay3 = oracle_lib.layout(numel, unit, n, 3)
        assert B.zero_stage3_peak_bytes(ctx) == oracle_lib.zero3_backward_peak(lay3.unit_padded, n)
    finally:
        B.zero_destroy(ctx)


def test_ledger_binding_with_fewer_ranks_than_the_context(B):
    # The library writes one entry per rank of the context; the binding's
    # array has room for the largest rank count whatever the caller asks for.
    pl = si.lecture_mlp()
    ctx = B.zero_plan(B.make_config(3, 16), pl.numel, pl.unit)
    try:
        full = B.zero_state_bytes(ctx, 2, 16)
        assert len(full) == 16 and len(set(full)) == 1
        assert B.zero_state_bytes(ctx, 2, 1) == full[:1]
    finally:
        B.zero_destroy(ctx)


@pytest.mark.parametrize("field,value", [
    ("stage", 4), ("stage", -1), ("n_ranks", 0), ("n_ranks", 17), ("grad_dtype", 2), ("adamw", 2),
    ("beta1", 1.0), ("beta2", -0.1), ("eps", -1.0), ("lr", float("inf")), ("weight_decay", -0.1),
])
def test_config_validation(B, field, value):
    cfg = B.make_config(1, 4)
    setattr(cfg, field, value)
    with pytest.raises(B.ZeroError) as e:
        B.zero_plan(cfg, [8], [0])
    assert e.value.status == B.ZERO_EINVAL
    assert B.zero_last_error(None)


def test_weight_decay_requires_adamw(B):
    with pytest.raises(B.ZeroError) as e:
        B.zero_plan(B.make_config(1, 4, weight_decay=0.1, adamw=False), [8], [0])
    assert e.value.status == B.ZERO_EINVAL
    ctx = B.zero_plan(B.make_config(1, 4, weight_decay=0.1, adamw=True), [8], [0])
    B.zero_destroy(ctx)


def test_bad_param_lists(B):
    cfg = B.make_config(1, 4)
    for numel, unit in [([4, 4], [1, 0]), ([-1], [0]), ([4], [-1])]:
        with pytest.raises(B.ZeroError) as e:
            B.zero_plan(cfg, numel, unit)
        assert e.value.status == B.ZERO_EINVAL


def test_plan_only_context_refuses_steps(B):
    ctx = B.zero_plan(B.make_config(2, 2), [10], [0])
    try:
        for call in (lambda: B.zero_step(ctx), lambda: B.zero_reduce_grads(ctx, 0, [0, 0]),
                     lambda: B.zero_gather_weights(ctx, 0, 0)):
            with pytest.raises(B.ZeroError) as e:
                call()
            assert e.value.status == B.ZERO_ESTATE
        with pytest.raises(B.ZeroError) as e:
            B.zero_post_step(ctx)
        assert e.value.status == B.ZERO_ESTATE
        with pytest.raises(B.ZeroError) as e:
            B.zero_layout(ctx, 1)
        assert e.value.status == B.ZERO_EINVAL
        assert "out of range" in B.zero_last_error(ctx)
        assert B.zero_step_count(ctx) == 0
        B.zero_set_lr(ctx, 5e-4)
        with pytest.raises(B.ZeroError):
            B.zero_set_lr(ctx, float("nan"))
    finally:
        B.zero_destroy(ctx)


def test_empty_parameter_list(B):
    ctx = B.zero_plan(B.make_config(3, 8), [], [])
    try:
        assert B.zero_padded_numel(ctx) == (0, 0)
        assert B.zero_num_units(ctx) == 0
        assert B.zero_stage3_peak_bytes(ctx) == (0, -1)
    finally:
        B.zero_destroy(ctx)


def test_product_path_has_no_oracle_import():
    # The CUDA package and its binding never touch the oracle.
    pkg = os.path.join(ROOT, "zero_sharded_mixed_flatparameter_gb300")
    for path in glob.glob(os.path.join(pkg, "**", "*"), recursive=True):
        if os.path.isfile(path) and path.endswith((".py", ".cu", ".cpp", ".h")):
            text = open(path).read()
            assert "oracle" not in text.lower(), path
