"""Invariants of the method, checked on the oracle (not gpu).

* ZeRO-1/2/3 are bit-identical to plain data parallelism when the gradient
  summation order is fixed and Adam is elementwise (CMU 15-779 Lecture 13
  notes §3.4; Femtotron dev log #6 "test results").
* Forgetting the post-update all-gather makes the replicas silently diverge;
  comparing replica checksums catches it (notes §4.3).  The mistake is planted
  in the oracle, on the CPU.
* Pads stay zero; make_master flattens in caller order; the ZeRO-3 gather is
  the rank-order concatenation of the unit's shards.
"""

import numpy as np
import pytest
import torch

import synth_inputs as si
from oracle import Hyper


def _bits(t):
    return si.as_numpy_bits(t)


def _scatter(pl, lay, per_param_values, dtype):
    """Place per-parameter arrays into a zero-padded flat buffer of the layout."""
    flat = np.zeros(lay.total_padded, dtype=dtype)
    for p, vals in enumerate(per_param_values):
        off = int(lay.param_offset[p])
        flat[off:off + len(vals)] = vals
    return flat


def _problem(pl, n, seed, grad_dtype="bf16", steps=10):
    """Per-parameter init values and per-step per-replica per-parameter grads."""
    init = [si.normal_fp32(k, 0.02, seed * 100 + p).numpy() for p, k in enumerate(pl.numel)]
    grads = []
    for t in range(steps):
        reps = []
        for r in range(n):
            per_param = []
            for p, k in enumerate(pl.numel):
                g = si.normal_fp32(k, 1e-2, seed * 100000 + t * 1000 + r * 37 + p)
                per_param.append(_bits(g.to(torch.bfloat16)) if grad_dtype == "bf16" else g.numpy())
            reps.append(per_param)
        grads.append(reps)
    return init, grads


def _run_stage(oracle_lib, pl, hyper, stage, init, grads, n_copies=1, plant=False):
    n = hyper.n_ranks
    lay = oracle_lib.layout(pl.numel, pl.unit, n, stage)
    master, m, v, p16 = oracle_lib.make_master(pl.numel, lay, init)
    copies = np.tile(p16, (n_copies, 1)) if n_copies > 1 else p16
    gdt = np.uint16 if hyper.grad_dtype == "bf16" else np.float32
    for t, reps in enumerate(grads, start=1):
        flat = [_scatter(pl, lay, per_param, gdt) for per_param in reps]
        if stage == 0:
            oracle_lib.dp_step(hyper, t, flat, master, m, v, copies)
        else:
            oracle_lib.zero_step(hyper, stage, t, lay, flat, master, m, v, copies, plant_skip_allgather=plant)
    return lay, master, m, v, copies


def _unflatten(pl, lay, flat):
    return np.concatenate([flat[int(lay.param_offset[p]):int(lay.param_offset[p]) + k]
                           for p, k in enumerate(pl.numel)]) if pl.numel else flat[:0]


CASES = [
    ("toy_mlp_n4", si.toy_mlp(), 4, "bf16", False),
    ("lecture_mlp_n3_padded", si.lecture_mlp(), 3, "bf16", False),
    ("odd_units_n16", si.from_units([1, 7, 15, 17, 33]), 16, "bf16", True),
    ("odd_units_n5_fp32", si.from_units([11, 1, 29]), 5, "fp32", True),
    ("single_n1", si.from_units([40]), 1, "bf16", False),
]


@pytest.mark.parametrize("name,pl,n,gd,adamw", CASES, ids=[c[0] for c in CASES])
def test_stages_bit_identical_to_data_parallel(oracle_lib, name, pl, n, gd, adamw):
    h = Hyper(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.1 if adamw else 0.0,
              adamw=adamw, n_ranks=n, grad_dtype=gd)
    init, grads = _problem(pl, n, seed=11, grad_dtype=gd, steps=10)
    ref = _run_stage(oracle_lib, pl, h, 0, init, grads)
    ref_vals = [_unflatten(pl, ref[0], a) for a in ref[1:]]
    for stage in (1, 2, 3):
        got = _run_stage(oracle_lib, pl, h, stage, init, grads)
        got_vals = [_unflatten(pl, got[0], a) for a in got[1:]]
        for a, b in zip(ref_vals, got_vals):
            assert np.array_equal(a.view(np.uint8), b.view(np.uint8)), (name, stage)
        # the pads of the sharded layout are still exactly zero
        lay = got[0]
        for i in range(len(lay.unit_numel)):
            lo, hi = int(lay.unit_base[i] + lay.unit_numel[i]), int(lay.unit_base[i] + lay.unit_padded[i])
            for arr in got[1:]:
                assert not np.any(arr[lo:hi])


def test_replicas_identical_after_allgather(oracle_lib):
    pl, n = si.lecture_mlp(), 4
    h = Hyper(n_ranks=n)
    init, grads = _problem(pl, n, seed=5, steps=3)
    for stage in (1, 2):
        lay, master, m, v, copies = _run_stage(oracle_lib, pl, h, stage, init, grads, n_copies=n)
        for q in range(1, n):
            assert np.array_equal(copies[q], copies[0])
        shared = _run_stage(oracle_lib, pl, h, stage, init, grads, n_copies=1)[4]
        assert np.array_equal(copies[0], shared)


def test_missing_allgather_diverges_silently(oracle_lib):
    # Planted mistake (oracle, CPU): each rank updates only its own 1/N of its
    # bf16 copy.  The run "succeeds", but the replica checksums differ.
    pl, n = si.lecture_mlp(), 4
    h = Hyper(lr=1e-2, n_ranks=n)
    init, grads = _problem(pl, n, seed=5, steps=3)
    lay, master, m, v, copies = _run_stage(oracle_lib, pl, h, 2, init, grads, n_copies=n, plant=True)
    good = _run_stage(oracle_lib, pl, h, 2, init, grads, n_copies=1)[4]
    sums = [int(copies[q].astype(np.int64).sum()) for q in range(n)]
    assert len(set(sums)) == n  # every replica's checksum differs
    for d in range(n):
        own = np.zeros(lay.total_padded, dtype=bool)
        for i in range(len(lay.unit_numel)):
            s = int(lay.unit_shard[i])
            own[int(lay.unit_base[i]) + d * s:int(lay.unit_base[i]) + (d + 1) * s] = True
        # each rank's own shard is right, everything else is stale
        assert np.array_equal(copies[d][own], good[own])
        assert not np.array_equal(copies[d][~own], good[~own])


def test_make_master_flattens_in_caller_order(oracle_lib):
    pl = si.from_units([3, 5, 2])
    pl = si.ParamList("mixed", [3, 2, 5, 2], [0, 0, 1, 2], ["a", "b", "c", "d"])
    n = 4
    lay = oracle_lib.layout(pl.numel, pl.unit, n, stage=1)
    init = [np.arange(k, dtype=np.float32) + 10 * (p + 1) for p, k in enumerate(pl.numel)]
    master, m, v, p16 = oracle_lib.make_master(pl.numel, lay, init)
    # unit 0 = a(3) b(2) + 3 pad, unit 1 = c(5) + 3 pad, unit 2 = d(2) + 2 pad
    want = np.array([10, 11, 12, 20, 21, 0, 0, 0, 30, 31, 32, 33, 34, 0, 0, 0, 40, 41, 0, 0], np.float32)
    assert np.array_equal(master, want)
    assert not m.any() and not v.any()
    assert np.array_equal(p16, (want.view(np.uint32) >> 16).astype(np.uint16))


def test_gather_unit_is_rank_order_concatenation(oracle_lib):
    n, padded, base = 4, 12, 5
    p16 = np.arange(30, dtype=np.uint16)
    out = oracle_lib.gather_unit(p16, base, padded, n)
    assert np.array_equal(out, p16[base:base + padded])
