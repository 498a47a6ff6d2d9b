"""Pins for the oracle's checkpoint export/import with resharding (not gpu).

The pads are not parameters (CMU 15-779 Lecture 13 notes §5.2), so a
checkpoint keeps only the real elements; importing it under another shard
count re-pads.  Because the step is elementwise and the pads stay zero,
training that is checkpointed at N ranks and resumed at N' ranks must match
an uninterrupted run bit for bit (the dp_size change of Femtotron #5, the
resharding checkpoints of the source guide)."""

import numpy as np

import synth_inputs as si
from oracle import Hyper


def test_export_import_round_trip(oracle_lib):
    pl = si.ParamList("mixed", [3, 2, 5, 0, 2], [0, 0, 1, 1, 2], list("abcde"))
    lay = oracle_lib.layout(pl.numel, pl.unit, 4, 3)
    padded = np.arange(lay.total_padded, dtype=np.float32) + 1
    for i in range(len(lay.unit_numel)):   # pads zero as in a real state
        padded[lay.unit_base[i] + lay.unit_numel[i]:lay.unit_base[i] + lay.unit_padded[i]] = 0
    compact = oracle_lib.export_state(lay, padded)
    # unit 0 = a(3) b(2) + 3 pad, unit 1 = c(5) + 3 pad, unit 2 = e(2) + 2 pad
    assert list(compact) == [1, 2, 3, 4, 5, 9, 10, 11, 12, 13, 17, 18]
    assert np.array_equal(oracle_lib.import_state(lay, compact), padded)
    other = oracle_lib.layout(pl.numel, pl.unit, 3, 1)
    assert np.array_equal(oracle_lib.export_state(other, oracle_lib.import_state(other, compact)), compact)


def _grads_for(lay, pl, per_param, n):
    flat = []
    for r in range(n):
        f = np.zeros(lay.total_padded, np.uint16)
        for p, k in enumerate(pl.numel):
            f[lay.param_offset[p]:lay.param_offset[p] + k] = per_param[r][p]
        flat.append(f)
    return flat


def test_resharded_resume_equals_uninterrupted(oracle_lib):
    import torch
    pl = si.from_units([1552, 7, 33, 9312])
    rng = np.random.default_rng(4)
    init = [rng.normal(0, 0.02, k).astype(np.float32) for k in pl.numel]
    # Every replica gets the same bf16 gradient, so the average is that
    # gradient exactly at any N: a power of two scales exactly, and for N = 3,
    # (3x) * fp32(1/3) = x (1 + 2^-25) lies less than half an ulp above x,
    # because x has only 8 significant bits.
    steps = 6

    def bf(x):
        return torch.tensor(x.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    g = [[bf(rng.normal(0, 1e-2, k)) for k in pl.numel] for _ in range(steps)]

    def run(n, stage, t0, t1, state):
        lay = oracle_lib.layout(pl.numel, pl.unit, n, stage)
        master, m, v, p16 = state(lay)
        h = Hyper(n_ranks=n, adamw=True, weight_decay=0.1)
        for t in range(t0, t1):
            flat = _grads_for(lay, pl, [g[t]] * n, n)   # identical replicas: the average is g[t] exactly
            oracle_lib.zero_step(h, stage, t + 1, lay, flat, master, m, v, p16)
        return lay, (master, m, v, p16)

    fresh = lambda lay: oracle_lib.make_master(pl.numel, lay, init)
    lay_a, st_a = run(8, 3, 0, steps, fresh)
    lay_b, st_b = run(8, 3, 0, 3, fresh)
    ckpt = [oracle_lib.export_state(lay_b, x) for x in st_b[:3]]

    def resumed(lay):
        master, m, v = (oracle_lib.import_state(lay, c) for c in ckpt)
        p16 = oracle_lib.bf16_round(master)
        return master, m, v, p16
    lay_c, st_c = run(3, 1, 3, steps, resumed)
    for a, c in zip(st_a[:3], st_c[:3]):
        assert np.array_equal(oracle_lib.export_state(lay_a, a).view(np.uint32),
                              oracle_lib.export_state(lay_c, c).view(np.uint32))
