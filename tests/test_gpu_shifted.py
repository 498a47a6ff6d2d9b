"""The shifted-gradient step kernel against the oracle: segments whose flat
base is not a multiple of 8 elements, or whose replica gradients are not
16-byte aligned where the aligned body starts (padding every unit to a
multiple of N, CMU 15-779 Lecture 13 notes §3.6, moves later unit bases off
8-element boundaries; gradients that arrive as one buffer per unit are each
aligned on their own).  The kernel peels each segment's head so that the
state arrays are aligned and shifts every replica's gradient words into
place; results must be bit-identical to the oracle's for every head length,
every per-replica gradient offset, N and gradient dtype."""

import numpy as np
import pytest
import torch

import oracle
import synth_inputs as si
from gpu_common import (assert_bit_exact, compare_state, ensure_built, gpu_flatstep, make_problem, oracle_run,
                        to_np, upload_grads)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


def _register_offsets(fs, flats, offsets, keep):
    """Registers every unit from its own buffer, replica r's gradient placed
    offsets[r] elements past a 16-byte boundary."""
    for i in range(fs.n_units):
        numel, padded, shard, base = fs.layout(i)
        views = []
        for r, f in enumerate(flats):
            o = offsets[r] if isinstance(offsets[r], int) else offsets[r][i % len(offsets[r])]
            buf = torch.zeros(padded + 16, dtype=f.dtype, device=f.device)
            buf[o:o + padded] = f[base:base + padded]
            views.append(buf[o:o + padded])
        keep.append(views)
        fs.reduce_grads(i, views)


def _run(pb, offsets, launches=None):
    ref_states = {}
    oracle_run(pb, every_step=lambda t, s: ref_states.__setitem__(t, s))
    fs = gpu_flatstep(pb)
    try:
        for t in range(1, len(pb.grads) + 1):
            keep = []
            _register_offsets(fs, upload_grads(pb, t), offsets, keep)
            if pb.max_norm > 0:
                fs.clip_grad_norm(pb.max_norm)
            fs.step()
            if launches is not None:
                launches.append(fs.last_launches())
            fs.post_step()
            torch.cuda.synchronize()
            compare_state(fs, ref_states[t], f"step {t}")
    finally:
        fs.close()


# unit sizes whose running bases take every residue modulo 8 at N = 1 (stage 0
# pads nothing), with lengths below, at and above one vector and long ones
HEADS = [5, 1, 9, 2, 17, 3, 8 * 300 + 6, 4, 11, 7, 8 * 1000 + 3, 6, 2 * 256 * 8 * 2 + 5]


@pytest.mark.parametrize("gd", ["bf16", "fp32"])
@pytest.mark.parametrize("n", [1, 2, 3, 5, 8, 16])
def test_every_head_and_offset(gd, n):
    # replica r's gradient sits (r * 3 + unit) % k elements past a 16-byte
    # boundary (k = 8 bf16, 4 fp32): every shift, different per replica
    k = 8 if gd == "bf16" else 4
    pl = si.from_units(HEADS)
    pb = make_problem(pl, n, 0 if n == 1 else 2, grad_dtype=gd, steps=2, seed=300 + n)
    offsets = [[(r * 3 + u) % k for u in range(k)] for r in range(n)]
    _run(pb, offsets)


# units summing to more than 2^23 elements (the size from which aligned
# launches take the tile-staged kernels): every head and offset at a size
# where many waves of the grid pass over each segment
LARGE = [3_000_001, 5, 2_500_003, 4099, 3_100_007, 17]


@pytest.mark.parametrize("n", [1, 2, 3, 4])
def test_large_every_head_and_offset(n):
    assert sum(LARGE) >= 1 << 23
    pl = si.from_units(LARGE)
    pb = make_problem(pl, n, 0 if n == 1 else 2, steps=2, seed=320 + n)
    offsets = [[(r * 3 + u) % 8 for u in range(8)] for r in range(n)]
    _run(pb, offsets)


def test_large_clipped_adamw_capturable():
    pl = si.from_units(LARGE)
    pb = make_problem(pl, 3, 3, steps=3, seed=325, max_norm=0.05, adamw=True, weight_decay=0.1)
    ref = oracle_run(pb)
    fs = gpu_flatstep(pb)
    try:
        fs.enable_capturable(max_steps=8)
        for t in range(1, 4):
            keep = []
            _register_offsets(fs, upload_grads(pb, t), [3, 0, 5], keep)
            fs.clip_grad_norm(pb.max_norm)
            fs.step()
            fs.post_step()
        torch.cuda.synchronize()
        compare_state(fs, ref, "large shifted layout, clipped AdamW, capturable")
    finally:
        fs.close()


@pytest.mark.parametrize("gd", ["bf16", "fp32"])
def test_aligned_gradients_with_unaligned_bases(gd):
    # separate 16-byte-aligned buffers per unit while the unit bases are not
    # multiples of 8: the head is peeled, every replica then has the same shift
    pl = si.from_units([1552, 7, 9312, 33, 17, 40_001, 3])
    pb = make_problem(pl, 3, 3, grad_dtype=gd, steps=3, seed=310)
    _run(pb, [0, 0, 0])


def test_long_segments_warp_edges():
    # long bodies: many waves of the grid, vectors at the ends of segments
    # and at the stride's wrap-around take the neighbour's word or their own
    pl = si.from_units([152 * 2 * 256 * 8 * 3 + 5, 1_000_003, 77])
    pb = make_problem(pl, 3, 2, steps=2, seed=311)
    _run(pb, [1, 6, 3])
    pb = make_problem(pl, 2, 1, grad_dtype="fp32", steps=1, seed=312)
    _run(pb, [3, 1])


def test_clipped_and_adamw():
    pl = si.from_units([4099, 16384 + 5, 1552])
    pb = make_problem(pl, 5, 3, steps=3, seed=313, max_norm=0.05, adamw=True, weight_decay=0.1)
    _run(pb, [2, 5, 0, 7, 1])


def test_many_segments_several_launches():
    # more unaligned units than one launch carries (48 segments per launch)
    sizes = [8 * (i % 7) + 1 + (i % 5) for i in range(110)]
    pb = make_problem(si.from_units(sizes), 3, 2, steps=2, seed=314)
    launches = []
    _run(pb, [[1, 2, 3], [0, 5, 7], [6, 4, 2]], launches)
    assert all(x >= 3 for x in launches)


def test_capturable_mode():
    # the step count and bias corrections read from the device (kDevBias instances)
    pl = si.from_units([1552, 7, 9312, 33])
    pb = make_problem(pl, 3, 3, steps=3, seed=315)
    ref = oracle_run(pb)
    fs = gpu_flatstep(pb)
    try:
        fs.enable_capturable(max_steps=8)
        for t in range(1, 4):
            keep = []
            _register_offsets(fs, upload_grads(pb, t), [3, 0, 5], keep)
            fs.step()
            fs.post_step()
        torch.cuda.synchronize()
        compare_state(fs, ref, "capturable shifted")
    finally:
        fs.close()


@pytest.mark.parametrize("n", [3, 6])
def test_llama_2048_units_one_buffer_per_unit(n):
    # The ZeRO-3 layout of the Llama-2048 model (654,346,240 params in 10
    # units) at N = 3 and N = 6: padding to a multiple of N moves the unit
    # bases off 8-element boundaries; each unit's gradients are their own
    # 16-byte-aligned buffers.  Windows at every unit's start and end and in
    # its middle are checked bit for bit against the oracle after 3 steps.
    pl = si.llama_2048_units()
    lay = oracle.layout(pl.numel, pl.unit, n, 3)
    assert any(int(b) % 8 for b in lay.unit_base)
    W = 4096
    init_flat = si.normal_fp32(pl.total, 0.02, 70 + n, device="cuda")
    offs = [0]
    for k in pl.numel:
        offs.append(offs[-1] + k)
    fs = gpu_flatstep_from(pl, n, [init_flat[offs[p]:offs[p + 1]] for p in range(len(pl.numel))])
    try:
        starts = []
        for i in range(fs.n_units):
            numel, padded, shard, base = fs.layout(i)
            starts += [base, base + padded // 2 - 3, base + padded - W]
        win = {a: [to_np(fs.master[a:a + W]).copy(), np.zeros(W, np.float32), np.zeros(W, np.float32),
                   np.zeros(W, np.uint16)] for a in starts}
        del init_flat
        h = oracle.Hyper(n_ranks=n)
        for t in (1, 2, 3):
            unit_grads = []
            for i in range(fs.n_units):
                numel, padded, shard, base = fs.layout(i)
                g = si.replica_grads(n, padded, 1e-3, 400 + 17 * t + i, "bf16", device="cuda", pad_from=numel)
                unit_grads.append(g)
                fs.reduce_grads(i, g)
            fs.step()
            fs.post_step()
            for a in starts:
                i = max(u for u in range(fs.n_units) if fs.layout(u)[3] <= a)
                base = fs.layout(i)[3]
                oracle.step_window(h, t, [to_np(g[a - base:a - base + W]) for g in unit_grads[i]], *win[a])
            del unit_grads
        torch.cuda.synchronize()
        for a in starts:
            got = (to_np(fs.master[a:a + W]), to_np(fs.exp_avg[a:a + W]), to_np(fs.exp_avg_sq[a:a + W]),
                   to_np(fs.param16[a:a + W]))
            for name, g, w in zip(("master", "m", "v", "param16"), got, win[a]):
                assert_bit_exact(g, w, f"N={n} window@{a} {name}")
        # the ZeRO-3 gathers of these unaligned units: one launch for all ten
        bufs = [torch.empty(int(fs.layout(i)[1]), dtype=torch.bfloat16, device="cuda") for i in range(fs.n_units)]
        fs.gather_units(0, bufs)
        assert fs.last_launches() == 1
        torch.cuda.synchronize()
        for i, buf in enumerate(bufs):
            numel, padded, shard, base = fs.layout(i)
            assert torch.equal(buf.view(torch.int16), fs.param16[base:base + padded].view(torch.int16)), i
        del bufs
    finally:
        fs.close()
        torch.cuda.empty_cache()


def gpu_flatstep_from(pl, n, init):
    from zero_sharded_mixed_flatparameter_gb300.runner import FlatStep
    return FlatStep(pl.numel, pl.unit, stage=3, n_ranks=n, init_params=init)
