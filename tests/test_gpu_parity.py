"""GPU parity: the CUDA path through the C ABI against the oracle, element by
element, on the same seeded inputs (small sizes the oracle finishes in
seconds, spanning several tiles and ragged tails)."""

import numpy as np
import pytest
import torch

import synth_inputs as si
from gpu_common import (compare_state, ensure_built, make_problem, oracle_run, run_gpu, to_np)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()
    yield
    torch.cuda.empty_cache()


def _per_step(pb, mode="units"):
    """Compare after every step (not only at the end)."""
    ref_states = {}
    oracle_run(pb, every_step=lambda t, s: ref_states.__setitem__(t, s))

    def check(t, fs):
        compare_state(fs, ref_states[t], f"step {t}")
    fs = run_gpu(pb, mode=mode, every_step=check)
    fs.close()


@pytest.mark.parametrize("stage", [0, 1, 2, 3])
def test_toy_mlp_n4_all_stages(stage):
    # 5-layer MLP 32-128-128-64-64-16 (34,192 params), N = 4, Adam, 10 steps
    pb = make_problem(si.toy_mlp(), 4, stage, steps=10, seed=1)
    _per_step(pb, mode="units")


@pytest.mark.parametrize("mode", ["all", "units", "separate"])
def test_registration_modes(mode):
    pb = make_problem(si.toy_mlp(), 4, 2, steps=3, seed=2)
    _per_step(pb, mode=mode)


@pytest.mark.parametrize("n", list(range(1, 17)))
def test_every_rank_count(n):
    # one unit spanning several CTAs' worth of vectors plus a ragged tail
    size = 3 * 256 * 8 + 5
    pb = make_problem(si.from_units([size, 40]), n, 2, steps=3, seed=10 + n)
    _per_step(pb)


@pytest.mark.parametrize("n", [2, 8])
def test_fp32_grads(n):
    pb = make_problem(si.from_units([4096 + 3, 1000]), n, 1, grad_dtype="fp32", steps=5, seed=3)
    _per_step(pb)


def test_adamw_decoupled_decay():
    pb = make_problem(si.toy_mlp(), 4, 3, steps=10, seed=4, weight_decay=0.1, adamw=True)
    _per_step(pb)


def test_lecture_mlp_n3_padding_and_misaligned_units():
    # N = 3 pads the last 1,552-param unit by 2 (CMU 15-779 notes §3.6); units
    # after a non-multiple-of-8 base take the element-wise kernel.
    pl = si.from_units([1552, 3168, 9312, 1552, 7])
    pb = make_problem(pl, 3, 2, steps=4, seed=5)
    assert pb.lay.total_padded == 1554 + 3168 + 9312 + 1554 + 9
    _per_step(pb, mode="separate")
    _per_step(pb, mode="units")


def test_odd_units_n16():
    pb = make_problem(si.from_units([1, 7, 15, 17, 0, 33, 16 * 8 + 1]), 16, 3, steps=4, seed=6)
    _per_step(pb)


def test_many_units_more_than_one_launch():
    # more segments than one launch carries
    sizes = [(8 * (i % 5) + 8) * 4 for i in range(130)]
    pb = make_problem(si.from_units(sizes), 4, 3, steps=2, seed=7)
    _per_step(pb, mode="separate")


def test_large_multi_wave():
    # several waves of the persistent grid plus a ragged tail
    size = 152 * 4 * 256 * 8 * 3 + 7
    pb = make_problem(si.from_units([size]), 2, 1, steps=2, seed=8)
    _per_step(pb, mode="all")


def test_outliers_and_extreme_values():
    pb = make_problem(si.from_units([20_000]), 8, 2, steps=3, seed=9, outlier_fraction=0.001)
    _per_step(pb)
    # large grads, tiny grads, +-inf and NaN in one replica: propagate like the oracle
    pb = make_problem(si.from_units([64]), 2, 2, steps=2, seed=10)
    for t in range(2):
        g = pb.grads[t][1]
        g[0] = 0x7F80  # +inf
        g[1] = 0xFF80  # -inf
        g[2] = 0x7FC0  # NaN
        g[3] = 0x7F7F  # largest finite bf16
        g[4] = 0x0001  # smallest subnormal bf16
    _per_step(pb)


def test_empty_layouts():
    pb = make_problem(si.from_units([0, 0]), 4, 2, steps=2, seed=11)
    fs = run_gpu(pb)
    assert fs.padded == 0 and fs.step_count() == 2
    fs.close()


def test_bf16_cast_rounds_to_nearest_even():
    # a master of exact ties: with lr = 0 the step leaves w unchanged and
    # param16 must be its round-to-nearest-even bf16
    ties = np.array([0x3F808000, 0x3F818000, 0x3F808001, 0x3F807FFF, 0x7F7FFFFF, 0x00018000],
                    dtype=np.uint32).view(np.float32)
    pl = si.from_units([len(ties)])
    pb = make_problem(pl, 1, 1, steps=1, seed=12, lr=0.0)
    pb.init = [ties.copy()]
    pb.grads[0][0][:] = 0
    ref = oracle_run(pb)
    fs = run_gpu(pb)
    assert np.array_equal(to_np(fs.param16), ref[3])
    assert list(ref[3]) == [0x3F80, 0x3F82, 0x3F81, 0x3F80, 0x7F80, 0x0002]
    fs.close()


def test_set_lr_between_steps():
    # a scheduler's lr change between steps: second step at lr 2e-3 on both sides
    import oracle as O
    from gpu_common import gpu_flatstep, register, upload_grads
    from zero_sharded_mixed_flatparameter_gb300 import binding as B
    pb = make_problem(si.toy_mlp(), 4, 1, steps=2, seed=13)
    master, m, v, p16 = O.make_master(pb.pl.numel, pb.lay, pb.init)
    fs = gpu_flatstep(pb)
    for t in (1, 2):
        if t == 2:
            pb.hyper.lr = 2e-3
            B.zero_set_lr(fs.ctx, 2e-3)
        O.zero_step(pb.hyper, 1, t, pb.lay, pb.grads[t - 1], master, m, v, p16)
        register(fs, pb, upload_grads(pb, t), "all", [])
        fs.step()
        fs.post_step()
    torch.cuda.synchronize()
    compare_state(fs, (master, m, v, p16), "set_lr")
    fs.close()


@pytest.mark.parametrize("n,gd", [(n, "bf16") for n in (1, 2, 3, 4, 5, 6, 7, 8, 10, 12, 13, 16)]
                         + [(n, "fp32") for n in (6, 7, 8, 9, 10, 11, 12, 16)])
def test_tile_staged_kernel(n, gd):
    # Over >= 2^23 elements per launch, N = 1..4 and N >= 7 bf16 and N >= 7
    # fp32 replicas take a tile-staged (bulk copy) kernel: 2,048-element
    # tiles for bf16 N >= 13 and fp32 N = 8, 9; the barrier-free pipelined
    # kernel (2,048-element tiles, four stages at N = 7, 8, three from 9) for
    # bf16 N = 7..12; 4
    # elements per thread (1,024- or 2,048-element tiles) for bf16 N = 1..4
    # and fp32 N = 7 and N >= 10.  The neighbours of the rank thresholds take
    # the register-staged one.  8.7 M elements in several segments, each with
    # full tiles and a ragged part after them, plus units too small for one
    # tile
    from zero_sharded_mixed_flatparameter_gb300 import binding as B
    timeouts = B.zero_kernel_timeouts()  # a process-wide count: compare against this
    pl = si.from_units([4_200_005, 1552, 2_500_000, 7, 2_000_000])
    pb = make_problem(pl, n, 3, grad_dtype=gd, steps=2, seed=14 + n)
    _per_step(pb, mode="separate")
    pb = make_problem(pl, n, 2, grad_dtype=gd, steps=2, seed=15 + n, max_norm=0.1)
    ref = oracle_run(pb)
    fs = run_gpu(pb, mode="all")
    compare_state(fs, ref, "tile-staged, clipped")
    fs.close()
    assert B.zero_kernel_timeouts() == timeouts


def test_tile_staged_threshold_neighbours():
    # padded to 2^23 - 16 elements the register-staged kernel runs, to
    # 2^23 + 16 the tile-staged one; both agree with the oracle
    for total in (2 ** 23 - 21, 2 ** 23 + 5):
        pb = make_problem(si.from_units([total]), 16, 2, steps=1, seed=77)
        ref = oracle_run(pb)
        fs = run_gpu(pb, mode="all")
        compare_state(fs, ref, f"{total} elements")
        fs.close()


@pytest.mark.parametrize("fresh", [False, True])
def test_long_run(fresh):
    # many steps, bit for bit: an error that grows step by step (the pages
    # found a silent bug only by running identical data every step and
    # watching the error grow) shows here.  N = 3 makes 1/N inexact; AdamW.
    steps = 100 if fresh else 200
    pl = si.from_units([1552, 7, 3000, 33])
    pb = make_problem(pl, 3, 3, steps=1 if not fresh else steps, seed=500 + fresh, adamw=True, weight_decay=0.1,
                      max_norm=0.05 if fresh else 0.0)
    if not fresh:
        pb.grads = pb.grads * steps              # the same gradients every step
    ref = oracle_run(pb)
    fs = run_gpu(pb, mode="units")
    compare_state(fs, ref, f"after {steps} steps")
    assert fs.step_count() == steps
    fs.close()
