"""The step's count of non-finite reduced gradients (zero_count_nonfinite)
against the oracle's count, in every kernel that runs a step: the
register-staged and both tile-staged kernels, the shifted-gradient kernel,
element-wise heads and tails, the kept reduced gradient of a clip and the
offloaded step.  Values are planted on the host: inf, NaN, and pairs of the
largest finite values whose fp32 sum overflows; nothing faults."""

import numpy as np
import pytest
import torch

import oracle
import synth_inputs as si
from gpu_common import compare_state, ensure_built, gpu_flatstep, make_problem, oracle_run, register, upload_grads
from zero_sharded_mixed_flatparameter_gb300 import binding as B

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


def _plant(pb, t, positions, rng):
    """Plants non-finite values at `positions` of step t's replicas: inf, NaN,
    -inf, or the largest finite value in every replica (the sum overflows)."""
    reps = pb.grads[t - 1]
    bf = pb.grad_dtype == "bf16"
    vals = ([np.uint16(0x7F80), np.uint16(0x7FC0), np.uint16(0xFF80)] if bf else
            [np.float32(np.inf), np.float32(np.nan), np.float32(-np.inf)])
    top = np.uint16(0x7F7F) if bf else np.float32(3.3e38)
    for k, p in enumerate(positions):
        if k % 4 == 3 and pb.n >= 2:
            for r in reps:
                r[p] = top
        else:
            reps[int(rng.integers(0, pb.n))][p] = vals[k % 3]


def _run_counted(pb, mode="units", positions=None, seed=0, clip_keep=False, offload=None, check_state=True,
                 offsets=None):
    rng = np.random.default_rng(seed)
    real = int(pb.lay.unit_numel[0])  # the first unit's real elements (no pads among them)
    for t in range(1, len(pb.grads) + 1):
        pos = positions(t) if positions else rng.choice(real, 5, replace=False)
        _plant(pb, t, pos, rng)
    want = [oracle.nonfinite_count(pb.hyper, pb.grads[t]) for t in range(len(pb.grads))]
    assert sum(want) > 0
    ref_states = {}
    if check_state:
        oracle_run(pb, every_step=lambda t, s: ref_states.__setitem__(t, s))
    fs = gpu_flatstep(pb, offload=offload)
    counter = torch.zeros(1, dtype=torch.int64, device="cuda")
    fs.count_nonfinite(counter)
    got = []
    try:
        for t in range(1, len(pb.grads) + 1):
            keep = []
            if offsets is not None:
                from test_gpu_shifted import _register_offsets
                _register_offsets(fs, upload_grads(pb, t), offsets, keep)
            else:
                register(fs, pb, upload_grads(pb, t), mode, keep)
            if pb.max_norm > 0:
                fs.clip_grad_norm(pb.max_norm, keep_reduced=clip_keep)
            fs.step()
            fs.post_step()
            got.append(B.zero_read_nonfinite(fs.ctx, fs.stream_handle()))
            if check_state:
                compare_state(fs, ref_states[t], f"step {t}")
    finally:
        fs.close()
    assert got == list(np.cumsum(want)), (got, want)


@pytest.mark.parametrize("gd", ["bf16", "fp32"])
def test_unclipped_small_layouts(gd):
    # register-staged kernel: vectors and ragged tails of several units
    pl = si.from_units([4096, 77, 5001, 8])
    pb = make_problem(pl, 3, 2, grad_dtype=gd, steps=3, seed=600)
    tail = int(pb.lay.unit_base[1] + 76)
    _run_counted(pb, positions=lambda t: [3, 1000 + t, tail, 9000 - t, 4096 + 77 + 5])


def test_shifted_kernel_heads_and_tails():
    # one buffer per unit with unaligned bases: heads, bodies and tails
    pl = si.from_units([1552, 7, 9312, 33, 17])
    pb = make_problem(pl, 3, 3, steps=3, seed=601)
    base = [int(b) for b in pb.lay.unit_base]
    _run_counted(pb, offsets=[0, 3, 5], positions=lambda t: [base[1] + 2, base[2], base[2] + 4000 + t,
                                                             base[3] + 32, base[4] + t])


@pytest.mark.parametrize("n,gd", [(2, "bf16"), (10, "bf16"), (16, "bf16"), (8, "fp32"), (12, "fp32")])
def test_tile_staged_kernels(n, gd):
    # launches of at least 2^23 elements take the tile-staged kernels;
    # the count only (the state of these kernels is checked elsewhere)
    pl = si.from_units([2 ** 23 + 1000, 300])
    pb = make_problem(pl, n, 1, grad_dtype=gd, steps=2, seed=602 + n)
    _run_counted(pb, mode="all", check_state=False, seed=n)


def test_clipped_with_kept_reduced_gradient():
    pl = si.from_units([40_000, 33])
    pb = make_problem(pl, 8, 2, steps=2, seed=606, max_norm=1e30)  # an inactive clip: the count still runs
    _run_counted(pb, clip_keep=True, seed=3)


def test_offloaded_step():
    pl = si.from_units([20_000, 77])
    pb = make_problem(pl, 4, 2, steps=2, seed=607)
    _run_counted(pb, offload=dict(chunk=4096, threads=2), seed=4)


def test_counter_off_and_errors():
    pl = si.from_units([4096])
    pb = make_problem(pl, 2, 2, steps=1, seed=608)
    _plant(pb, 1, [5, 6, 7], np.random.default_rng(0))
    fs = gpu_flatstep(pb)
    try:
        with pytest.raises(B.ZeroError) as e:
            B.zero_read_nonfinite(fs.ctx, 0)
        assert e.value.status == B.ZERO_ESTATE
        buf = torch.full((4,), 7, dtype=torch.int64, device="cuda")
        with pytest.raises(B.ZeroError) as e:
            B.zero_count_nonfinite(fs.ctx, buf.data_ptr() + 4)  # misaligned
        assert e.value.status == B.ZERO_EINVAL
        host = torch.zeros(1, dtype=torch.int64).pin_memory()
        with pytest.raises(B.ZeroError) as e:
            B.zero_count_nonfinite(fs.ctx, host.data_ptr())
        assert e.value.status == B.ZERO_EINVAL
        # counting switched on, then off again: the counter is left alone
        fs.count_nonfinite(buf[:1])
        fs.count_nonfinite(None)
        fs.reduce_grads(-1, upload_grads(pb, 1))
        fs.step()
        fs.post_step()
        torch.cuda.synchronize()
        assert buf.tolist() == [7, 7, 7, 7]
    finally:
        fs.close()
