"""Failure detection of the C ABI on a GPU: every bad call returns a
status (never a fault) and leaves the context unchanged; the failures are
made on the host (bad pointers, wrong order of calls).  The one device-side
failure tested is a bounded wait that runs out because the test hook never
issues the copy it waits for; no test here asks the GPU to fault, trap or
hang."""

import ctypes

import numpy as np
import pytest
import torch

import synth_inputs as si
from gpu_common import (check_guards, compare_state, ensure_built, make_problem, oracle_run, register, run_gpu,
                        upload_grads)
from gpu_common import gpu_flatstep
from zero_sharded_mixed_flatparameter_gb300 import binding as B

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


def _status(fn):
    with pytest.raises(B.ZeroError) as e:
        fn()
    return e.value.status


def test_make_master_rejects_bad_buffers():
    cfg = B.make_config(1, 2)
    dev = torch.zeros(64, dtype=torch.float32, device="cuda")
    p16 = torch.zeros(64, dtype=torch.bfloat16, device="cuda")
    init = torch.zeros(16, dtype=torch.float32, device="cuda")
    host = torch.zeros(64, dtype=torch.float32)
    ok = dict(master=dev.data_ptr(), exp_avg=dev.data_ptr(), exp_avg_sq=dev.data_ptr(), param16=p16.data_ptr())

    def mk(**over):
        args = dict(ok)
        args.update(over)
        return B.zero_make_master(cfg, [16], [0], [init.data_ptr()], **args)

    assert _status(lambda: mk(master=0)) == B.ZERO_EINVAL
    assert _status(lambda: mk(exp_avg=dev.data_ptr() + 4)) == B.ZERO_EINVAL          # misaligned
    assert _status(lambda: mk(exp_avg_sq=host.data_ptr())) == B.ZERO_EINVAL          # host memory
    assert "not CUDA device memory" in B.zero_last_error(None)
    assert _status(lambda: B.zero_make_master(cfg, [16], [0], [0], **ok)) == B.ZERO_EINVAL
    assert _status(lambda: B.zero_make_master(cfg, [16], [0], [host.data_ptr()], **ok)) == B.ZERO_EINVAL
    ctx = mk()
    B.zero_destroy(ctx)


def test_state_machine_and_no_side_effects():
    pb = make_problem(si.toy_mlp(), 4, 2, steps=2, seed=31)
    ref = oracle_run(pb, steps=1)
    fs = gpu_flatstep(pb)
    try:
        # step before gradients are registered
        assert _status(fs.step) == B.ZERO_ESTATE
        assert "no registered gradients" in B.zero_last_error(fs.ctx)
        # post_step without a step
        assert _status(fs.post_step) == B.ZERO_ESTATE
        flats = upload_grads(pb, 1)
        # the runner refuses replica buffers shorter than the padded length
        # (the kernels read every padded element)
        with pytest.raises(ValueError, match="padded"):
            fs.reduce_grads(-1, [f[:fs.padded - 1] for f in flats])
        with pytest.raises(ValueError, match="padded"):
            fs.reduce_grads(0, [f[:fs.layout(0)[1] - 1] for f in flats])
        # partial registration is not enough
        numel, padded, shard, base = fs.layout(0)
        fs.reduce_grads(0, [f[base:base + padded] for f in flats])
        assert _status(fs.step) == B.ZERO_ESTATE
        # bad registrations
        assert _status(lambda: B.zero_reduce_grads(fs.ctx, 9, [f.data_ptr() for f in flats])) == B.ZERO_EINVAL
        assert _status(lambda: B.zero_reduce_grads(fs.ctx, 1, [0] * 4)) == B.ZERO_EINVAL
        assert _status(lambda: B.zero_reduce_grads(fs.ctx, 1, [flats[0].data_ptr() + 1] * 4)) == B.ZERO_EINVAL
        assert fs.step_count() == 0
        register(fs, pb, flats, "units", [])
        fs.step()
        assert fs.step_count() == 1
        # a second step or new gradients before post_step
        assert _status(fs.step) == B.ZERO_ESTATE
        assert _status(lambda: fs.reduce_grads(-1, flats)) == B.ZERO_ESTATE
        assert fs.step_count() == 1
        fs.post_step()
        assert _status(fs.post_step) == B.ZERO_ESTATE  # double post_step
        # gradients are forgotten after post_step
        assert _status(fs.step) == B.ZERO_ESTATE
        torch.cuda.synchronize()
        compare_state(fs, ref, "after refused calls")
        # gather on a non-stage-3 context is a no-op that accepts NULL
        fs.gather_weights(0, None)
        assert _status(lambda: fs.gather_weights(7, None)) == B.ZERO_EINVAL
        fs.gather_units(0, [None] * fs.n_units)
        assert fs.last_launches() == 0
        assert _status(lambda: fs.gather_units(1, [None] * fs.n_units)) == B.ZERO_EINVAL
    finally:
        fs.close()


def test_stage3_gather_argument_checks():
    pb = make_problem(si.toy_mlp(), 4, 3, steps=1, seed=32)
    fs = run_gpu(pb)
    try:
        assert _status(lambda: fs.gather_weights(0, None)) == B.ZERO_EINVAL
        buf = torch.empty(4224 + 1, dtype=torch.bfloat16, device="cuda")
        assert _status(lambda: B.zero_gather_weights(fs.ctx, 0, buf.data_ptr() + 1, 0)) == B.ZERO_EINVAL
        # the runner refuses a buffer shorter than the padded unit, or not bf16
        with pytest.raises(ValueError, match="padded"):
            fs.gather_weights(0, buf[2:])
        with pytest.raises(ValueError, match="bf16"):
            fs.gather_weights(0, torch.empty(4224, dtype=torch.float32, device="cuda"))
        # unaligned (2-byte) destination works through the element-wise copy
        fs.gather_weights(0, buf[1:])
        torch.cuda.synchronize()
        assert torch.equal(buf[1:].view(torch.int16), fs.param16[:4224].view(torch.int16))
        # whole-buffer gather
        full = torch.empty(fs.padded, dtype=torch.bfloat16, device="cuda")
        fs.gather_weights(-1, full)
        torch.cuda.synchronize()
        assert torch.equal(full.view(torch.int16), fs.param16.view(torch.int16))
        # several units at once: range, NULL and alignment checks
        nu = fs.n_units
        assert _status(lambda: B.zero_gather_units(fs.ctx, 0, [0] * nu, 0)) == B.ZERO_EINVAL
        assert _status(lambda: B.zero_gather_units(fs.ctx, -1, [buf.data_ptr()], 0)) == B.ZERO_EINVAL
        assert _status(lambda: B.zero_gather_units(fs.ctx, nu, [buf.data_ptr()], 0)) == B.ZERO_EINVAL
        assert _status(lambda: B.zero_gather_units(fs.ctx, 0, [buf.data_ptr()] * (nu + 1), 0)) == B.ZERO_EINVAL
        assert _status(lambda: B.zero_gather_units(fs.ctx, 0, [buf.data_ptr() + 1], 0)) == B.ZERO_EINVAL
        assert B.load().zero_gather_units(fs.ctx, 0, 1, None, None) == B.ZERO_EINVAL  # NULL array
        assert B.load().zero_gather_units(fs.ctx, 0, -1, None, None) == B.ZERO_EINVAL  # negative count
        B.zero_gather_units(fs.ctx, nu, [], 0)  # an empty range at the end
        assert fs.last_launches() == 0
        with pytest.raises(ValueError, match="padded"):
            fs.gather_units(0, [buf[2:]])
    finally:
        fs.close()


@pytest.mark.parametrize("n,gd,tile,ctas_per_sm,threads", [(16, "bf16", 2048, 1, 256), (12, "fp32", 1024, 1, 256),
                                                            (2, "bf16", 1024, 2, 256), (4, "bf16", 2048, 1, 512),
                                                            (10, "bf16", 2048, 1, 512), (8, "bf16", 2048, 1, 512)])
def test_staged_wait_runs_out_and_the_device_stays_usable(n, gd, tile, ctas_per_sm, threads):
    # The tile-staged step kernel bounds every wait for its bulk copies.  The
    # test hook announces the launch's first tile to its mbarrier without
    # issuing the copy, so CTA 0's wait runs out (after ~1 s): it counts a
    # timeout, waits for the copies it did issue and leaves.  Exactly CTA 0's
    # elements (its tiles and its part of the ragged tail) keep their old
    # values; every other element is the oracle's; the next step on the same
    # context runs normally.
    import time
    from gpu_common import to_np
    total = (1 << 23) + 2048 * 3 + 300          # padded to a multiple of N below
    pb = make_problem(si.from_units([total]), n, 2, grad_dtype=gd, steps=2, seed=97)
    padded = pb.lay.total_padded
    fs = gpu_flatstep(pb, guard=64)
    try:
        before = B.zero_kernel_timeouts(fs.ctx)
        init = tuple(to_np(x).copy() for x in (fs.master, fs.exp_avg, fs.exp_avg_sq, fs.param16))
        flats = upload_grads(pb, 1)
        fs.reduce_grads(-1, flats)
        B.zero_debug_inject(fs.ctx, B.ZERO_INJECT_MISSING_COPY)
        t0 = time.perf_counter()
        fs.step()
        torch.cuda.synchronize()
        waited = time.perf_counter() - t0
        assert B.zero_kernel_timeouts(fs.ctx) == before + 1
        assert 0.5 < waited < 10.0, waited
        # CTA 0's elements: tiles 0, G, 2G, ... (G = the grid: SMs x CTAs per
        # SM) and the first `threads` elements after the last full tile
        grid = torch.cuda.get_device_properties(0).multi_processor_count * ctas_per_sm
        full = padded // tile
        mine = np.zeros(padded, bool)
        for tid in range(0, full, grid):
            mine[tid * tile:(tid + 1) * tile] = True
        mine[full * tile:min(full * tile + threads, padded)] = True
        ref = oracle_run(pb, steps=1)
        got = tuple(to_np(x) for x in (fs.master, fs.exp_avg, fs.exp_avg_sq, fs.param16))
        for name, g, r, i0 in zip(("master", "m", "v", "param16"), got, ref, init):
            assert np.array_equal(g[mine], i0[mine]), f"{name}: CTA 0's elements changed"
            assert np.array_equal(g[~mine], r[~mine]), f"{name}: other elements differ from the oracle"
        check_guards(fs, "after the injected timeout")
        fs.post_step()
        # the same context steps normally afterwards (no timeout, valid results
        # for every element that the first step did update)
        fs.reduce_grads(-1, upload_grads(pb, 2))
        fs.step()
        torch.cuda.synchronize()
        assert B.zero_kernel_timeouts(fs.ctx) == before + 1
        assert not np.isnan(to_np(fs.master)).any()
    finally:
        fs.close()
