"""Host-side failure detection of the C ABI on a GPU machine: every bad call
returns a status (never a fault) and leaves the context unchanged.  The
failures are made on the host (bad pointers, wrong order of calls); no test
here asks the GPU to fault, trap or hang."""

import ctypes

import pytest
import torch

import synth_inputs as si
from gpu_common import compare_state, ensure_built, make_problem, oracle_run, register, run_gpu, upload_grads
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
    finally:
        fs.close()


def test_stage3_gather_argument_checks():
    pb = make_problem(si.toy_mlp(), 4, 3, steps=1, seed=32)
    fs = run_gpu(pb)
    try:
        assert _status(lambda: fs.gather_weights(0, None)) == B.ZERO_EINVAL
        buf = torch.empty(4224 + 1, dtype=torch.bfloat16, device="cuda")
        assert _status(lambda: B.zero_gather_weights(fs.ctx, 0, buf.data_ptr() + 1, 0)) == B.ZERO_EINVAL
        # unaligned (2-byte) destination works through the element-wise copy
        fs.gather_weights(0, buf[1:])
        torch.cuda.synchronize()
        assert torch.equal(buf[1:].view(torch.int16), fs.param16[:4224].view(torch.int16))
        # whole-buffer gather
        full = torch.empty(fs.padded, dtype=torch.bfloat16, device="cuda")
        fs.gather_weights(-1, full)
        torch.cuda.synchronize()
        assert torch.equal(full.view(torch.int16), fs.param16.view(torch.int16))
    finally:
        fs.close()
