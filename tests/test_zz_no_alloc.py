"""zero_clip_grad_norm_static — gradient clipping for callers that cannot
allocate device memory (code inside an allocator or an out-of-memory handler,
or a loop where allocation is forbidden), so cannot hand in a workspace.

The static-scratch call must give what the workspace call gives.  Two twin
contexts run the same seeded problem for two steps in a row: one clips with
a caller workspace, the other through the library's fixed scratch; norms must
agree within the clip tests' 1e-12 and the states within the parity
tolerances (they are expected to be bit-identical).  This file is collected
last so that a failure here comes after every other test has run."""

import os
import subprocess
import sys

import pytest
import torch

import synth_inputs as si
from gpu_common import compare_state, ensure_built, gpu_flatstep, make_problem, register, to_np, upload_grads
from zero_sharded_mixed_flatparameter_gb300 import binding as B

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


def _state(fs):
    return (to_np(fs.master), to_np(fs.exp_avg), to_np(fs.exp_avg_sq), to_np(fs.param16))


@pytest.mark.parametrize("n,stage", [(4, 2), (3, 3)])
def test_static_scratch_clip_matches_workspace_clip(n, stage):
    pl = si.from_units([4224, 16384 * 2 + 5, 1552, 7])
    pb = make_problem(pl, n, stage, steps=2, seed=61 + n, max_norm=0.5)
    with_ws, static = gpu_flatstep(pb), gpu_flatstep(pb)
    try:
        for t in (1, 2):
            flats = upload_grads(pb, t)
            keep = []
            register(with_ws, pb, flats, "units", keep)
            register(static, pb, flats, "units", keep)
            with_ws.clip_grad_norm(pb.max_norm)
            B.zero_clip_grad_norm_static(static.ctx, pb.max_norm, static.stream_handle())
            n_ws, n_static = with_ws.grad_norm(), static.grad_norm()
            assert n_ws > pb.max_norm  # the clip is active
            assert abs(n_static - n_ws) <= 1e-12 * n_ws
            with_ws.step()
            static.step()
            with_ws.post_step()
            static.post_step()
            torch.cuda.synchronize()
            compare_state(_state(static), _state(with_ws), f"static-scratch clip, call {t}")
    finally:
        with_ws.close()
        static.close()


def test_static_scratch_rejects_layouts_beyond_its_size():
    ctx = B.zero_plan(B.make_config(2, 8), [3_000_000_000], [0])
    try:
        with pytest.raises(B.ZeroError) as e:
            B.zero_clip_grad_norm_static(ctx, 1.0, 0)
        assert e.value.status == B.ZERO_EINVAL
        assert "static scratch" in B.zero_last_error(ctx)
    finally:
        B.zero_destroy(ctx)


def test_static_scratch_in_every_cuda_context():
    # The scratch array has one copy per CUDA context; a caller running in a
    # second context of the GPU (or in one created after another was
    # destroyed) must get its own context's copy, never an address from
    # another context.  Run in a subprocess without torch, every buffer made
    # with the driver API in the context that uses it (the scenario also
    # steps a tile-staged kernel in each context).
    here = os.path.dirname(os.path.abspath(__file__))
    r = subprocess.run([sys.executable, os.path.join(here, "no_alloc_contexts_scenario.py")], capture_output=True,
                       text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-3000:]
    assert r.stdout.strip().splitlines()[-1] == "all contexts ok"
