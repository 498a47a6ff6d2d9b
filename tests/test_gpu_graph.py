"""Capturable steps and CUDA graphs: with the step count on the device, a
step (registration, clip, step, post_step) captured once into a CUDA graph
and replayed every iteration must give the oracle's result after every
replay; without graphs the mode must not change any result either."""

import numpy as np
import pytest
import torch

import synth_inputs as si
from gpu_common import compare_state, ensure_built, gpu_flatstep, make_problem, oracle_run, run_gpu, upload_grads
from zero_sharded_mixed_flatparameter_gb300 import binding as B

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()
    yield
    torch.cuda.empty_cache()


def _refs(pb):
    refs = {}
    oracle_run(pb, every_step=lambda t, s: refs.__setitem__(t, s))
    return refs


@pytest.mark.parametrize("name,pl,n,stage,gd,max_norm,keep", [
    ("toy MLP ZeRO-3", si.toy_mlp(), 4, 3, "bf16", 0.0, False),
    ("odd units, clipped, kept gradient", si.from_units([1552, 7, 9312, 33]), 3, 2, "bf16", 0.05, True),
    ("tile-staged N = 16", si.from_units([4_200_005, 2_000_000, 2_300_003]), 16, 2, "bf16", 0.0, False),
    ("pipelined staged N = 10, clipped", si.from_units([4_200_005, 2_000_000, 2_300_003]), 10, 3, "bf16", 0.5,
     False),
    ("fp32 N = 9 staged, clipped", si.from_units([4_200_005, 4_300_003]), 9, 1, "fp32", 0.5, False),
    ("fp32 N = 12 staged, 1,024-element tiles", si.from_units([4_200_005, 4_300_003]), 12, 2, "fp32", 0.0, False),
    ("bf16 N = 2 staged, 4 elements per thread, clipped", si.from_units([4_200_005, 4_300_003]), 2, 3, "bf16", 0.5,
     False),
])
def test_capturable_mode_matches_oracle(name, pl, n, stage, gd, max_norm, keep):
    steps = 3
    pb = make_problem(pl, n, stage, grad_dtype=gd, steps=steps, seed=400 + n, max_norm=max_norm)
    refs = _refs(pb)
    fs = gpu_flatstep(pb)
    try:
        fs.enable_capturable(max_steps=10)
        for t in range(1, steps + 1):
            fs.reduce_grads(-1, upload_grads(pb, t))
            if max_norm > 0:
                fs.clip_grad_norm(max_norm, keep_reduced=keep)
            fs.step()
            fs.post_step()
            torch.cuda.synchronize()
            compare_state(fs, refs[t], f"{name} capturable step {t}")
        assert fs.step_count() == steps
        fs.disable_capturable()
        assert fs.step_count() == steps
    finally:
        fs.close()


@pytest.mark.parametrize("stage,max_norm", [(2, 0.0), (3, 0.05), (1, 0.5)])
def test_cuda_graph_replay(stage, max_norm):
    # step 1 runs eagerly (warm-up: workspaces allocated, launch shapes
    # cached), then one step is captured and replayed for steps 2..6, each
    # replay after fresh gradients were copied into the captured buffers
    steps = 6
    pb = make_problem(si.toy_mlp(), 4, stage, steps=steps, seed=430 + stage, max_norm=max_norm)
    refs = _refs(pb)
    fs = gpu_flatstep(pb)
    try:
        fs.enable_capturable(max_steps=steps)
        static = [g.clone() for g in upload_grads(pb, 1)]

        def one_step():
            fs.reduce_grads(-1, static)
            if max_norm > 0:
                fs.clip_grad_norm(max_norm)
            fs.step()
            fs.post_step()
        one_step()
        torch.cuda.synchronize()
        compare_state(fs, refs[1], "eager step 1")
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            one_step()          # recorded, not run
        torch.cuda.synchronize()
        assert fs.step_count() == 1
        for t in range(2, steps + 1):
            for dst, src in zip(static, upload_grads(pb, t)):
                dst.copy_(src)
            graph.replay()
            torch.cuda.synchronize()
            compare_state(fs, refs[t], f"graph replay, step {t}")
        assert fs.step_count() == steps
        fs.disable_capturable()
        assert fs.step_count() == steps
    finally:
        fs.close()


def test_exhausted_table_skips_steps():
    pb = make_problem(si.toy_mlp(), 4, 2, steps=3, seed=450)
    refs = _refs(pb)
    fs = gpu_flatstep(pb)
    try:
        fs.enable_capturable(max_steps=2)
        for t in range(1, 4):
            fs.reduce_grads(-1, upload_grads(pb, t))
            fs.step()
            fs.post_step()
        torch.cuda.synchronize()
        compare_state(fs, refs[2], "third step skipped")     # the state after two steps
        with pytest.raises(B.ZeroError) as e:
            fs.step_count()
        assert e.value.status == B.ZERO_ESTATE and "exhausted" in str(e.value)
        fs.disable_capturable()
        assert fs.step_count() == 2
    finally:
        fs.close()


def test_capturable_refusals():
    pb = make_problem(si.toy_mlp(), 4, 2, steps=2, seed=460)
    fs = gpu_flatstep(pb)
    off = gpu_flatstep(pb, offload=dict(chunk=4096, threads=2))
    try:
        def status(fn):
            with pytest.raises(B.ZeroError) as e:
                fn()
            return e.value.status
        ws = torch.empty(B.zero_capturable_workspace_bytes(fs.ctx, 4), dtype=torch.uint8, device="cuda")
        host = torch.empty(ws.numel(), dtype=torch.uint8)
        assert status(lambda: B.zero_enable_capturable(fs.ctx, host.data_ptr(), ws.numel(), 4)) == B.ZERO_EINVAL
        assert status(lambda: B.zero_enable_capturable(fs.ctx, ws.data_ptr(), ws.numel() - 1, 4)) == B.ZERO_EINVAL
        assert status(lambda: B.zero_enable_capturable(fs.ctx, ws.data_ptr(), ws.numel(), 0)) == B.ZERO_EINVAL
        assert status(lambda: B.zero_disable_capturable(fs.ctx)) == B.ZERO_ESTATE
        assert status(lambda: B.zero_enable_capturable(off.ctx, ws.data_ptr(), ws.numel(), 4)) == B.ZERO_ENOTSUP
        fs.enable_capturable(max_steps=4)
        assert status(lambda: fs.export_state()) == B.ZERO_ESTATE
        fs.disable_capturable()
        # two eager steps, then a table no longer than the steps taken is refused
        for t in (1, 2):
            fs.reduce_grads(-1, upload_grads(pb, t))
            fs.step()
            fs.post_step()
        assert status(lambda: B.zero_enable_capturable(fs.ctx, ws.data_ptr(), ws.numel(), 2)) == B.ZERO_EINVAL
        torch.cuda.synchronize()
        compare_state(fs, oracle_run(pb), "after refused calls")
    finally:
        fs.close()
        off.close()


def test_capturable_step_over_several_launches():
    # 100 units registered separately: the step spans three launches (48
    # segments each), which must all read the same device step count, and
    # the count advances once per step; replayed as a graph too
    pl = si.from_units([211 + 17 * (i % 5) for i in range(100)])
    steps = 4
    pb = make_problem(pl, 3, 2, steps=steps, seed=480)
    refs = _refs(pb)
    fs = gpu_flatstep(pb)
    try:
        fs.enable_capturable(max_steps=steps)
        # one separately allocated buffer per unit and replica: the units do
        # not merge into one segment, so the step takes several launches
        spans = [fs.layout(i) for i in range(fs.n_units)]
        views = [[torch.empty(padded, dtype=torch.bfloat16, device="cuda") for _ in range(pb.n)]
                 for (numel, padded, shard, base) in spans]

        def load(t):
            for f_r, r in zip(upload_grads(pb, t), range(pb.n)):
                for (numel, padded, shard, base), v in zip(spans, views):
                    v[r].copy_(f_r[base:base + padded])
        load(1)

        def one_step():
            for i, v in enumerate(views):
                fs.reduce_grads(i, v)
            fs.step()
            fs.post_step()
        one_step()
        torch.cuda.synchronize()
        assert fs.last_launches() == 4  # 100 segments in three step launches, then the count
        compare_state(fs, refs[1], "eager step over several launches")
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            one_step()
        for t in range(2, steps + 1):
            load(t)
            graph.replay()
            torch.cuda.synchronize()
            compare_state(fs, refs[t], f"replay {t} over several launches")
        assert fs.step_count() == steps
    finally:
        fs.close()
