"""fp32 gradient accumulation over micro-steps on the GPU against the oracle
(bit-exact: one fp32 addition per micro-step on both sides), and the
accumulate -> reduce_grads -> step pipeline on an fp32-gradient context."""

import numpy as np
import pytest
import torch

import oracle
import synth_inputs as si
from gpu_common import compare_state, ensure_built, gpu_flatstep, make_problem, oracle_run, to_np
from zero_sharded_mixed_flatparameter_gb300 import binding as B

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


def _micro(n, total, k, seed):
    return [si.replica_grads(n, total, 1e-2, seed * 1000 + i, "bf16") for i in range(k)]


@pytest.mark.parametrize("n", [1, 2, 5, 8, 16])
@pytest.mark.parametrize("offset", [0, 1])
def test_accumulate_parity(n, offset):
    # buffers offset by one element take the element-wise kernel
    pl = si.from_units([3 * 256 * 8 + 5])
    pb = make_problem(pl, n, 1, grad_dtype="fp32", steps=1, seed=71)
    fs = gpu_flatstep(pb)
    try:
        total, K = fs.padded, 4
        micro = _micro(n, total, K, 72 + n)
        acc_host = [np.full(total, np.nan, np.float32) for _ in range(n)]
        dev_acc_bufs = [torch.full((total + 8,), float("nan"), device="cuda") for _ in range(n)]
        dev_acc = [b[offset:offset + total] for b in dev_acc_bufs]
        for k in range(K):
            oracle.accumulate([to_np(g) for g in micro[k]], acc_host, first=(k == 0))
            dev_micro_bufs = [torch.zeros(total + 8, dtype=torch.bfloat16, device="cuda") for _ in range(n)]
            for b, g in zip(dev_micro_bufs, micro[k]):
                b[offset:offset + total] = g.cuda()
            fs.accumulate_grads(-1, [b[offset:offset + total] for b in dev_micro_bufs], dev_acc, first=(k == 0))
        torch.cuda.synchronize()
        for a, b in zip(dev_acc, acc_host):
            assert np.array_equal(to_np(a).view(np.uint32), b.view(np.uint32))
        # the guard elements around the accumulators are untouched
        for b in dev_acc_bufs:
            assert torch.isnan(b[:offset]).all() and torch.isnan(b[offset + total:]).all()
    finally:
        fs.close()


def test_accumulate_then_step_pipeline():
    # K = 3 micro-steps per optimizer step, 3 steps, ZeRO-2, N = 4, per-unit accumulation
    pl = si.toy_mlp()
    n, K, steps = 4, 3, 3
    pb = make_problem(pl, n, 2, grad_dtype="fp32", steps=steps, seed=73)
    fs = gpu_flatstep(pb)
    master, m, v, p16 = oracle.make_master(pl.numel, pb.lay, pb.init)
    try:
        total = fs.padded
        acc = [torch.empty(total, dtype=torch.float32, device="cuda") for _ in range(n)]
        acc_host = [np.zeros(total, np.float32) for _ in range(n)]
        for t in range(1, steps + 1):
            micro = _micro(n, total, K, 74 + t)
            for k in range(K):
                # zero the pads like the hook does, then accumulate unit by unit
                for i in range(fs.n_units):
                    numel, padded, shard, base = fs.layout(i)
                    for g in micro[k]:
                        g[base + numel:base + padded] = 0
                    fs.accumulate_grads(i, [g[base:base + padded].cuda() for g in micro[k]],
                                        [a[base:base + padded] for a in acc], first=(k == 0))
                oracle.accumulate([to_np(g) for g in micro[k]], acc_host, first=(k == 0))
            fs.reduce_grads(-1, acc)
            fs.step()
            fs.post_step()
            oracle.zero_step(pb.hyper, 2, t, pb.lay, acc_host, master, m, v, p16)
        torch.cuda.synchronize()
        compare_state(fs, (master, m, v, p16), "accumulate+step")
    finally:
        fs.close()


def test_accumulate_errors():
    pb = make_problem(si.from_units([64]), 2, 1, steps=1, seed=75)  # bf16 context
    fs = gpu_flatstep(pb)
    g = torch.zeros(64, dtype=torch.bfloat16, device="cuda")
    a = torch.zeros(64, dtype=torch.float32, device="cuda")
    try:
        with pytest.raises(B.ZeroError) as e:
            B.zero_accumulate_grads(fs.ctx, -1, [g.data_ptr()] * 2, [a.data_ptr()] * 2, True, 0)
        assert e.value.status == B.ZERO_EINVAL and "fp32" in B.zero_last_error(fs.ctx)
    finally:
        fs.close()
    pb = make_problem(si.from_units([64]), 2, 1, grad_dtype="fp32", steps=1, seed=75)
    fs = gpu_flatstep(pb)
    try:
        for micro, accs, unit in [([g.data_ptr(), 0], [a.data_ptr()] * 2, -1),
                                  ([g.data_ptr() + 1] * 2, [a.data_ptr()] * 2, -1),
                                  ([g.data_ptr()] * 2, [a.data_ptr() + 2] * 2, -1),
                                  ([g.data_ptr()] * 2, [a.data_ptr()] * 2, 3)]:
            with pytest.raises(B.ZeroError) as e:
                B.zero_accumulate_grads(fs.ctx, unit, micro, accs, False, 0)
            assert e.value.status == B.ZERO_EINVAL
        B.zero_accumulate_grads(fs.ctx, -1, [g.data_ptr()] * 2, [a.data_ptr()] * 2, True, 0)
        assert B.zero_last_launches(fs.ctx) == 1
    finally:
        fs.close()
