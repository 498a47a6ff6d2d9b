"""Checkpoint export/import with resharding on the GPU.

A checkpoint keeps the real elements only (the pads are not parameters), so
it can be resumed under another shard count N' and stage.  Every replica
receives the same bf16 gradient here, which makes the average the same at
any N (see the oracle test), so the resumed run must match an uninterrupted
one bit for bit."""

import numpy as np
import pytest
import torch

import oracle
import synth_inputs as si
from gpu_common import ensure_built, to_np
from zero_sharded_mixed_flatparameter_gb300 import binding as B
from zero_sharded_mixed_flatparameter_gb300.runner import FlatStep

pytestmark = pytest.mark.gpu

PL = si.from_units([1552, 7, 33, 9312, 16384 + 3])


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


def _grads(step):
    rng = np.random.default_rng(100 + step)
    return [torch.tensor(rng.normal(0, 1e-2, k).astype(np.float32)).to(torch.bfloat16) for k in PL.numel]


def _make(n, stage, init):
    return FlatStep(PL.numel, PL.unit, stage=stage, n_ranks=n, adamw=True, weight_decay=0.1,
                    init_params=[x.cuda() for x in init], guard=64)


def _run(fs, t0, t1):
    for t in range(t0, t1):
        per_param = _grads(t)
        flat = torch.zeros(fs.padded, dtype=torch.bfloat16, device="cuda")
        for p, g in enumerate(per_param):
            off = fs.param_offset(p)
            flat[off:off + g.numel()] = g.cuda()
        fs.reduce_grads(-1, [flat] * fs.n_ranks)
        fs.step()
        fs.post_step()
    torch.cuda.synchronize()


def _init():
    rng = np.random.default_rng(99)
    return [torch.tensor(rng.normal(0, 0.02, k).astype(np.float32)) for k in PL.numel]


def test_export_matches_oracle():
    init = _init()
    fs = _make(4, 3, init)
    try:
        _run(fs, 0, 2)
        (master, m, v), t = fs.export_state()
        torch.cuda.synchronize()
        assert t == 2
        ref = [to_np(x) for x in (fs.master, fs.exp_avg, fs.exp_avg_sq)]
        lay = oracle.layout(PL.numel, PL.unit, 4, 3)
        for got, padded in zip((master, m, v), ref):
            assert np.array_equal(to_np(got).view(np.uint32), oracle.export_state(lay, padded).view(np.uint32))
    finally:
        fs.close()


@pytest.mark.parametrize("first,second", [((8, 3), (3, 1)), ((3, 2), (16, 3)), ((5, 1), (1, 0))])
def test_resharded_resume_equals_uninterrupted(first, second):
    init = _init()
    whole = _make(*first, init)
    part = _make(*first, init)
    try:
        _run(whole, 0, 6)
        _run(part, 0, 3)
        (master, m, v), t = part.export_state()
        torch.cuda.synchronize()
        resumed = _make(*second, init)
        try:
            resumed.import_state(master, m, v, t)
            assert resumed.step_count() == 3
            # param16 is the bf16 of the imported master; pads are zero
            lay = oracle.layout(PL.numel, PL.unit, second[0], second[1])
            assert np.array_equal(to_np(resumed.param16), oracle.bf16_round(to_np(resumed.master)))
            for i in range(resumed.n_units):
                numel, padded, shard, base = resumed.layout(i)
                assert not torch.any(resumed.master[base + numel:base + padded] != 0).item()
            _run(resumed, 3, 6)
            (a, b, c), ta = whole.export_state()
            (x, y, z), tr = resumed.export_state()
            torch.cuda.synchronize()
            assert ta == tr == 6
            for p, q in ((a, x), (b, y), (c, z)):
                assert torch.equal(p.view(torch.int32), q.view(torch.int32))
            for gbuf in resumed.guards():
                assert torch.isnan(gbuf.float()).all().item()
        finally:
            resumed.close()
    finally:
        whole.close()
        part.close()


def test_checkpoint_errors():
    init = _init()
    fs = _make(4, 2, init)
    host = torch.zeros(fs.numel)
    dev = torch.zeros(fs.numel, device="cuda")
    try:
        def st(fn):
            with pytest.raises(B.ZeroError) as e:
                fn()
            return e.value.status
        assert st(lambda: B.zero_export_state(fs.ctx, 0, dev.data_ptr(), dev.data_ptr(), 0)) == B.ZERO_EINVAL
        assert st(lambda: B.zero_export_state(fs.ctx, host.data_ptr(), dev.data_ptr(), dev.data_ptr(), 0)) \
            == B.ZERO_EINVAL
        assert st(lambda: B.zero_import_state(fs.ctx, dev.data_ptr(), dev.data_ptr(), dev.data_ptr(), -1, 0)) \
            == B.ZERO_EINVAL
        assert st(lambda: B.zero_import_state(fs.ctx, dev.data_ptr() + 2, dev.data_ptr(), dev.data_ptr(), 0, 0)) \
            == B.ZERO_EINVAL
        flat = torch.zeros(fs.padded, dtype=torch.bfloat16, device="cuda")
        fs.reduce_grads(-1, [flat] * 4)
        fs.step()
        assert st(lambda: B.zero_import_state(fs.ctx, dev.data_ptr(), dev.data_ptr(), dev.data_ptr(), 0, 0)) \
            == B.ZERO_ESTATE
        assert fs.step_count() == 1
        fs.post_step()
    finally:
        fs.close()
