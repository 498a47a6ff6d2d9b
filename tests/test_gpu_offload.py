"""ZeRO-Offload on the GPU: fp32 master / m / v in host memory, the reduced
gradient copied down chunk by chunk, the library's CPU Adam on the host and
the bf16 parameters copied back up (CMU 15-779 Lecture 13 notes §7.1-7.2).

The offloaded step is the device step's arithmetic, so it is checked against
the oracle bit for bit and against a GPU-resident run of the same problem."""

import numpy as np
import pytest
import torch

import synth_inputs as si
from gpu_common import (compare_state, ensure_built, make_problem, oracle_run, run_gpu, to_np, upload_grads,
                        gpu_flatstep)
from zero_sharded_mixed_flatparameter_gb300 import binding as B
from zero_sharded_mixed_flatparameter_gb300.runner import FlatStep

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()
    yield
    torch.cuda.empty_cache()


def _per_step(pb, mode, offload):
    refs = {}
    oracle_run(pb, every_step=lambda t, s: refs.__setitem__(t, s))
    fs = run_gpu(pb, mode=mode, offload=offload,
                 every_step=lambda t, f: compare_state(f, refs[t], f"offload {offload} step {t}"))
    fs.close()


@pytest.mark.parametrize("stage", [0, 1, 2, 3])
def test_toy_mlp_all_stages(stage):
    # 34,192 params, N = 4, 5 steps; chunks of 1,000 elements cut units (and
    # 8-element groups) anywhere, so both the vector and the element path of
    # the chunk reduction run
    pb = make_problem(si.toy_mlp(), 4, stage, steps=5, seed=31 + stage)
    _per_step(pb, "units", dict(chunk=1000, threads=3))


@pytest.mark.parametrize("chunk,threads", [(1, 1), (64, 2), (4096, 0), (1 << 22, 4)])
def test_chunk_and_thread_counts(chunk, threads):
    # chunk = 1 element (every chunk its own ring slot), a multiple of 8,
    # larger than the buffer; 1..all threads
    pl = si.from_units([1552, 7, 9312, 33])
    n_steps = 2 if chunk == 1 else 4
    pb = make_problem(pl, 3, 2, steps=n_steps, seed=40 + threads)
    _per_step(pb, "separate", dict(chunk=chunk, threads=threads))


@pytest.mark.parametrize("n,gd", [(1, "bf16"), (8, "bf16"), (16, "bf16"), (2, "fp32"), (5, "fp32")])
def test_rank_counts_and_dtypes(n, gd):
    pl = si.from_units([3 * 2048 + 5, 40, 1000])
    pb = make_problem(pl, n, 2, grad_dtype=gd, steps=3, seed=50 + n)
    _per_step(pb, "all", dict(chunk=2000, threads=4))


def test_adamw_and_clip():
    pl = si.from_units([9312, 1552, 17])
    pb = make_problem(pl, 4, 3, steps=4, seed=61, adamw=True, weight_decay=0.1, max_norm=0.05)
    norms_ref, norms = [], []
    ref = oracle_run(pb, norms=norms_ref)
    fs = run_gpu(pb, mode="units", offload=dict(chunk=3000, threads=2), norms=norms)
    compare_state(fs, ref, "offload adamw + clip")
    fs.close()
    assert np.allclose(norms, norms_ref, rtol=1e-12, atol=0)
    assert all(x > 0.05 for x in norms_ref)  # the clip was active


def test_equals_gpu_resident_run():
    # 2.1 M params, 10 units, N = 8, clipped: offloaded and GPU-resident
    # states bit-identical after every step
    pl = si.from_units([200_003] * 10 + [7])
    pb = make_problem(pl, 8, 2, steps=3, seed=70, max_norm=1.0)
    a = gpu_flatstep(pb)
    b = gpu_flatstep(pb, offload=dict(chunk=1 << 18, threads=0))
    try:
        for t in range(1, 4):
            flats = upload_grads(pb, t)
            for fs in (a, b):
                fs.reduce_grads(-1, flats)
                fs.clip_grad_norm(pb.max_norm)
                fs.step()
                fs.post_step()
            torch.cuda.synchronize()
            for name in ("master", "exp_avg", "exp_avg_sq", "param16"):
                x, y = to_np(getattr(a, name)), to_np(getattr(b, name))
                assert np.array_equal(x.view(np.uint32) if x.dtype == np.float32 else x,
                                      y.view(np.uint32) if y.dtype == np.float32 else y), f"step {t} {name}"
    finally:
        a.close()
        b.close()


def test_checkpoint_between_offload_and_gpu_contexts():
    # GPU-resident run -> export -> import into an offload context (other N
    # and stage) -> continue; and back.  Identical replicas make the reduced
    # gradient independent of N, so every path must equal the uninterrupted run.
    pl = si.from_units([1552, 7, 9312, 16384 + 3])
    steps = 6
    rng = np.random.default_rng(5)
    gs = [rng.normal(0, 1e-2, sum(pl.numel)).astype(np.float32) for _ in range(steps)]

    def make(n, stage, offload):
        init = [torch.from_numpy(np.random.default_rng(9).normal(0, 0.02, k).astype(np.float32)).cuda()
                for k in pl.numel]
        kw = dict(offload=True, offload_chunk=5000, offload_threads=2) if offload else {}
        return FlatStep(pl.numel, pl.unit, stage=stage, n_ranks=n, init_params=init, **kw)

    def do_step(fs, t):
        flat = torch.zeros(fs.padded, dtype=torch.bfloat16, device="cuda")
        cum = 0
        for p, k in enumerate(pl.numel):
            o = fs.param_offset(p)
            flat[o:o + k] = torch.from_numpy(gs[t][cum:cum + k]).cuda().to(torch.bfloat16)
            cum += k
        fs.reduce_grads(-1, [flat] * fs.n_ranks)
        fs.step()
        fs.post_step()

    def real(fs):
        out, t = fs.export_state()
        torch.cuda.synchronize()
        return [to_np(x) for x in out], t

    ref = make(4, 2, False)
    for t in range(steps):
        do_step(ref, t)
    want, want_t = real(ref)
    ref.close()
    for first, second in ((False, True), (True, False)):
        a = make(3, 1, first)
        for t in range(3):
            do_step(a, t)
        state, t0 = a.export_state()
        b = make(5, 3, second)
        b.import_state(*state, t0)
        a.close()
        for t in range(3, steps):
            do_step(b, t)
        got, got_t = real(b)
        assert got_t == want_t
        for x, y in zip(got, want):
            assert np.array_equal(x.view(np.uint32), y.view(np.uint32))
        b.close()


def test_errors_and_refusals():
    pl = si.from_units([1000, 24])
    pb = make_problem(pl, 2, 2, steps=1, seed=80)
    fs = gpu_flatstep(pb, offload=dict(chunk=256, threads=1))
    gpu = gpu_flatstep(pb)
    try:
        flats = upload_grads(pb, 1)
        fs.reduce_grads(-1, flats)
        gpu.reduce_grads(-1, flats)
        s = fs.stream_handle()
        with pytest.raises(B.ZeroError) as e:
            B.zero_step(fs.ctx, s)  # the offload context steps through zero_offload_step only
        assert e.value.status == B.ZERO_ESTATE
        hb, db = B.zero_offload_workspace_bytes(fs.ctx, 256)
        hw, dw = fs._host_ws.data_ptr(), fs._dev_ws.data_ptr()
        with pytest.raises(B.ZeroError) as e:
            B.zero_offload_step(gpu.ctx, 256, hw, hb, dw, db, 1, s)  # not an offload context
        assert e.value.status == B.ZERO_ESTATE
        for bad in (dict(chunk=0), dict(hb=hb - 1), dict(db=db - 4), dict(threads=-1)):
            kw = dict(chunk=256, hb=hb, db=db, threads=1)
            kw.update(bad)
            with pytest.raises(B.ZeroError) as e:
                B.zero_offload_step(fs.ctx, kw["chunk"], hw, kw["hb"], dw, kw["db"], kw["threads"], s)
            assert e.value.status == B.ZERO_EINVAL
        pageable = torch.empty(hb, dtype=torch.uint8)
        with pytest.raises(B.ZeroError) as e:
            B.zero_offload_step(fs.ctx, 256, pageable.data_ptr(), hb, dw, db, 1, s)
        assert e.value.status == B.ZERO_EINVAL and "pinned" in str(e.value)
        with pytest.raises(B.ZeroError) as e:  # device workspace given as host memory
            B.zero_offload_step(fs.ctx, 256, hw, hb, hw, db, 1, s)
        assert e.value.status == B.ZERO_EINVAL
        ws = torch.empty(B.zero_clip_workspace_bytes_ex(fs.ctx, B.ZERO_CLIP_KEEP_REDUCED), dtype=torch.uint8,
                         device="cuda")
        with pytest.raises(B.ZeroError) as e:
            B.zero_clip_grad_norm_ex(fs.ctx, 1.0, B.ZERO_CLIP_KEEP_REDUCED, ws.data_ptr(), ws.numel(), s)
        assert e.value.status == B.ZERO_ENOTSUP
        # nothing above changed the state: the step still runs and matches the oracle
        fs.step()
        fs.post_step()
        torch.cuda.synchronize()
        compare_state(fs, oracle_run(pb), "after refused calls")
    finally:
        fs.close()
        gpu.close()


def test_make_master_offload_rejects_device_state():
    pl = si.from_units([64])
    cfg = B.make_config(2, 2)
    dev = [torch.zeros(64, device="cuda") for _ in range(3)]
    p16 = torch.zeros(64, dtype=torch.bfloat16, device="cuda")
    init = torch.zeros(64, device="cuda")
    with pytest.raises(B.ZeroError) as e:
        B.zero_make_master_offload(cfg, pl.numel, pl.unit, [init.data_ptr()], *(d.data_ptr() for d in dev),
                                   p16.data_ptr())
    assert e.value.status == B.ZERO_EINVAL
    host = [torch.zeros(64) for _ in range(3)]
    with pytest.raises(B.ZeroError) as e:  # param16 must be device memory
        B.zero_make_master_offload(cfg, pl.numel, pl.unit, [init.data_ptr()], *(h.data_ptr() for h in host),
                                   torch.zeros(64, dtype=torch.bfloat16).data_ptr())
    assert e.value.status == B.ZERO_EINVAL


def test_many_units_span_several_reduce_launches():
    # 100 units (more than the 48 segments one reduce launch takes) with
    # chunks that span dozens of units each, ZeRO-3, clipped
    pl = si.from_units([97 + 13 * (i % 7) for i in range(100)])
    pb = make_problem(pl, 4, 3, steps=3, seed=470, max_norm=0.05)
    _per_step(pb, "separate", dict(chunk=5000, threads=3))
