"""Global-norm gradient clipping on the GPU against the oracle.

The oracle sums the squares of the reduced gradient in fp64 in element order
(the plain definition); the GPU sums fixed chunks in a fixed order with
~48-bit per-thread accumulation.  Norms must agree to 1e-12 relative; the
fp32 clip coefficients (and hence all state) then agree bit for bit except
when the two norms straddle an fp32 rounding boundary, which these seeded
cases do not.  GPU runs of every stage must be bit-identical (the chunking
is unit-relative and the pads add zeros)."""

import numpy as np
import pytest
import torch

import oracle
import synth_inputs as si
from gpu_common import (compare_state, ensure_built, gpu_flatstep, make_problem, oracle_run, register, run_gpu,
                        to_np, upload_grads)
from zero_sharded_mixed_flatparameter_gb300 import binding as B

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


def _clip_parity(pb, mode="units", keep=False):
    ref_states, ref_norms, gpu_norms = {}, [], []
    oracle_run(pb, every_step=lambda t, s: ref_states.__setitem__(t, s), norms=ref_norms)

    def check(t, fs):
        compare_state(fs, ref_states[t], f"clipped step {t}")
    fs = run_gpu(pb, mode=mode, every_step=check, norms=gpu_norms, clip_keep=keep)
    fs.close()
    for a, b in zip(gpu_norms, ref_norms):
        assert abs(a - b) <= 1e-12 * abs(b), (a, b)
    return ref_norms


@pytest.mark.parametrize("stage", [0, 1, 2, 3])
def test_toy_mlp_clipped(stage):
    # grads ~N(0, 1e-2) over 34,192 params: norm ~1.85, clipped to 0.5
    pb = make_problem(si.toy_mlp(), 4, stage, steps=10, seed=41, max_norm=0.5)
    norms = _clip_parity(pb)
    assert all(x > 0.5 for x in norms)


def test_inactive_clip_equals_no_clip():
    pb = make_problem(si.toy_mlp(), 4, 2, steps=3, seed=42, max_norm=1e6)
    fs_clip = run_gpu(pb)
    pb.max_norm = 0.0
    fs_plain = run_gpu(pb)
    for a, b in ((fs_clip.master, fs_plain.master), (fs_clip.exp_avg, fs_plain.exp_avg),
                 (fs_clip.exp_avg_sq, fs_plain.exp_avg_sq), (fs_clip.param16, fs_plain.param16)):
        assert torch.equal(a.view(torch.int16 if a.dtype == torch.bfloat16 else torch.int32),
                           b.view(torch.int16 if b.dtype == torch.bfloat16 else torch.int32))
    fs_clip.close()
    fs_plain.close()


@pytest.mark.parametrize("n,gd", [(5, "fp32"), (16, "bf16"), (3, "bf16"), (6, "fp32"), (7, "fp32"), (12, "fp32")])
def test_odd_layouts_clipped(n, gd):
    # units straddling chunk boundaries, an exact multiple of the chunk, empty
    # units; fp32 from 7 replicas on loads one group at a time
    pl = si.from_units([16384 * 2, 16384 + 1, 0, 7, 16384 * 3 - 5, 33])
    pb = make_problem(pl, n, 3, grad_dtype=gd, steps=3, seed=43 + n, max_norm=0.1)
    _clip_parity(pb, mode="separate")
    _clip_parity(pb, mode="units")


def test_clipped_stages_bit_identical():
    pl = si.from_units([16384 * 2, 1552, 16384 + 3, 9])
    out = {}
    for stage in (0, 1, 2, 3):
        pb = make_problem(pl, 3, stage, steps=4, seed=44, max_norm=0.3)
        norms = []
        fs = run_gpu(pb, norms=norms)
        vals = []
        for buf in (fs.master, fs.exp_avg, fs.exp_avg_sq, fs.param16):
            a = to_np(buf)
            vals.append(np.concatenate([a[fs.param_offset(p):fs.param_offset(p) + k] for p, k in enumerate(pl.numel)]))
        out[stage] = (norms, vals)
        fs.close()
    for stage in (1, 2, 3):
        assert out[stage][0] == out[0][0]
        for a, b in zip(out[0][1], out[stage][1]):
            assert np.array_equal(a.view(np.uint8), b.view(np.uint8))


def test_norm_independent_of_alignment():
    # the same gradients through 16-byte-aligned buffers (vector loads) and
    # buffers offset by one element (element-wise loads) give the same norm
    pl = si.from_units([40_000])
    pb = make_problem(pl, 4, 2, steps=1, seed=45, max_norm=0.1)
    norms = []
    for offset in (0, 1):
        fs = gpu_flatstep(pb)
        flats = upload_grads(pb, 1)
        shifted = []
        for f in flats:
            buf = torch.zeros(f.numel() + 8, dtype=f.dtype, device=f.device)
            buf[offset:offset + f.numel()] = f
            shifted.append(buf[offset:offset + f.numel()])
        fs.reduce_grads(0, shifted)
        fs.clip_grad_norm(0.1)
        norms.append(fs.grad_norm())
        fs.step()
        fs.post_step()
        fs.close()
    assert norms[0] == norms[1]


def test_many_units_clipped():
    sizes = [(8 * (i % 5) + 8) * 4 for i in range(130)]
    pb = make_problem(si.from_units(sizes), 4, 3, steps=2, seed=46, max_norm=0.05)
    _clip_parity(pb, mode="separate")


def test_clip_errors():
    pb = make_problem(si.toy_mlp(), 4, 2, steps=1, seed=47)
    fs = gpu_flatstep(pb)
    try:
        need = B.zero_clip_workspace_bytes(fs.ctx)
        assert need == 32 + 8 * sum(-(-k // 16384) for k in [4224, 16512, 8256, 4160, 1040])
        ws = torch.empty(need + 16, dtype=torch.uint8, device="cuda")
        host = torch.empty(need, dtype=torch.uint8)

        def st(fn):
            with pytest.raises(B.ZeroError) as e:
                fn()
            return e.value.status
        assert st(lambda: B.zero_grad_norm(fs.ctx, 0)) == B.ZERO_ESTATE
        assert st(lambda: B.zero_clip_grad_norm(fs.ctx, 1.0, ws.data_ptr(), need, 0)) == B.ZERO_ESTATE  # no grads
        register(fs, pb, upload_grads(pb, 1), "units", [])
        assert st(lambda: B.zero_clip_grad_norm(fs.ctx, 0.0, ws.data_ptr(), need, 0)) == B.ZERO_EINVAL
        assert st(lambda: B.zero_clip_grad_norm(fs.ctx, float("nan"), ws.data_ptr(), need, 0)) == B.ZERO_EINVAL
        assert st(lambda: B.zero_clip_grad_norm(fs.ctx, 1.0, 0, need, 0)) == B.ZERO_EINVAL
        assert st(lambda: B.zero_clip_grad_norm(fs.ctx, 1.0, ws.data_ptr() + 8, need, 0)) == B.ZERO_EINVAL
        assert st(lambda: B.zero_clip_grad_norm(fs.ctx, 1.0, ws.data_ptr(), need - 8, 0)) == B.ZERO_EINVAL
        assert st(lambda: B.zero_clip_grad_norm(fs.ctx, 1.0, host.data_ptr(), need, 0)) == B.ZERO_EINVAL
        stream = fs.stream_handle()
        B.zero_clip_grad_norm(fs.ctx, 1.0, ws.data_ptr(), need, stream)
        assert B.zero_last_launches(fs.ctx) == 2
        nrm = B.zero_grad_norm(fs.ctx, stream)
        ref = oracle.grad_norm(pb.hyper, pb.grads[0])
        assert abs(nrm - ref) <= 1e-12 * ref
        fs.step()
        assert st(lambda: B.zero_clip_grad_norm(fs.ctx, 1.0, ws.data_ptr(), need, stream)) == B.ZERO_ESTATE
        fs.post_step()
        assert B.zero_grad_norm(fs.ctx, stream) == nrm  # still readable after the step
    finally:
        fs.close()


def test_full_size_llama_1024_clipped():
    # 73,417,728 params, N = 8, ZeRO-2, two clipped steps; the oracle computes
    # the full norm from the gradients copied back, then checks windows
    pl = si.llama_1024()
    n, steps, max_norm = 8, 2, 1.0
    lay = oracle.layout(pl.numel, pl.unit, n, 2)
    init_flat = si.normal_fp32(pl.total, 0.02, 51, device="cuda")
    from zero_sharded_mixed_flatparameter_gb300.runner import FlatStep
    fs = FlatStep(pl.numel, pl.unit, stage=2, n_ranks=n, init_params=[init_flat[int(o):int(o) + k]
                  for o, k in zip(np.concatenate([[0], np.cumsum(pl.numel)[:-1]]), pl.numel)])
    rng = np.random.default_rng(52)
    starts = sorted({0, lay.total_padded - 256, *rng.integers(0, lay.total_padded - 256, 40).tolist()})
    win = {a: [to_np(init_flat[a:a + 256]), np.zeros(256, np.float32), np.zeros(256, np.float32),
               np.zeros(256, np.uint16)] for a in starts}
    del init_flat
    h = oracle.Hyper(n_ranks=n)
    try:
        for t in range(1, steps + 1):
            grads = si.replica_grads(n, lay.total_padded, 1e-3, 53 + t, "bf16", device="cuda")
            host = [to_np(g) for g in grads]
            ref_norm = oracle.grad_norm(h, host)
            coef = oracle.clip_coef(ref_norm, max_norm)
            assert coef < 1.0
            fs.reduce_grads(-1, grads)
            fs.clip_grad_norm(max_norm)
            gpu_norm = fs.grad_norm()
            assert abs(gpu_norm - ref_norm) <= 1e-12 * ref_norm
            fs.step()
            fs.post_step()
            for a in starts:
                oracle.step_window(h, t, [x[a:a + 256] for x in host], *win[a], clip_coef=coef)
            del grads, host
        torch.cuda.synchronize()
        for a in starts:
            got = (to_np(fs.master[a:a + 256]), to_np(fs.exp_avg[a:a + 256]), to_np(fs.exp_avg_sq[a:a + 256]),
                   to_np(fs.param16[a:a + 256]))
            compare_state(got, win[a], f"window@{a}")
    finally:
        fs.close()
        torch.cuda.empty_cache()


@pytest.mark.parametrize("n,gd,stage", [(8, "bf16", 2), (3, "fp32", 3), (16, "bf16", 0), (5, "bf16", 1)])
def test_keep_reduced_gradient(n, gd, stage):
    # the step reads the kept reduced gradient instead of the replicas; the
    # results are the oracle's bit for bit.  Units of 1,552 at N = 3 or 5 give
    # unit bases that are not multiples of 4, i.e. unaligned kept stores.
    pl = si.from_units([16384 * 2 + 5, 1552, 7, 4099])
    pb = make_problem(pl, n, stage, grad_dtype=gd, steps=3, seed=48 + n, max_norm=0.2)
    _clip_parity(pb, mode="separate", keep=True)
    _clip_parity(pb, mode="units", keep=True)


def test_keep_reduced_errors():
    pb = make_problem(si.toy_mlp(), 4, 2, steps=1, seed=49)
    fs = gpu_flatstep(pb)
    try:
        register(fs, pb, upload_grads(pb, 1), "units", [])
        small = B.zero_clip_workspace_bytes(fs.ctx)
        big = B.zero_clip_workspace_bytes_ex(fs.ctx, B.ZERO_CLIP_KEEP_REDUCED)
        assert big >= small + 4 * fs.padded
        ws = torch.empty(big, dtype=torch.uint8, device="cuda")
        for flags, nbytes in ((2, big), (B.ZERO_CLIP_KEEP_REDUCED, big - 4)):
            with pytest.raises(B.ZeroError) as e:
                B.zero_clip_grad_norm_ex(fs.ctx, 1.0, flags, ws.data_ptr(), nbytes, 0)
            assert e.value.status == B.ZERO_EINVAL
        with pytest.raises(B.ZeroError):
            B.zero_clip_workspace_bytes_ex(fs.ctx, 4)
        B.zero_clip_grad_norm_ex(fs.ctx, 1.0, B.ZERO_CLIP_KEEP_REDUCED, ws.data_ptr(), big, fs.stream_handle())
        fs.step()
        assert B.zero_last_launches(fs.ctx) == 1
        fs.post_step()
    finally:
        fs.close()


def test_registration_after_clip_is_refused():
    pb = make_problem(si.toy_mlp(), 4, 2, steps=1, seed=50, max_norm=0.5)
    fs = gpu_flatstep(pb)
    try:
        flats = upload_grads(pb, 1)
        register(fs, pb, flats, "units", [])
        fs.clip_grad_norm(0.5)
        with pytest.raises(B.ZeroError) as e:
            fs.reduce_grads(-1, flats)
        assert e.value.status == B.ZERO_ESTATE and "clip" in B.zero_last_error(fs.ctx)
        fs.step()   # the pending clip and the earlier registration still stand
        fs.post_step()
        register(fs, pb, flats, "all", [])   # allowed again after post_step
        fs.step()
        fs.post_step()
    finally:
        fs.close()


def _same_norm(a, b):
    if np.isnan(b):
        return np.isnan(a)
    if np.isinf(b):
        return a == b
    return abs(a - b) <= 1e-12 * abs(b)


@pytest.mark.parametrize("gd,keep", [("bf16", False), ("bf16", True), ("fp32", False)])
def test_non_finite_gradients(gd, keep):
    # step 1: an inf gradient (norm inf: every gradient scaled by 0, inf * 0 = NaN);
    # step 2: the largest finite values in both replicas at one position, whose
    #         fp32 sum overflows (the reduced gradient is inf);
    # step 3: finite again;
    # step 4: a NaN in an element-wise tail (norm NaN: coefficient NaN, every
    #         gradient NaN, every state element NaN).
    # Norms and every state element follow the oracle.
    pl = si.from_units([3000, 77, 5001])
    pb = make_problem(pl, 2, 2, grad_dtype=gd, steps=4, seed=90, max_norm=0.5)
    lay = pb.lay
    tail = int(lay.unit_base[1] + 76)  # last element of the 77-element unit
    if gd == "bf16":
        inf, nan, top = np.uint16(0x7F80), np.uint16(0x7FC0), np.uint16(0x7F7F)
    else:
        inf, nan, top = np.float32(np.inf), np.float32(np.nan), np.float32(3.0e38)
    pb.grads[0][0][1234] = inf
    pb.grads[1][0][4321] = top
    pb.grads[1][1][4321] = top
    pb.grads[3][1][tail] = nan
    ref_states, ref_norms, gpu_norms = {}, [], []
    oracle_run(pb, every_step=lambda t, s: ref_states.__setitem__(t, s), norms=ref_norms)
    assert ref_norms[0] == np.inf and ref_norms[1] == np.inf and np.isfinite(ref_norms[2]) and np.isnan(ref_norms[3])
    assert np.isnan(ref_states[4][0]).all() and not np.isnan(ref_states[3][0][:100]).any()

    def check(t, fs):
        compare_state(fs, ref_states[t], f"non-finite step {t}")
    fs = run_gpu(pb, mode="units", every_step=check, norms=gpu_norms, clip_keep=keep)
    fs.close()
    for a, b in zip(gpu_norms, ref_norms):
        assert _same_norm(a, b), (a, b)


def _scale_grads(pb, scale, lo=None, hi=None):
    """Multiplies replica gradients [lo, hi) of every step by `scale` (host
    arrays; bf16 patterns are rescaled through fp32 and rounded back)."""
    for reps in pb.grads:
        for k, flat in enumerate(reps):
            sl = slice(lo, hi)
            if pb.grad_dtype == "bf16":
                f = torch.from_numpy(flat[sl].view(np.int16)).view(torch.bfloat16).float() * scale
                flat[sl] = f.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
            else:
                flat[sl] = (flat[sl].astype(np.float64) * scale).astype(np.float32)


@pytest.mark.parametrize("gd,scale", [("fp32", 1e-28), ("bf16", 1e-18), ("fp32", 1e-40), ("bf16", 0.0)])
def test_norm_of_tiny_and_zero_gradients(gd, scale):
    # Sums of squares below 2^-60 (and all-zero gradients) take the kernel's
    # exact fp64 path: gradients ~1e-30 (squares underflow fp32), ~1e-20
    # (squares are fp32 denormals), fp32 denormal gradients and zeros.  The
    # layout spans several chunks and a ragged tail; norms follow the oracle
    # to 1e-12 (0 exactly for zeros) and every state element bit for bit.
    pl = si.from_units([16384 * 2 + 5, 1552, 9])
    pb = make_problem(pl, 3, 2, grad_dtype=gd, steps=2, seed=91, max_norm=0.5)
    _scale_grads(pb, scale)
    norms = _clip_parity(pb, mode="units")
    if scale == 0.0:
        assert norms == [0.0, 0.0]
    else:
        assert all(0.0 < x < 2.0 ** -30 for x in norms)


@pytest.mark.parametrize("gd", ["fp32", "bf16"])
def test_norm_with_tiny_and_normal_elements_mixed(gd):
    # Chunk 0: every thread's first group tiny, the rest normal (the fast
    # path, where the tiny squares' product errors may be lost: far below the
    # tolerance); chunk 1 entirely tiny (the exact path for all its threads);
    # the rest normal.  Norms follow the oracle and the stages agree bit for bit.
    pl = si.from_units([16384 * 3 + 77])
    out = {}
    for stage in (0, 2, 3):
        pb = make_problem(pl, 2, stage, grad_dtype=gd, steps=2, seed=92, max_norm=0.5)
        _scale_grads(pb, 1e-25, 0, 2048)
        _scale_grads(pb, 1e-25, 16384, 2 * 16384)
        _clip_parity(pb, mode="units")
        norms = []
        fs = run_gpu(pb, mode="separate", norms=norms)
        out[stage] = (norms, to_np(fs.master)[:pl.total].copy())
        fs.close()
    for stage in (2, 3):
        assert out[stage][0] == out[0][0]
        assert np.array_equal(out[stage][1].view(np.uint32), out[0][1].view(np.uint32))


@pytest.mark.parametrize("n,gd", [(1, "bf16"), (3, "bf16"), (6, "bf16"), (8, "bf16"), (16, "bf16"), (2, "fp32"),
                                  (5, "fp32"), (9, "fp32")])
def test_norm_of_unaligned_gradients(n, gd):
    # Every unit's gradients placed 0..7 (bf16) or 0..3 (fp32) elements past a
    # 16-byte boundary, differently per replica: the norm pass reads whole
    # groups through shifted aligned words.  The norm must equal the one from
    # 16-byte-aligned buffers bit for bit (same order) and the oracle's to
    # 1e-12; the clipped state follows the oracle bit for bit.  Units span
    # several chunks, a ragged last chunk and one shorter than a group.
    from test_gpu_shifted import _register_offsets
    pl = si.from_units([16384 * 3 + 77, 1552, 5, 40_003])
    pb = make_problem(pl, n, 2, grad_dtype=gd, steps=2, seed=700 + n, max_norm=0.05)
    k = 8 if gd == "bf16" else 4
    offsets = [[(3 * r + u + 1) % k for u in range(k)] for r in range(n)]
    ref_states, ref_norms = {}, []
    oracle_run(pb, every_step=lambda t, s: ref_states.__setitem__(t, s), norms=ref_norms)
    norms = {}
    for mode in ("aligned", "shifted"):
        fs = gpu_flatstep(pb)
        try:
            got = []
            for t in (1, 2):
                keep = []
                flats = upload_grads(pb, t)
                if mode == "aligned":
                    register(fs, pb, flats, "separate", keep)
                else:
                    _register_offsets(fs, flats, offsets, keep)
                fs.clip_grad_norm(pb.max_norm)
                got.append(fs.grad_norm())
                fs.step()
                fs.post_step()
                torch.cuda.synchronize()
                compare_state(fs, ref_states[t], f"{mode} step {t}")
            norms[mode] = got
        finally:
            fs.close()
    assert norms["shifted"] == norms["aligned"]
    for a, b in zip(norms["shifted"], ref_norms):
        assert abs(a - b) <= 1e-12 * b, (a, b)
