"""Full-size GPU runs checked on sampled windows against the oracle.

The step is elementwise (CMU 15-779 Lecture 13 notes §3.1: element j's update
uses only gradient j, m_j and v_j), so the oracle can update any window of
the flat buffer on its own.  Inputs are drawn on the device with seeded
generators; the oracle gets the windows' bytes copied back before each step
(its initial master window is rebuilt from the init parameters and its own
layout, not read from the GPU's master).  Windows: the first and last
elements, both sides of every unit boundary, and seeded random positions at
arbitrary (unaligned) offsets.
"""

from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import synth_inputs as si
from gpu_common import assert_bf16_1ulp, assert_bit_exact, assert_rel_close, ensure_built, to_np
from zero_sharded_mixed_flatparameter_gb300.runner import FlatStep

pytestmark = pytest.mark.gpu

W = 256  # elements per window


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()
    yield
    torch.cuda.empty_cache()


def _windows(total, unit_bases, seed, n_random=64):
    rng = np.random.default_rng(seed)
    starts = {0, max(total - W, 0)}
    for b in unit_bases:
        starts.add(int(min(max(b - W // 2, 0), max(total - W, 0))))
    for s in rng.integers(0, max(total - W, 1), n_random):
        starts.add(int(s))
    return sorted(starts)


def _master_window(init_flat_host_fn, lay, pl, a, b):
    """Initial fp32 master on [a, b) from the init params and the oracle layout."""
    out = np.zeros(b - a, np.float32)
    offs = lay.param_offset
    cum = np.concatenate([[0], np.cumsum(pl.numel)])
    p_lo = max(int(np.searchsorted(offs, a, side="right")) - 1, 0)
    for p in range(p_lo, len(pl.numel)):
        o, k = int(offs[p]), pl.numel[p]
        if o >= b:
            break
        lo, hi = max(a, o), min(b, o + k)
        if lo < hi:
            out[lo - a:hi - a] = init_flat_host_fn(int(cum[p]) + lo - o, int(cum[p]) + hi - o)
    return out


def run_full(pl, n, stage, grad_dtype, steps, seed, grad_std, outlier_fraction=0.0, gather=False,
             register_units=True, offload=False):
    lay = oracle.layout(pl.numel, pl.unit, n, stage)
    total = lay.total_padded
    # init params: one flat fp32 draw of all parameters, per-param views
    init_flat = si.normal_fp32(pl.total, 0.02, seed, device="cuda")
    cum = np.concatenate([[0], np.cumsum(pl.numel)])
    init = [init_flat[int(cum[p]):int(cum[p + 1])] for p in range(len(pl.numel))]
    fs = FlatStep(pl.numel, pl.unit, stage=stage, n_ranks=n, grad_dtype=grad_dtype, init_params=init,
                  offload=offload)
    try:
        assert (fs.padded, fs.n_units) == (total, len(lay.unit_numel))
        for i in range(fs.n_units):
            assert fs.layout(i) == (lay.unit_numel[i], lay.unit_padded[i], lay.unit_shard[i], lay.unit_base[i])
        starts = _windows(total, lay.unit_base, seed)
        init_host = lambda lo, hi: to_np(init_flat[lo:hi])
        win_master = {a: _master_window(init_host, lay, pl, a, a + W) for a in starts}
        torch.cuda.synchronize()
        for a in starts[:8]:  # make_master flattening, checked exactly on a few windows
            assert np.array_equal(to_np(fs.master[a:a + W]), win_master[a])
        del init, init_flat
        win_grads = {a: [] for a in starts}
        for t in range(1, steps + 1):
            grads = si.replica_grads(n, total, grad_std, seed * 131 + t, grad_dtype, device="cuda",
                                     outlier_fraction=outlier_fraction)
            # zero pads, as the ZeRO-2 hook's padding makes them
            for i in range(fs.n_units):
                lo, hi = int(lay.unit_base[i] + lay.unit_numel[i]), int(lay.unit_base[i] + lay.unit_padded[i])
                for g in grads:
                    g[lo:hi] = 0
            for a in starts:
                win_grads[a].append([to_np(g[a:a + W]) for g in grads])
            if register_units:
                for i in range(fs.n_units):
                    b, p = int(lay.unit_base[i]), int(lay.unit_padded[i])
                    fs.reduce_grads(i, [g[b:b + p] for g in grads])
            else:
                fs.reduce_grads(-1, grads)
            fs.step()
            if gather:
                for i in range(fs.n_units):
                    b, p = int(lay.unit_base[i]), int(lay.unit_padded[i])
                    unit_buf = torch.empty(p, dtype=torch.bfloat16, device="cuda")
                    fs.gather_weights(i, unit_buf)
                    torch.cuda.synchronize()
                    assert torch.equal(unit_buf.view(torch.int16), fs.param16[b:b + p].view(torch.int16))
                    del unit_buf
                if t == steps:  # every unit in one call (the prefetch form)
                    bufs = [torch.empty(int(p), dtype=torch.bfloat16, device="cuda") for p in lay.unit_padded]
                    fs.gather_units(0, bufs)
                    assert fs.last_launches() == 1
                    torch.cuda.synchronize()
                    for i, buf in enumerate(bufs):
                        b, p = int(lay.unit_base[i]), int(lay.unit_padded[i])
                        assert torch.equal(buf.view(torch.int16), fs.param16[b:b + p].view(torch.int16)), i
                    del bufs
            fs.post_step()
            torch.cuda.synchronize()
            del grads
        hyper = oracle.Hyper(n_ranks=n, grad_dtype=grad_dtype)
        for a in starts:
            master = win_master[a].copy()
            m = np.zeros(W, np.float32)
            v = np.zeros(W, np.float32)
            p16 = np.zeros(W, np.uint16)
            for t in range(1, steps + 1):
                oracle.step_window(hyper, t, win_grads[a][t - 1], master, m, v, p16)
            got = (to_np(fs.master[a:a + W]), to_np(fs.exp_avg[a:a + W]), to_np(fs.exp_avg_sq[a:a + W]),
                   to_np(fs.param16[a:a + W]))
            what = f"window@{a}"
            for name, g, w in zip(("master", "m", "v"), got[:3], (master, m, v)):
                assert_rel_close(g, w, f"{what} {name}")
            assert_bf16_1ulp(got[3], p16, f"{what} param16")
            for name, g, w in zip(("master", "m", "v", "param16"), got, (master, m, v, p16)):
                assert_bit_exact(g, w, f"{what} {name}")
        return fs.step_count()
    finally:
        fs.close()
        torch.cuda.empty_cache()


def test_llama_1024_zero2_n8():
    # 73,417,728 params in one FlatParameter, N = 8, ZeRO-2, bf16 grads N(0, 1e-3), 10 steps
    assert run_full(si.llama_1024(), 8, 2, "bf16", 10, seed=2, grad_std=1e-3, register_units=False) == 10


def test_llama_1024_zero2_n8_offload():
    # the same workload as a ZeRO-Offload context (host fp32 state, 8 M-element chunks), 3 steps
    assert run_full(si.llama_1024(), 8, 2, "bf16", 3, seed=12, grad_std=1e-3, register_units=False,
                    offload=True) == 3


def test_llama_2048_zero3_units_n8_gather():
    # 654,346,240 params, one unit per decoder layer + embedding / norm+head, N = 8,
    # ZeRO-3 with a per-unit gather into a bf16 unit buffer, 10 steps
    assert run_full(si.llama_2048_units(), 8, 3, "bf16", 10, seed=3, grad_std=1e-3, gather=True) == 10


def test_llama_2048_stage_buffer_zero1_fp32_n2():
    # 2,030,174,208 params (32 layers + embedding), N = 2, ZeRO-1, fp32 grads, 5 steps
    assert run_full(si.llama_2048_stage_buffer(), 2, 1, "fp32", 5, seed=4, grad_std=1e-3,
                    register_units=False) == 5


@pytest.mark.parametrize("numel,n", [(1_000_000_000, 16), (128_000_000, 1), (16_000_000, 4), (1_000_000, 8),
                                     (512_000_000, 2)])
def test_flat_sweep_points(numel, n):
    # single flat fp32 buffer, bf16 grads N(0, 1e-2) with 0.1% entries set to +-1, one step
    assert run_full(si.single_buffer(numel), n, 2, "bf16", 1, seed=5, grad_std=1e-2, outlier_fraction=0.001,
                    register_units=False) == 1


def test_beyond_2_pow_31_elements():
    # 2^31 + 4,105 elements in one unit: every index and pointer offset must be
    # 64-bit (windows straddle 2^31 and the end), with the clip on as well
    numel = 2 ** 31 + 4105
    pl = si.single_buffer(numel)
    n = 1
    lay = oracle.layout(pl.numel, pl.unit, n, 1)
    init_flat = si.normal_fp32(numel, 0.02, 61, device="cuda")
    fs = FlatStep(pl.numel, pl.unit, stage=1, n_ranks=n, init_params=[init_flat])
    starts = [0, 2 ** 31 - W // 2, 2 ** 31 + 1000, numel - W]
    win = {a: [to_np(init_flat[a:a + W]), np.zeros(W, np.float32), np.zeros(W, np.float32),
               np.zeros(W, np.uint16)] for a in starts}
    del init_flat
    h = oracle.Hyper(n_ranks=n)
    try:
        for t in (1, 2):
            grads = si.replica_grads(n, numel, 1e-3, 62 + t, "bf16", device="cuda")
            fs.reduce_grads(-1, grads)
            ws = torch.empty(B_ws_bytes(fs), dtype=torch.uint8, device="cuda")
            from zero_sharded_mixed_flatparameter_gb300 import binding as B
            B.zero_clip_grad_norm(fs.ctx, 1e6, ws.data_ptr(), ws.numel(), fs.stream_handle())  # inactive clip
            fs.step()
            fs.post_step()
            for a in starts:
                oracle.step_window(h, t, [to_np(grads[0][a:a + W])], *win[a])
            del grads, ws
        torch.cuda.synchronize()
        for a in starts:
            got = (to_np(fs.master[a:a + W]), to_np(fs.exp_avg[a:a + W]), to_np(fs.exp_avg_sq[a:a + W]),
                   to_np(fs.param16[a:a + W]))
            for name, g, w in zip(("master", "m", "v", "param16"), got, win[a]):
                assert_bit_exact(g, w, f"window@{a} {name}")
        assert lay.total_padded == numel
    finally:
        fs.close()
        torch.cuda.empty_cache()


def B_ws_bytes(fs):
    from zero_sharded_mixed_flatparameter_gb300 import binding as B
    return B.zero_clip_workspace_bytes(fs.ctx)
