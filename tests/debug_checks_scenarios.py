"""Parity scenarios run against the index-checking debug build of the library
(not collected by pytest: tests/test_gpu_debug_checks.py runs this file in a
subprocess so that the debug library is the one this process loads).

Every scenario must match the oracle, and the debug build must report that
no index check failed.  Exit status 0 on success."""

import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(HERE))
sys.path.insert(0, HERE)

from zero_sharded_mixed_flatparameter_gb300 import binding as B, build_lib  # noqa: E402

B.load(build_lib.build(debug_checks=True))

import synth_inputs as si  # noqa: E402
from gpu_common import compare_state, ensure_built, make_problem, oracle_run, run_gpu  # noqa: E402


def scenario(name, pb, mode="units", **kw):
    ref = oracle_run(pb)
    fs = run_gpu(pb, mode=mode, **kw)
    compare_state(fs, ref, name)
    fs.close()
    print("ok", name, flush=True)


def main():
    ensure_built()
    for stage in (0, 1, 2, 3):
        scenario(f"toy MLP stage {stage}", make_problem(si.toy_mlp(), 4, stage, steps=3, seed=200 + stage))
    odd = si.from_units([1552, 7, 9312, 33, 17])
    scenario("odd units N = 3 (padding, unaligned unit starts)", make_problem(odd, 3, 3, steps=2, seed=210))
    scenario("odd units N = 16 fp32", make_problem(odd, 16, 2, grad_dtype="fp32", steps=2, seed=211))
    scenario("odd units N = 3, one buffer per unit (shifted gradients)", make_problem(odd, 3, 3, steps=2, seed=222),
             mode="separate")
    scenario("odd units N = 5 fp32, one buffer per unit (shifted gradients)",
             make_problem(odd, 5, 2, grad_dtype="fp32", steps=2, seed=223), mode="separate")
    big = si.from_units([4_200_005, 1552, 2_500_000, 7, 2_000_000])
    scenario("tile-staged N = 16 bf16", make_problem(big, 16, 2, steps=1, seed=212), mode="separate")
    scenario("tile-staged N = 9 fp32", make_problem(big, 9, 3, grad_dtype="fp32", steps=1, seed=213), mode="all")
    scenario("tile-staged N = 12 fp32 (1,024-element tiles)",
             make_problem(big, 12, 2, grad_dtype="fp32", steps=1, seed=218), mode="separate")
    scenario("tile-staged N = 2 bf16 (4 elements per thread)", make_problem(big, 2, 3, steps=1, seed=219),
             mode="separate")
    scenario("tile-staged N = 4 bf16 (512-thread CTAs)", make_problem(big, 4, 2, steps=1, seed=220), mode="all")
    scenario("pipelined tile-staged N = 10 bf16", make_problem(big, 10, 3, steps=1, seed=224), mode="separate")
    scenario("shifted gradients over 2^23 elements, N = 3 bf16 (unaligned unit bases, one buffer per unit)",
             make_problem(big, 3, 2, steps=2, seed=226), mode="separate")
    scenario("clipped N = 8", make_problem(odd, 8, 2, steps=2, seed=214, max_norm=0.05))
    scenario("clipped, reduced gradient kept", make_problem(odd, 8, 1, steps=2, seed=215, max_norm=0.05),
             clip_keep=True)
    scenario("offload, 1,000-element chunks", make_problem(odd, 4, 2, steps=2, seed=216),
             offload=dict(chunk=1000, threads=3))
    # capturable mode: the kernels read the step count and bias corrections from the device
    import torch
    from gpu_common import gpu_flatstep, upload_grads
    pb = make_problem(odd, 8, 3, steps=3, seed=217, max_norm=0.05)
    ref = oracle_run(pb)
    fs = gpu_flatstep(pb)
    fs.enable_capturable(max_steps=8)
    for t in range(1, 4):
        fs.reduce_grads(-1, upload_grads(pb, t))
        fs.clip_grad_norm(pb.max_norm)
        fs.step()
        fs.post_step()
    torch.cuda.synchronize()
    compare_state(fs, ref, "capturable mode")
    fs.close()
    print("ok capturable mode", flush=True)
    failures = B.zero_debug_check_failures()
    print("debug check failures:", failures, flush=True)
    if failures != 0:
        return 1
    # Positive control: the kernels are told that the arrays end 8 elements
    # early (they do not, so nothing can leave them); the checks must refuse
    # exactly those 8 elements and let every other one match the oracle.
    import numpy as np
    import torch
    from gpu_common import gpu_flatstep, to_np, upload_grads
    pb = make_problem(si.toy_mlp(), 4, 2, steps=1, seed=221)
    fs = gpu_flatstep(pb)
    before = tuple(to_np(x).copy() for x in (fs.master, fs.exp_avg, fs.exp_avg_sq, fs.param16))
    fs.reduce_grads(-1, upload_grads(pb, 1))
    B.zero_debug_inject(fs.ctx, B.ZERO_INJECT_SHORT_BOUNDS)
    fs.step()
    torch.cuda.synchronize()
    refused = B.zero_debug_check_failures()
    ref = oracle_run(pb)
    got = tuple(to_np(x) for x in (fs.master, fs.exp_avg, fs.exp_avg_sq, fs.param16))
    tail = np.zeros(fs.padded, bool)
    tail[-8:] = True
    ok = refused >= 1 and all(np.array_equal(g[tail], b[tail]) and np.array_equal(g[~tail], r[~tail])
                              for g, b, r in zip(got, before, ref))
    fs.close()
    print("positive control: refused checks", refused, "ok" if ok else "FAILED", flush=True)
    return 0 if ok else 1


if __name__ == "__main__":
    sys.exit(main())
