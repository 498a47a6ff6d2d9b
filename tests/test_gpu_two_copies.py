"""Two copies of the library in one process (say a release and a debug
build, or two packages that each ship it): each copy must raise the dynamic
shared memory limit of its own staged kernels.  A record of that kept in a
function-local static of a launch template would be one object for the whole
process, and the second copy's staged launches would then fail.

Run in a subprocess, so that this test process keeps its own library."""

import os
import shutil
import subprocess
import sys

import pytest

from gpu_common import ensure_built
from zero_sharded_mixed_flatparameter_gb300 import binding as B

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))

SCRIPT = r"""
import sys
sys.path.insert(0, {root!r}); sys.path.insert(0, {tests!r})
import numpy as np, torch
import synth_inputs as si
from gpu_common import compare_state, make_problem, oracle_run, run_gpu, to_np
from zero_sharded_mixed_flatparameter_gb300 import binding as B
import oracle
oracle.build()
states = []
# bf16 N = 2 (4-element staged kernel) and N = 16 (2,048-element staged
# kernel), fp32 N = 12: launches of more than 2^23 elements
cases = [(2, "bf16"), (16, "bf16"), (12, "fp32")]
for path in ({first!r}, {second!r}):
    B._lib = None
    B.load(path)
    for n, gd in cases:
        pb = make_problem(si.from_units([(1 << 23) + 4099]), n, 2, grad_dtype=gd, steps=1, seed=600 + n)
        fs = run_gpu(pb, mode="all")
        states.append(tuple(to_np(x).copy() for x in (fs.master, fs.exp_avg, fs.exp_avg_sq, fs.param16)))
        if path == {first!r}:
            compare_state(fs, oracle_run(pb), f"first copy, N = {{n}} {{gd}}")
        fs.close()
k = len(cases)
for i in range(k):
    for a, b in zip(states[i], states[k + i]):
        assert np.array_equal(a.view(np.uint8), b.view(np.uint8)), f"case {{i}}: the copies differ"
print("two copies ok")
"""


def test_two_copies_raise_their_own_shared_memory_limits(tmp_path):
    ensure_built()
    copy = str(tmp_path / "libzero_flatstep_copy.so")
    shutil.copy(B.LIB_PATH, copy)
    script = SCRIPT.format(root=os.path.dirname(HERE), tests=HERE, first=B.LIB_PATH, second=copy)
    r = subprocess.run([sys.executable, "-c", script], capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-3000:]
    assert "two copies ok" in r.stdout
