"""Seeded random parity cases: layouts, rank counts, gradient dtypes, stages,
registration modes, AdamW, clipping (with and without the kept reduced
gradient) and the offloaded step drawn together, each run for a few steps
and compared with the oracle after every step, bit for bit."""

import numpy as np
import pytest
import torch

import synth_inputs as si
from gpu_common import compare_state, ensure_built, make_problem, oracle_run, run_gpu

pytestmark = pytest.mark.gpu

N_CASES = 64


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()
    yield
    torch.cuda.empty_cache()


def _case(seed):
    rng = np.random.default_rng(1000 + seed)
    n_units = int(rng.integers(1, 7))
    sizes = []
    for _ in range(n_units):
        kind = rng.random()
        if kind < 0.25:
            sizes.append(int(rng.integers(1, 20)))          # tiny units: all tail
        elif kind < 0.8:
            sizes.append(int(rng.integers(20, 20_000)))
        else:
            sizes.append(int(rng.integers(20_000, 120_000)))
    n = int(rng.integers(1, 17))
    grad_dtype = "fp32" if rng.random() < 0.3 else "bf16"
    stage = int(rng.integers(0, 4))
    mode = ["all", "units", "separate"][int(rng.integers(0, 3))]
    adamw = bool(rng.random() < 0.4)
    clip = rng.random()
    max_norm = 0.0 if clip < 0.4 else float(rng.choice([0.01, 0.1, 10.0]))
    keep = bool(max_norm > 0 and rng.random() < 0.5)
    offload = None
    if rng.random() < 0.3 and not keep:
        offload = dict(chunk=int(rng.integers(1, 50_000)), threads=int(rng.integers(0, 5)))
    return dict(sizes=sizes, n=n, grad_dtype=grad_dtype, stage=stage, mode=mode, adamw=adamw,
                max_norm=max_norm, keep=keep, offload=offload)


@pytest.mark.parametrize("seed", range(N_CASES))
def test_random_case(seed):
    c = _case(seed)
    pb = make_problem(si.from_units(c["sizes"]), c["n"], c["stage"], grad_dtype=c["grad_dtype"], steps=3,
                      seed=300 + seed, adamw=c["adamw"], weight_decay=0.05 if c["adamw"] else 0.0,
                      max_norm=c["max_norm"])
    refs = {}
    oracle_run(pb, every_step=lambda t, s: refs.__setitem__(t, s))
    fs = run_gpu(pb, mode=c["mode"], clip_keep=c["keep"], offload=c["offload"],
                 every_step=lambda t, f: compare_state(f, refs[t], f"case {seed} {c} step {t}"))
    fs.close()
