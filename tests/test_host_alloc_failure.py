"""Host allocation failure inside the library (an injected host fault, no
GPU): the library allocates no device memory, so the failure is
made on its host metadata — a child process limits its address space
(RLIMIT_AS) just before zero_plan builds the tables of a 4 M-unit layout.
The call must return ZERO_ENOMEM and no context, and the same call must
succeed once the limit is lifted."""

import os
import subprocess
import sys

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.mark.skipif(not sys.platform.startswith("linux"), reason="RLIMIT_AS and /proc are Linux-only")
def test_zero_plan_reports_enomem_and_recovers():
    from zero_sharded_mixed_flatparameter_gb300 import binding as B
    B.load()  # built (and loadable) before the child runs
    r = subprocess.run([sys.executable, os.path.join(HERE, "host_alloc_failure_scenario.py")],
                       capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    st_limited, ctx_limited, st_after, elems = (int(x) for x in r.stdout.split())
    assert st_limited == B.ZERO_ENOMEM
    assert ctx_limited == 0
    assert st_after == B.ZERO_OK
    assert elems == 4 * 4_000_000  # each one-element unit padded to N = 4
