"""The index-checking debug build (compute-sanitizer is not available here):
every kernel index is checked before the access it guards, a failed check is
counted instead of trapping.  The parity scenarios of
tests/debug_checks_scenarios.py run against that build in a subprocess and
must match the oracle with no failed check; a positive control then tells the
kernels that the arrays end 8 elements early (they do not, so no access can
leave them) and the checks must refuse exactly those elements."""

import os
import subprocess
import sys

import pytest

from gpu_common import ensure_built
from zero_sharded_mixed_flatparameter_gb300 import binding as B

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))


def test_release_build_has_no_checks():
    ensure_built()
    with pytest.raises(B.ZeroError) as e:
        B.zero_debug_check_failures()
    assert e.value.status == B.ZERO_ENOTSUP


def test_debug_build_scenarios_pass_every_check():
    r = subprocess.run([sys.executable, os.path.join(HERE, "debug_checks_scenarios.py")], capture_output=True,
                       text=True, timeout=900)
    assert r.returncode == 0, r.stdout[-4000:] + r.stderr[-4000:]
    assert "debug check failures: 0" in r.stdout
    assert r.stdout.strip().splitlines()[-1].endswith("ok"), r.stdout[-2000:]
