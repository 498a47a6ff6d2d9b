"""Run as a child process by tests/test_host_alloc_failure.py (not collected
by pytest): the address space is limited so that the library's host
allocations for a large layout fail; zero_plan must report ZERO_ENOMEM, hand
back no context, and work again once the limit is lifted.  No CUDA call is
made.  Prints one line: "<status under the limit> <context under the limit>
<status after> <layout elements after>"."""

import ctypes
import os
import resource
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(HERE))

from zero_sharded_mixed_flatparameter_gb300 import binding as B  # noqa: E402


def vm_bytes() -> int:
    with open("/proc/self/status") as f:
        for line in f:
            if line.startswith("VmSize:"):
                return int(line.split()[1]) * 1024
    raise RuntimeError("no VmSize")


def main() -> int:
    lib = B.load()
    n = 4_000_000  # one parameter per unit: ~5 tables of 4 M 64-bit entries (~160 MB)
    numel = np.ones(n, dtype=np.int64)
    unit = np.arange(n, dtype=np.int32)
    cfg = B.make_config(2, 4)
    p64 = numel.ctypes.data_as(ctypes.POINTER(ctypes.c_int64))
    p32 = unit.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))
    soft, hard = resource.getrlimit(resource.RLIMIT_AS)
    resource.setrlimit(resource.RLIMIT_AS, (vm_bytes() + (48 << 20), hard))
    out = ctypes.c_void_p()
    st_limited = lib.zero_plan(ctypes.byref(cfg), p64, p32, n, ctypes.byref(out))
    ctx_limited = out.value or 0
    resource.setrlimit(resource.RLIMIT_AS, (soft, hard))
    out2 = ctypes.c_void_p()
    st_after = lib.zero_plan(ctypes.byref(cfg), p64, p32, n, ctypes.byref(out2))
    elems = B.zero_padded_numel(out2.value)[0] if st_after == 0 else -1
    if out2.value:
        lib.zero_destroy(out2)
    print(st_limited, ctx_limited, st_after, elems, flush=True)
    return 0


if __name__ == "__main__":
    sys.exit(main())
