"""Build of the CUDA library (``libzero_flatstep.so``) for sm_103a.

The CUDA and runtime translation units are compiled in parallel with nvcc,
the host CPU-Adam unit with the host C++ compiler (portable flags only, so it
builds the same on x86-64 and aarch64), then all are linked into a shared
library next to this file's package (in-tree, git-ignored).  No fast-math
and no FMA contraction anywhere: the step's arithmetic is reproducible bit
for bit, on the device and on the host.
"""

from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB_NAME = "libzero_flatstep.so"
LIB_PATH = os.path.join(PKG, LIB_NAME)
# The same sources with every kernel index checked (-DZFS_DEBUG_CHECKS): a
# failed check is counted (zero_debug_check_failures) and its access skipped.
DEBUG_LIB_PATH = os.path.join(PKG, "libzero_flatstep_debug.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
COMMON = ["-std=c++17", "-O3", "-lineinfo", "--fmad=false", "-Xcompiler", "-fPIC,-O2",
          "-I" + INCLUDE, "-I" + CSRC]
SOURCES = ["zero_step_kernels.cu", "zero_aux_kernels.cu", "zero_runtime.cpp", "zero_no_alloc.cu"]
HOST_SOURCES = ["zero_host_adam.cpp"]
HOST_FLAGS = ["-std=c++17", "-O3", "-ffp-contract=off", "-fno-math-errno", "-fPIC", "-pthread", "-I" + CSRC]


def _nvcc() -> str:
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build the library")
    return nvcc


def _cxx() -> str:
    cxx = os.environ.get("CXX") or shutil.which("g++") or shutil.which("c++")
    if not cxx:
        raise RuntimeError("no host C++ compiler (g++) found")
    return cxx


def _inputs():
    files = [os.path.join(CSRC, s) for s in SOURCES + HOST_SOURCES]
    files += [os.path.join(CSRC, "zero_internal.h"), os.path.join(CSRC, "zero_device.cuh"),
              os.path.join(CSRC, "zero_aux_internal.h"), os.path.join(CSRC, "zero_host.h"),
              os.path.join(INCLUDE, "zero_flatstep.h")]
    return files


def up_to_date(path: str = LIB_PATH) -> bool:
    if not os.path.exists(path):
        return False
    t = os.path.getmtime(path)
    return all(os.path.getmtime(f) <= t for f in _inputs())


def build(force: bool = False, verbose: bool = False, extra_flags=(), debug_checks: bool = False) -> str:
    """Build the library (or, with debug_checks, its index-checking variant)."""
    out_path = DEBUG_LIB_PATH if debug_checks else LIB_PATH
    build_dir = os.path.join(BUILD, "debug") if debug_checks else BUILD
    if debug_checks:
        extra_flags = (*extra_flags, "-DZFS_DEBUG_CHECKS")
    if not force and up_to_date(out_path):
        return out_path
    os.makedirs(build_dir, exist_ok=True)
    nvcc = _nvcc()

    cxx = _cxx()

    def compile_one(src):
        obj = os.path.join(build_dir, os.path.splitext(src)[0] + ".o")
        if src in HOST_SOURCES:
            cmd = [cxx, *HOST_FLAGS, *[f for f in extra_flags if f.startswith("-D")], "-c",
                   os.path.join(CSRC, src), "-o", obj]
        else:
            cmd = [nvcc, *ARCH, *COMMON, *extra_flags, "-c", os.path.join(CSRC, src), "-o", obj]
        if verbose:
            print(" ".join(cmd), flush=True)
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"compiling {src} failed:\n{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            print(r.stdout + r.stderr, flush=True)
        return obj

    with cf.ThreadPoolExecutor(max_workers=len(SOURCES) + len(HOST_SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES + HOST_SOURCES))
    tmp = out_path + f".tmp{os.getpid()}"
    cmd = [nvcc, *ARCH, "-shared", "-o", tmp, *objs, "-cudart", "static", "-lpthread"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, out_path)
    return out_path


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose=True))
