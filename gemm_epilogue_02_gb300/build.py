"""Build step for the CUDA library: nvcc, sm_103a only, in-tree.

Produces gemm_epilogue_02_gb300/libtgemm.so (git-ignored) from
csrc/tgemm_api.cu, and its debug build libtgemm_debug.so (-DTGEMM_DEBUG: the
device-side bounds and alignment checks of csrc/debug_checks.cuh), the two
compiled in parallel.  The CUDA runtime is linked statically and the
driver's tensor-map encoder is looked up at run time, so the libraries load
(for symbol checks) on a host without a GPU driver.
"""
from __future__ import annotations

import glob
import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
SRC = os.path.join(HERE, "csrc", "tgemm_api.cu")
# Every header the translation unit includes: all of csrc/*.cuh and the C ABI.
DEPS = sorted(glob.glob(os.path.join(HERE, "csrc", "*.cuh"))) + [os.path.join(ROOT, "include", "tgemm.h")]
LIB = os.path.join(HERE, "libtgemm.so")
DEBUG_LIB = os.path.join(HERE, "libtgemm_debug.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def command(out: str, extra=()) -> list:
    return [nvcc(), *ARCH, "-lineinfo", "-O3", "-std=c++17", "--expt-relaxed-constexpr",
            "-Xcompiler", "-fPIC", "-shared", "-cudart", "static", *extra, "-o", out, SRC]


def stale(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    return any(os.path.getmtime(p) > t for p in [SRC, *DEPS])


def _start(lib: str, verbose: bool):
    tmp = lib + f".tmp{os.getpid()}"
    extra = (["-DTGEMM_DEBUG"] if lib == DEBUG_LIB else []) + (["-Xptxas", "-v"] if verbose else [])
    cmd = command(tmp, extra)
    return lib, tmp, cmd, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)


def build(force: bool = False, verbose: bool = False, debug: bool = True) -> str:
    """Compile libtgemm.so (and, with debug, libtgemm_debug.so) if missing or
    older than the sources, in parallel; return the release library's path."""
    libs = [LIB] + ([DEBUG_LIB] if debug else [])
    jobs = [_start(lib, verbose) for lib in libs if force or stale(lib)]
    errors = []
    for lib, tmp, cmd, proc in jobs:
        out, _ = proc.communicate()
        if proc.returncode != 0:
            errors.append("nvcc failed:\n" + " ".join(cmd) + "\n" + out)
            continue
        if verbose:
            print(out)
        os.replace(tmp, lib)
    if errors:
        raise RuntimeError("\n".join(errors))
    return LIB


if __name__ == "__main__":
    import sys
    print(build(force=True, verbose="-v" in sys.argv))
