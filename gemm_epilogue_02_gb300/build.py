"""Build step for the CUDA library: one nvcc invocation, sm_103a only, in-tree.

Produces gemm_epilogue_02_gb300/libtgemm.so (git-ignored) from csrc/tgemm_api.cu.
The CUDA runtime is linked statically and the driver's tensor-map encoder is
looked up at run time, so the library loads (for symbol checks) on a host
without a GPU driver.
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
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def command(out: str, extra=()) -> list:
    return [nvcc(), *ARCH, "-lineinfo", "-O3", "-std=c++17", "--expt-relaxed-constexpr",
            "-Xcompiler", "-fPIC", "-shared", "-cudart", "static", *extra, "-o", out, SRC]


def stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    return any(os.path.getmtime(p) > t for p in [SRC, *DEPS])


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile libtgemm.so if missing or older than its sources; return its path."""
    if not force and not stale():
        return LIB
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = command(tmp, ["-Xptxas", "-v"] if verbose else [])
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("nvcc failed:\n" + " ".join(cmd) + "\n" + r.stdout + r.stderr)
    if verbose:
        print(r.stdout + r.stderr)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    import sys
    print(build(force=True, verbose="-v" in sys.argv))
