"""Thin ctypes binding of the C ABI in include/tgemm.h.

Argument marshalling only: every step of the computation runs in the CUDA
library.  There is no CPU fallback; if the library cannot be loaded, every
call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

TGEMM_F16, TGEMM_BF16 = 0, 1
TGEMM_EPI_NONE, TGEMM_EPI_RELU, TGEMM_EPI_BIAS, TGEMM_EPI_BIAS_RELU = 0, 1, 2, 3
TGEMM_EPI_GELU, TGEMM_EPI_BIAS_GELU = 4, 5
STATUS = {0: "TGEMM_OK", 1: "TGEMM_ERR_INVALID_ARG", 2: "TGEMM_ERR_ALIGNMENT",
          3: "TGEMM_ERR_UNSUPPORTED_DEVICE", 4: "TGEMM_ERR_ALIAS", 5: "TGEMM_ERR_CUDA",
          6: "TGEMM_ERR_TIMEOUT", 7: "TGEMM_ERR_SCRATCH_LIMIT", 8: "TGEMM_ERR_DEBUG_CHECK"}
EXPORTED = ("tgemm_run", "tgemm_run_ex", "tgemm_run_host", "tgemm_status_string",
            "tgemm_last_device_status", "tgemm_version", "tgemm_run_noalloc", "tgemm_plan",
            "tgemm_attention_fwd", "tgemm_debug_last_check")
PLAN_FIELDS = ("bn", "cg", "stages", "tiles", "groups", "split_k", "split_first", "narrow_first",
               "narrow_parts", "units")
NOALLOC_SCRATCH_BYTES = 64 << 20

_lock = threading.Lock()
_lib = None
_debug_lib = None


class TgemmError(RuntimeError):
    def __init__(self, status: int, where: str = "tgemm_run"):
        self.status = int(status)
        super().__init__(f"{where}: {STATUS.get(self.status, self.status)}")


def library_path() -> str:
    """The library load() uses: the debug build when TGEMM_DEBUG=1 is set."""
    return _build.DEBUG_LIB if os.environ.get("TGEMM_DEBUG") == "1" else _build.LIB


def _configure(lib: ctypes.CDLL) -> ctypes.CDLL:
    p, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
    for name in ("tgemm_run", "tgemm_run_host", "tgemm_run_noalloc"):
        f = getattr(lib, name)
        f.argtypes = [p, p, p, p, i64, i64, i64, i64, i64, i64, i32, i32, p]
        f.restype = i32
    lib.tgemm_run_ex.argtypes = [p, p, p, p, i64, i64, i64, i64, i64, i64, i32, i32, i32, i32, p]
    lib.tgemm_run_ex.restype = i32
    lib.tgemm_status_string.argtypes = [i32]
    lib.tgemm_status_string.restype = ctypes.c_char_p
    lib.tgemm_last_device_status.argtypes = []
    lib.tgemm_last_device_status.restype = i32
    lib.tgemm_debug_last_check.argtypes = []
    lib.tgemm_debug_last_check.restype = i32
    lib.tgemm_version.argtypes = []
    lib.tgemm_version.restype = i32
    lib.tgemm_plan.argtypes = [i64, i64, i64, i32, p]
    lib.tgemm_plan.restype = i32
    lib.tgemm_attention_fwd.argtypes = [p, p, p, p, i64, i64, i64, i64, i32, i32, p]
    lib.tgemm_attention_fwd.restype = i32
    return lib


def load(build_if_missing: bool = True) -> ctypes.CDLL:
    """Load libtgemm.so, or libtgemm_debug.so when TGEMM_DEBUG=1 is set at the
    first call (building them with nvcc if missing or stale)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if build_if_missing:
            _build.build()
        path = library_path()
        if not os.path.exists(path):
            raise RuntimeError(f"CUDA library {path} is missing; run build() first")
        _lib = _configure(ctypes.CDLL(path))
        return _lib


def load_debug(build_if_missing: bool = True) -> ctypes.CDLL:
    """The debug build, loaded beside the library load() returns (its own
    device state); for tests that run both on the same inputs."""
    global _debug_lib
    with _lock:
        if _debug_lib is None:
            if build_if_missing:
                _build.build()
            if not os.path.exists(_build.DEBUG_LIB):
                raise RuntimeError(f"CUDA library {_build.DEBUG_LIB} is missing; run build() first")
            _debug_lib = _configure(ctypes.CDLL(_build.DEBUG_LIB))
        return _debug_lib


def tgemm_run(A: int, B: int, bias: int, C: int, M: int, N: int, K: int, lda: int, ldb: int,
              ldc: int, dtype: int, epilogue: int, stream: int = 0) -> int:
    """Raw C-ABI call with device pointers (ints); returns the status code."""
    lib = _lib if _lib is not None else load()
    return lib.tgemm_run(A or None, B or None, bias or None, C or None, M, N, K, lda, ldb, ldc,
                         dtype, epilogue, stream or None)


def tgemm_run_ex(A: int, B: int, bias: int, C: int, M: int, N: int, K: int, lda: int, ldb: int,
                 ldc: int, dtype: int, epilogue: int, transpose_a: int, transpose_b: int,
                 stream: int = 0) -> int:
    """Raw C-ABI call with either operand stored transposed; returns the status code."""
    return load().tgemm_run_ex(A or None, B or None, bias or None, C or None, M, N, K, lda, ldb, ldc,
                               dtype, epilogue, int(transpose_a), int(transpose_b), stream or None)


def tgemm_run_host(A: int, B: int, bias: int, C: int, M: int, N: int, K: int, lda: int, ldb: int,
                   ldc: int, dtype: int, epilogue: int, stream: int = 0) -> int:
    """Raw C-ABI call with host pointers (ints); returns the status code."""
    return load().tgemm_run_host(A or None, B or None, bias or None, C or None, M, N, K, lda, ldb,
                                 ldc, dtype, epilogue, stream or None)


def tgemm_run_noalloc(A: int, B: int, bias: int, C: int, M: int, N: int, K: int, lda: int,
                      ldb: int, ldc: int, dtype: int, epilogue: int, stream: int = 0) -> int:
    """Raw C-ABI call of the allocation-free variant (device pointers as ints).

    For callers that must not allocate GPU memory (memory reserved up front by
    another allocator, allocation-free latency loops): any operand repack uses
    the library's fixed 64 MiB device array instead of allocating; calls that
    may overlap on the GPU race on that array.  Returns the status code."""
    return load().tgemm_run_noalloc(A or None, B or None, bias or None, C or None, M, N, K, lda,
                                    ldb, ldc, dtype, epilogue, stream or None)


def tgemm_status_string(status: int) -> str:
    return load().tgemm_status_string(int(status)).decode()


def tgemm_last_device_status() -> int:
    return int(load().tgemm_last_device_status())


def tgemm_debug_last_check() -> int:
    """Id of the first failed device-side check of the debug build since the
    last call (0: none; -1: the loaded library is the release build)."""
    return int(load().tgemm_debug_last_check())


def tgemm_version() -> int:
    return int(load().tgemm_version())


def tgemm_plan(M: int, N: int, K: int, num_sms: int) -> dict:
    """The work plan of an M x N x K problem on `num_sms` SMs (host logic, no GPU)."""
    out = (ctypes.c_int32 * len(PLAN_FIELDS))()
    st = load().tgemm_plan(M, N, K, num_sms, ctypes.cast(out, ctypes.c_void_p))
    if st != 0:
        raise TgemmError(st, "tgemm_plan")
    return dict(zip(PLAN_FIELDS, (int(v) for v in out)))


def tgemm_attention_fwd(Q: int, K: int, V: int, O: int, batch: int, seq: int, heads: int, dim: int,
                        causal: int, dtype: int, stream: int = 0) -> int:
    return int(load().tgemm_attention_fwd(Q, K, V, O, batch, seq, heads, dim, int(causal), dtype, stream))
