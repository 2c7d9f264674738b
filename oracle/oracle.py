"""ctypes binding and build step for the C oracle (gemm_oracle.c).

TEST INFRASTRUCTURE ONLY (tests, smoke check, CPU-baseline benchmark leg).

Arrays are numpy uint16 bit patterns of fp16 or bf16 values, row-major with an
explicit leading dimension (the row pitch in elements), exactly as the GPU
library sees them.  Results are fp64 (unrounded) plus a separate
round-to-nearest-even step to the 16-bit output dtype.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

F16, BF16 = 0, 1
EPI_NONE, EPI_RELU, EPI_BIAS, EPI_BIAS_RELU, EPI_GELU, EPI_BIAS_GELU = 0, 1, 2, 3, 4, 5

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gemm_oracle.c")
_SRCS = [_SRC, os.path.join(_HERE, "attention_oracle.c")]
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def dtype_code(name) -> int:
    """Map 'fp16'/'f16'/'float16' or 'bf16'/'bfloat16' (or a torch dtype) to 0/1."""
    s = str(name).replace("torch.", "").lower()
    if s in ("fp16", "f16", "float16", "half"):
        return F16
    if s in ("bf16", "bfloat16"):
        return BF16
    raise ValueError(f"unsupported dtype {name!r}")


def build(force: bool = False) -> str:
    """Compile liboracle.so with gcc (OpenMP if the compiler supports it)."""
    if not force and os.path.exists(_LIB) and all(os.path.getmtime(_LIB) >= os.path.getmtime(f) for f in _SRCS):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    base = ["gcc", "-O2", "-std=c11", "-shared", "-fPIC", "-o", tmp] + _SRCS + ["-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True,
                       capture_output=True, text=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True, text=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            p = ctypes.c_void_p
            i64 = ctypes.c_int64
            lib.oracle_gemm_epilogue_f64.argtypes = [p, p, p, p, i64, i64, i64, i64, i64,
                                                     p, i64, ctypes.c_int, ctypes.c_int]
            lib.oracle_gemm_epilogue_f64.restype = ctypes.c_int
            lib.oracle_round.argtypes = [p, p, i64, ctypes.c_int]
            lib.oracle_round.restype = ctypes.c_int
            lib.oracle_decode.argtypes = [p, p, i64, ctypes.c_int]
            lib.oracle_decode.restype = ctypes.c_int
            lib.oracle_max_threads.restype = ctypes.c_int
            lib.oracle_attention_f64.argtypes = [p, p, p, p, i64, i64, i64, i64, ctypes.c_int, ctypes.c_int,
                                                 p, i64, ctypes.c_int]
            lib.oracle_attention_f64.restype = ctypes.c_int
            lib.oracle_set_threads.argtypes = [ctypes.c_int]
            _lib = lib
    return _lib


def _u16(x) -> np.ndarray:
    a = np.asarray(x)
    if a.dtype != np.uint16:
        a = a.view(np.uint16)
    return a


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def gemm_epilogue_f64(A, B, bias, M: int, N: int, K: int, dtype: int, epilogue: int,
                      rows=None) -> np.ndarray:
    """Unrounded fp64 result epi(A.B + bias) for all rows, or for `rows` only.

    A: uint16 array [M, lda] (lda >= K), B: uint16 array [K, ldb] (ldb >= N),
    bias: uint16 array [N] or None.  Returns float64 [len(rows) or M, N].
    """
    lib = _load()
    A = np.ascontiguousarray(_u16(A)) if A is not None else np.zeros((max(M, 1), max(K, 1)), np.uint16)
    B = np.ascontiguousarray(_u16(B)) if B is not None else np.zeros((max(K, 1), max(N, 1)), np.uint16)
    lda = A.shape[1] if A.ndim == 2 else K
    ldb = B.shape[1] if B.ndim == 2 else N
    if bias is not None:
        bias = np.ascontiguousarray(_u16(bias))
    rows_arr = None
    nrows = M
    if rows is not None:
        rows_arr = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
        nrows = rows_arr.shape[0]
    out = np.empty((nrows, N), dtype=np.float64)
    rc = lib.oracle_gemm_epilogue_f64(
        _ptr(A), _ptr(B), _ptr(bias) if bias is not None else None, _ptr(out),
        M, N, K, lda, ldb, _ptr(rows_arr) if rows_arr is not None else None, nrows,
        int(dtype), int(epilogue))
    if rc != 0:
        raise ValueError(f"oracle rejected the arguments (rc={rc})")
    return out


def round_to(ref: np.ndarray, dtype: int) -> np.ndarray:
    """Round fp64 values to fp16/bf16 bit patterns (uint16), ties to even."""
    lib = _load()
    ref = np.ascontiguousarray(ref, dtype=np.float64)
    out = np.empty(ref.shape, dtype=np.uint16)
    if lib.oracle_round(_ptr(ref), _ptr(out), ref.size, int(dtype)) != 0:
        raise ValueError("bad dtype")
    return out


def decode(bits, dtype: int) -> np.ndarray:
    """Exact fp16/bf16 bit patterns -> float64."""
    lib = _load()
    bits = np.ascontiguousarray(_u16(bits))
    out = np.empty(bits.shape, dtype=np.float64)
    if lib.oracle_decode(_ptr(bits), _ptr(out), bits.size, int(dtype)) != 0:
        raise ValueError("bad dtype")
    return out


def max_threads() -> int:
    return int(_load().oracle_max_threads())


def set_threads(n: int) -> None:
    _load().oracle_set_threads(int(n))


def attention_f64(Q, K, V, B: int, S: int, H: int, D: int, causal: bool, dtype: int, rows=None,
                  abs_v: bool = False) -> np.ndarray:
    """Unrounded fp64 attention output of "TileLang で GPU カーネル設計を解説" §6.

    Q, K, V: uint16 bit patterns [B, S, H, D] (any shape with that many
    elements, row-major).  Returns float64 [B*S*H, D] (every row, in [B, S, H]
    order) or [len(rows), D] for rows given as flat (b * S + i) * H + h.  With
    abs_v, |V| replaces V (the magnitude sum_j w_ij |V_j|).
    """
    lib = _load()
    q = np.ascontiguousarray(_u16(Q)).reshape(-1)
    k = np.ascontiguousarray(_u16(K)).reshape(-1)
    v = np.ascontiguousarray(_u16(V)).reshape(-1)
    if not (q.size == k.size == v.size == B * S * H * D):
        raise ValueError("Q, K, V must each hold B*S*H*D elements")
    rows_arr = None
    nrows = B * S * H
    if rows is not None:
        rows_arr = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
        nrows = rows_arr.shape[0]
    out = np.empty((nrows, D), dtype=np.float64)
    rc = lib.oracle_attention_f64(_ptr(q), _ptr(k), _ptr(v), _ptr(out), B, S, H, D, int(bool(causal)),
                                  int(bool(abs_v)), _ptr(rows_arr) if rows_arr is not None else None, nrows,
                                  int(dtype))
    if rc != 0:
        raise ValueError(f"oracle rejected the arguments (rc={rc})")
    return out
