"""Shared helpers of the GPU parity tests: seeded inputs -> device (with the
requested pitches) -> C-ABI call -> comparison against the fp64 oracle."""
from __future__ import annotations

import numpy as np
import torch

import oracle
import seeded_inputs as si

EPI = {"none": 0, "relu": 1, "bias": 2, "bias_relu": 3, "gelu": 4, "bias_gelu": 5}
BIAS_EPIS = ("bias", "bias_relu", "bias_gelu")
ODT = {"fp16": oracle.F16, "bf16": oracle.BF16}
TDT = {"fp16": torch.float16, "bf16": torch.bfloat16}
SENTINEL = 0x7E5A          # a NaN bit pattern in both fp16 and bf16; must survive in C's pad

# Bounds from the method's evaluation: relative Frobenius <= 2e-3 and
# |err| <= 1e-2 + 1e-2 |ref| per element, against the unrounded fp64 oracle.
FROB_TOL = 2e-3
ATOL, RTOL = 1e-2, 1e-2


def to_device_pitched(x: torch.Tensor, width: int) -> torch.Tensor:
    """Copy a CPU [rows, ld] tensor to the GPU and return the [rows, width] view."""
    d = x.to("cuda")
    return d[:, :width]


GUARD_ROWS = 3


def alloc_c(M: int, N: int, ldc: int, dtype: str) -> torch.Tensor:
    """C [M, N] with pitch ldc inside a sentinel-filled buffer with guard rows below."""
    full = torch.full((M + GUARD_ROWS, ldc), SENTINEL, dtype=torch.int16, device="cuda")
    return full.view(TDT[dtype])[:M, :N]


def c_bits(C: torch.Tensor, M: int, ldc: int) -> np.ndarray:
    """All of C's rows including the pad columns, as uint16 [M, ldc]; checks
    that the guard rows below C kept their sentinel."""
    whole = C.as_strided((M + GUARD_ROWS, ldc), (ldc, 1))
    bits = whole.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
    assert (bits[M:] == SENTINEL).all(), "rows below C were written"
    return bits[:M]


def run_tgemm(tg, M, N, K, dtype="fp16", epilogue="bias_relu", seed=0, kind="normal",
              lda=None, ldb=None, ldc=None):
    """Returns (A, B, bias) CPU inputs and the uint16 [M, ldc] result (pad included)."""
    lda = lda or K
    ldb = ldb or N
    ldc = ldc or N
    with_bias = epilogue in BIAS_EPIS
    A, B, bias = si.make_inputs(M, N, K, dtype, seed, kind, with_bias=True,
                                lda=lda if lda != K else None, ldb=ldb if ldb != N else None)
    Ad = to_device_pitched(A, K) if M * K > 0 else torch.empty((M, K), dtype=TDT[dtype], device="cuda")
    Bd = to_device_pitched(B, N) if K * N > 0 else torch.empty((K, N), dtype=TDT[dtype], device="cuda")
    biasd = bias.to("cuda") if with_bias else None
    Cd = alloc_c(M, N, ldc, dtype)
    tg.run(Ad, Bd, biasd, Cd, epilogue)
    torch.cuda.synchronize()
    return (A, B, bias if with_bias else None), c_bits(Cd, M, ldc)


def oracle_ref(inputs, M, N, K, dtype, epilogue, rows=None):
    A, B, bias = inputs
    return oracle.gemm_epilogue_f64(si.bits(A) if M * K else None, si.bits(B) if K * N else None,
                                    si.bits(bias) if bias is not None else None, M, N, K,
                                    ODT[dtype], EPI[epilogue], rows=rows)


def decode(bits: np.ndarray, dtype: str) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(TDT[dtype])
    return t.to(torch.float64).numpy()


# Unit roundoff of the output format and half its smallest subnormal step.
U_OUT = {"fp16": 2.0 ** -11, "bf16": 2.0 ** -8}
TINY = {"fp16": 2.0 ** -25, "bf16": 2.0 ** -134}
# Below this many compared elements the Frobenius bound is not a meaningful
# statistic (a handful of bf16 roundings can exceed 2e-3 on their own).
FROB_MIN_ELEMENTS = 4096


def magnitude(inputs, N, K, rows=None) -> np.ndarray:
    """sum_k |A[i,k] B[k,j]| + |bias[j]| over the logical [M, N] (fp32 is ample for a bound)."""
    A, B, bias = inputs
    m = A.shape[0] if rows is None else len(rows)
    if K == 0:
        mag = np.zeros((m, N), np.float32)
    else:
        a = A[:, :K].float().abs()
        if rows is not None:
            a = a[rows]
        mag = (a @ B[:, :N].float().abs()).numpy()
    if bias is not None:
        mag = mag + bias.float().abs().numpy()[None, :]
    return mag.astype(np.float64)


def assert_close(got_bits: np.ndarray, ref: np.ndarray, dtype: str, what="", mag=None, K=None,
                 pre=None):
    """Two bounds against the unrounded fp64 oracle:
    * derived from the arithmetic (every element, any size): the fp32 sum of K
      exact products carries at most (K+2) ulp-sized errors, taken twice over
      for the tensor core's internal alignment, and one rounding to the output
      format:  |got - ref| <= u_out |ref| + (1 + u_out) 2 (K+2) 2^-24 mag + tiny;
    * the method's own statistical bounds (relative Frobenius <= 2e-3,
      |err| <= 1e-2 + 1e-2 |ref|) when at least FROB_MIN_ELEMENTS are compared.
    With a GELU epilogue `pre` is the unrounded pre-activation: the sum's error
    passes through GELU with slope at most 1.13 (taken as 1.2), and the fp32
    evaluation of the activation adds at most 1e-5 |pre|."""
    got = decode(got_bits, dtype)
    assert got.shape == ref.shape
    finite = np.isfinite(ref)
    assert np.array_equal(np.isnan(got), np.isnan(ref)), what
    diff = np.abs(got[finite] - ref[finite])
    if mag is not None:
        gamma = 2.0 * (K + 2) * 2.0 ** -24
        u = U_OUT[dtype]
        if pre is None:
            bound = u * np.abs(ref[finite]) + (1 + u) * gamma * mag[finite] + TINY[dtype]
        else:
            bound = (u * np.abs(ref[finite]) + 1.2 * (1 + u) * gamma * mag[finite]
                     + 1e-5 * np.abs(pre[finite]) + TINY[dtype])
        bad = diff > bound
        assert not bad.any(), (f"{what}: {int(bad.sum())} elements outside the derived bound, "
                               f"worst excess {(diff - bound).max():.3e}")
    rel = np.linalg.norm(diff) / max(np.linalg.norm(ref[finite]), 1e-12)
    if diff.size >= FROB_MIN_ELEMENTS:
        assert rel <= FROB_TOL, f"{what}: relative Frobenius error {rel:.3e}"
        bad = diff > ATOL + RTOL * np.abs(ref[finite])
        assert not bad.any(), f"{what}: {int(bad.sum())} elements outside 1e-2 + 1e-2|ref|, max {diff.max():.3e}"
    return rel


def canon_zero(bits: np.ndarray) -> np.ndarray:
    """-0.0 -> +0.0 (the sign of an exact zero sum is not fixed by the method)."""
    b = bits.copy()
    b[b == 0x8000] = 0
    return b


def assert_bit_exact(got_bits: np.ndarray, ref: np.ndarray, dtype: str, what=""):
    want = oracle.round_to(ref, ODT[dtype])
    g, w = canon_zero(got_bits), canon_zero(want)
    mism = g != w
    assert not mism.any(), f"{what}: {int(mism.sum())} mismatches, first at {np.argwhere(mism)[0]}"


def assert_pad_untouched(bits_full: np.ndarray, N: int, what=""):
    if bits_full.shape[1] > N:
        assert (bits_full[:, N:] == SENTINEL).all(), f"{what}: C's pitch padding was written"


def check_epilogue(got_bits: np.ndarray, inputs, M, N, K, dtype, epilogue, what="", rows=None):
    """Tolerance check of any epilogue (GELU included) against the oracle."""
    ref = oracle_ref(inputs, M, N, K, dtype, epilogue, rows=rows)
    pre = None
    if epilogue in ("gelu", "bias_gelu"):
        pre = oracle_ref(inputs, M, N, K, dtype, "bias" if epilogue == "bias_gelu" else "none", rows=rows)
    return assert_close(got_bits, ref, dtype, what, magnitude(inputs, N, K, rows), K, pre)


def run_tgemm_layout(tg, M, N, K, dtype="fp16", epilogue="bias_relu", seed=0, kind="normal",
                     transpose_a=False, transpose_b=False, pad_a=0, pad_b=0):
    """Like run_tgemm, with A stored as [K, M] (transpose_a) and/or B stored as
    [N, K] (transpose_b), each with `pad_*` extra (NaN) columns of pitch.
    Returns the logical (A [M, K], B [K, N], bias) inputs and C's bits."""
    A, B, bias = si.make_inputs(M, N, K, dtype, seed, kind, with_bias=True)
    def stored(x, transpose, pad):
        x = x.t().contiguous() if transpose else x
        if pad:
            full = torch.full((x.shape[0], x.shape[1] + pad), float("nan"), dtype=x.dtype)
            full[:, : x.shape[1]] = x
            x = full
        return x.to("cuda")[:, : (x.shape[1] - pad)]
    Ad = stored(A, transpose_a, pad_a)
    Bd = stored(B, transpose_b, pad_b)
    with_bias = epilogue in BIAS_EPIS
    Cd = alloc_c(M, N, N, dtype)
    tg.run(Ad, Bd, bias.to("cuda") if with_bias else None, Cd, epilogue,
           transpose_a=transpose_a, transpose_b=transpose_b)
    torch.cuda.synchronize()
    return (A, B, bias if with_bias else None), c_bits(Cd, M, N)
