"""Pins for the CPU oracle, against facts other than the oracle itself.

The pages print no worked numeric example for the GEMM epilogue, so the pins
are mathematical (the definition C[i,j] = sum_k A[i,k] B[k,j] of "从零开始学习
TileLang…" §10.1, the epilogue relu(a @ b + bias) of its §10.8, and max(x, 0)
of "Writing high-performance kernels in TileLang", "Écrivons un GEMM"):

  * brute force in exact rational arithmetic on tiny shapes (incl. the
    M=2, N=8, K=4 debugging shape of that tutorial's §16.1), within the fp64
    summation error bound;
  * special cases with closed forms: identity / permutation / all-ones / zero
    operands, K = 0;
  * small-integer inputs whose sums are exact, against numpy int64 matmul;
  * invariants: ReLU output >= +0 with no -0.0, RELU = max(NONE, 0),
    linearity in A, power-of-two homogeneity;
  * an fp32 library matmul (torch CPU) within the fp32 error bound;
  * exhaustive decode of all 65536 bit patterns and rounding against numpy,
    torch and a brute-force nearest-value search.

Every pin takes the oracle function as an argument so the mutation tests at
the bottom can show that a planted mistake (transposed operand, dropped bias,
bias indexed by row, ReLU before the bias, dropped k term, sign flip, -0.0
kept, wrong row pitch) fails at least one pin.
"""
from __future__ import annotations

import math
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
import seeded_inputs as si

EPIS = [oracle.EPI_NONE, oracle.EPI_RELU, oracle.EPI_BIAS, oracle.EPI_BIAS_RELU]
DTS = {oracle.F16: "fp16", oracle.BF16: "bf16"}


def has_bias(epi):
    return epi in (oracle.EPI_BIAS, oracle.EPI_BIAS_RELU, oracle.EPI_BIAS_GELU)


def has_relu(epi):
    return epi in (oracle.EPI_RELU, oracle.EPI_BIAS_RELU)


def has_gelu(epi):
    return epi in (oracle.EPI_GELU, oracle.EPI_BIAS_GELU)


# Library decoders, independent of the oracle's C decode.
def lib_decode(bits: np.ndarray, dt: int) -> np.ndarray:
    bits = np.ascontiguousarray(bits, dtype=np.uint16)
    if dt == oracle.F16:
        return bits.view(np.float16).astype(np.float64)
    t = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16)
    return t.to(torch.float64).numpy()


def to_bits(x: np.ndarray, dt: int) -> np.ndarray:
    """Library rounding of float64 values that are exactly representable in float32."""
    if dt == oracle.F16:
        return np.asarray(x, np.float64).astype(np.float16).view(np.uint16)
    t = torch.from_numpy(np.asarray(x, np.float64).astype(np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def rand_bits(shape, dt, rng, scale=1.0):
    x = rng.standard_normal(shape).astype(np.float32) * np.float32(scale)
    return to_bits(x.astype(np.float64), dt)


def pad(bits: np.ndarray, extra: int, dt: int) -> np.ndarray:
    """Append `extra` NaN columns (a wider row pitch)."""
    if extra == 0:
        return bits
    nan = to_bits(np.array([np.nan]), dt)[0]
    out = np.full((bits.shape[0], bits.shape[1] + extra), nan, dtype=np.uint16)
    out[:, : bits.shape[1]] = bits
    return out


def epi_f64(x: np.ndarray, bias_d, epi):
    """Apply the epilogue to exact (or library) fp64 values for comparisons."""
    if has_bias(epi):
        x = x + bias_d[None, :]
    if has_relu(epi):
        x = np.where(x > 0, x, 0.0)
    return x


# --------------------------------------------------------------------------- pins
def pin_bruteforce_tiny(fn):
    rng = np.random.default_rng(1234)
    sizes = [1, 2, 3, 5, 8]
    cases = [(m, n, k) for m in sizes for n in sizes for k in sizes]
    cases += [(2, 8, 4)] * 8
    for idx, (M, N, K) in enumerate(cases):
        epi = EPIS[idx % 4]
        dt = [oracle.F16, oracle.BF16][(idx // 4) % 2]
        A = rand_bits((M, K), dt, rng)
        B = rand_bits((K, N), dt, rng)
        bias = rand_bits((N,), dt, rng, 0.1)
        Ap, Bp = pad(A, idx % 3, dt), pad(B, (idx // 3) % 4, dt)
        got = fn(Ap, Bp, bias if has_bias(epi) else None, M, N, K, dt, epi)
        Ad, Bd, bd = lib_decode(A, dt), lib_decode(B, dt), lib_decode(bias, dt)
        for i in range(M):
            for j in range(N):
                exact = sum((Fraction(Ad[i, k]) * Fraction(Bd[k, j]) for k in range(K)), Fraction(0))
                mag = sum(abs(Ad[i, k] * Bd[k, j]) for k in range(K))
                if has_bias(epi):
                    exact += Fraction(bd[j])
                    mag += abs(bd[j])
                if has_relu(epi) and exact <= 0:
                    exact = Fraction(0)
                bound = (K + 2) * 2.0 ** -53 * mag
                err = abs(Fraction(float(got[i, j])) - exact)
                assert err <= Fraction(bound), (M, N, K, epi, dt, i, j, float(err), bound)


def pin_identity_and_permutation(fn):
    rng = np.random.default_rng(7)
    for dt in (oracle.F16, oracle.BF16):
        for (K, N) in [(37, 53), (16, 16)]:
            eye = to_bits(np.eye(K), dt)
            B = rand_bits((K, N), dt, rng)
            bias = rand_bits((N,), dt, rng, 0.1)
            Bd, bd = lib_decode(B, dt), lib_decode(bias, dt)
            got = fn(pad(eye, 3, dt), pad(B, 5, dt), None, K, N, K, dt, oracle.EPI_NONE)
            assert np.array_equal(got, Bd)
            got = fn(eye, B, bias, K, N, K, dt, oracle.EPI_BIAS_RELU)
            assert np.array_equal(got, np.maximum(Bd + bd[None, :], 0.0))
            perm = rng.permutation(K)
            P = to_bits(np.eye(K)[perm], dt)
            got = fn(P, B, None, K, N, K, dt, oracle.EPI_NONE)
            assert np.array_equal(got, Bd[perm])
            # B = I: C = A.
            A = rand_bits((N, K), dt, rng)
            got = fn(A, to_bits(np.eye(K), dt), None, N, K, K, dt, oracle.EPI_NONE)
            assert np.array_equal(got, lib_decode(A, dt))


def pin_zero_and_ones(fn):
    rng = np.random.default_rng(8)
    for dt in (oracle.F16, oracle.BF16):
        M, N, K = 9, 21, 13
        bias = rand_bits((N,), dt, rng, 0.1)
        bd = lib_decode(bias, dt)
        zeros_a = to_bits(np.zeros((M, K)), dt)
        B = rand_bits((K, N), dt, rng)
        for epi in EPIS:
            got = fn(zeros_a, B, bias if has_bias(epi) else None, M, N, K, dt, epi)
            want = epi_f64(np.zeros((M, N)), bd, epi)
            assert np.array_equal(got, want)
            if has_relu(epi):
                assert not np.signbit(got).any()
            # K = 0: the empty sum is 0.
            got0 = fn(None, None, bias if has_bias(epi) else None, M, N, 0, dt, epi)
            assert np.array_equal(got0, want)
        ones_a = to_bits(np.ones((M, K)), dt)
        ones_b = to_bits(np.ones((K, N)), dt)
        got = fn(ones_a, ones_b, bias, M, N, K, dt, oracle.EPI_BIAS)
        assert np.array_equal(got, np.full((M, N), float(K)) + bd[None, :])


def pin_integer_exact(fn):
    """Small integers: every partial sum is an exact integer (|s| <= 4K + 2 < 2^24)."""
    g = torch.Generator().manual_seed(1)
    M, N, K = 24, 40, 4096
    a = torch.randint(-2, 3, (M, K), generator=g)
    b = torch.randint(-2, 3, (K, N), generator=g)
    bias = torch.randint(-2, 3, (N,), generator=g)
    exact = a.numpy().astype(np.int64) @ b.numpy().astype(np.int64)
    for dt in (oracle.F16, oracle.BF16):
        Ab, Bb, bb = (to_bits(x.numpy().astype(np.float64), dt) for x in (a, b, bias))
        for epi in EPIS:
            got = fn(Ab, Bb, bb if has_bias(epi) else None, M, N, K, dt, epi)
            want = exact + (bias.numpy()[None, :] if has_bias(epi) else 0)
            if has_relu(epi):
                want = np.maximum(want, 0)
            assert np.array_equal(got, want.astype(np.float64))
            assert np.array_equal(oracle.round_to(got, dt), to_bits(want.astype(np.float64), dt))


def pin_relu_invariants(fn):
    rng = np.random.default_rng(9)
    for dt in (oracle.F16, oracle.BF16):
        M, N, K = 33, 47, 70
        A, B = rand_bits((M, K), dt, rng), rand_bits((K, N), dt, rng)
        bias = rand_bits((N,), dt, rng, 0.1)
        none = fn(A, B, None, M, N, K, dt, oracle.EPI_NONE)
        relu = fn(A, B, None, M, N, K, dt, oracle.EPI_RELU)
        withb = fn(A, B, bias, M, N, K, dt, oracle.EPI_BIAS)
        br = fn(A, B, bias, M, N, K, dt, oracle.EPI_BIAS_RELU)
        assert (none < 0).any() and (none > 0).any()
        for r, pre in ((relu, none), (br, withb)):
            assert (r >= 0).all() and not np.signbit(r).any()
            assert np.array_equal(r, np.where(pre > 0, pre, 0.0))
        bd = lib_decode(bias, dt)
        assert np.array_equal(withb, none + bd[None, :])
        # Exact zeros before the activation become +0.0, never -0.0.
        Aneg = to_bits(-np.ones((2, 4)), dt)
        Bz = to_bits(np.array([[0.0] * 3] * 4), dt)
        z = fn(Aneg, Bz, None, 2, 3, 4, dt, oracle.EPI_RELU)
        assert np.array_equal(z, np.zeros((2, 3))) and not np.signbit(z).any()


def pin_linearity_homogeneity(fn):
    rng = np.random.default_rng(10)
    for dt in (oracle.F16, oracle.BF16):
        M, N, K = 17, 29, 64
        a1 = rng.integers(-8, 9, (M, K)) / 8.0
        a2 = rng.integers(-8, 9, (M, K)) / 8.0
        B = rand_bits((K, N), dt, rng)
        A1, A2, A12 = to_bits(a1, dt), to_bits(a2, dt), to_bits(a1 + a2, dt)
        c1 = fn(A1, B, None, M, N, K, dt, oracle.EPI_NONE)
        c2 = fn(A2, B, None, M, N, K, dt, oracle.EPI_NONE)
        c12 = fn(A12, B, None, M, N, K, dt, oracle.EPI_NONE)
        Bd = lib_decode(B, dt)
        mag = (np.abs(a1) + np.abs(a2)) @ np.abs(Bd)
        assert np.all(np.abs(c12 - (c1 + c2)) <= 1e-12 * mag + 1e-300)
        # Scaling A and bias by 2^3 scales the result by 2^3 exactly.
        A = rand_bits((M, K), dt, rng)
        bias = rand_bits((N,), dt, rng, 0.1)
        A8 = to_bits(lib_decode(A, dt) * 8.0, dt)
        b8 = to_bits(lib_decode(bias, dt) * 8.0, dt)
        c = fn(A, B, bias, M, N, K, dt, oracle.EPI_BIAS_RELU)
        c8 = fn(A8, B, b8, M, N, K, dt, oracle.EPI_BIAS_RELU)
        assert np.array_equal(c8, 8.0 * c)


def pin_fp32_library(fn):
    """fp32 CPU matmul (a library routine) agrees within the fp32 error bound."""
    A, B, _ = si.make_inputs(256, 256, 256, "fp16", seed=0, with_bias=False)
    got = fn(si.bits(A), si.bits(B), None, 256, 256, 256, oracle.F16, oracle.EPI_RELU)
    lib = torch.relu(A.float() @ B.float()).double().numpy()
    mag = (A.double().abs() @ B.double().abs()).numpy()
    assert np.all(np.abs(got - lib) <= 256 * 2.0 ** -24 * mag * 1.01)


def pin_row_subset(fn):
    rng = np.random.default_rng(11)
    dt = oracle.BF16
    M, N, K = 40, 24, 19
    A, B = rand_bits((M, K), dt, rng), rand_bits((K, N), dt, rng)
    bias = rand_bits((N,), dt, rng, 0.1)
    full = fn(A, B, bias, M, N, K, dt, oracle.EPI_BIAS_RELU)
    rows = [39, 0, 17, 17, 5]
    sub = fn(A, B, bias, M, N, K, dt, oracle.EPI_BIAS_RELU, rows=rows)
    assert np.array_equal(sub, full[rows])


def pin_nan_inf(fn):
    """NaN/Inf inputs (the tutorial's edge-case list): NaN propagates through the
    ReLU as in torch.relu; +-Inf follow IEEE arithmetic."""
    for dt in (oracle.F16, oracle.BF16):
        A = to_bits(np.array([[1.0, np.nan], [1.0, 1.0], [np.inf, 0.5]]), dt)
        B = to_bits(np.array([[1.0, -1.0], [2.0, 3.0]]), dt)
        got = fn(A, B, None, 3, 2, 2, dt, oracle.EPI_RELU)
        assert np.isnan(got[0]).all()
        assert np.array_equal(got[1], [3.0, 2.0])
        assert got[2, 0] == np.inf                      # inf*1 + 0.5*2
        assert got[2, 1] == 0.0 and not np.signbit(got[2, 1])   # relu(-inf) = +0
        none = fn(A, B, None, 3, 2, 2, dt, oracle.EPI_NONE)
        assert none[2, 1] == -np.inf


def pin_gelu(fn):
    """GELU epilogue of "TileLang で GPU カーネル設計を解説" §4 (tanh form, after the
    bias): with A = I the pre-activation is exactly B + bias, so the output must
    equal torch's own tanh-approximation GELU of it (a library routine written
    with tanh, not the page's sigmoid form) to fp64 rounding; the sigmoid form
    satisfies gelu(x) - gelu(-x) = x exactly in real arithmetic; gelu(0) = +0."""
    rng = np.random.default_rng(13)
    for dt in (oracle.F16, oracle.BF16):
        K, N = 24, 40
        eye = to_bits(np.eye(K), dt)
        neg = to_bits(-np.eye(K), dt)
        B = rand_bits((K, N), dt, rng, 3.0)
        bias = rand_bits((N,), dt, rng, 1.0)
        pre = lib_decode(B, dt) + lib_decode(bias, dt)[None, :]
        got = fn(eye, B, bias, K, N, K, dt, oracle.EPI_BIAS_GELU)
        lib = torch.nn.functional.gelu(torch.from_numpy(pre), approximate="tanh").numpy()
        # The page prints 2*sqrt(2/pi) to 10 decimals (5.7e-12 short); with
        # sigma' <= 1/4 that moves gelu by at most ~1e-12 |x| over this range.
        assert np.all(np.abs(got - lib) <= 2e-12 * np.abs(pre) + 1e-300)
        pos = fn(eye, B, None, K, N, K, dt, oracle.EPI_GELU)
        negv = fn(neg, B, None, K, N, K, dt, oracle.EPI_GELU)
        x = lib_decode(B, dt)
        assert np.all(np.abs((pos - negv) - x) <= 4e-16 * np.abs(x))
        zero = fn(to_bits(np.zeros((3, K)), dt), B, None, 3, N, K, dt, oracle.EPI_GELU)
        assert np.array_equal(zero, np.zeros((3, N))) and not np.signbit(zero).any()
        # Saturation: far right of 0 the GELU is the identity, far left it vanishes.
        big = to_bits(np.array([[30.0], [-30.0]]), dt)
        one = to_bits(np.ones((1, 1)), dt)
        ends = fn(big, one, None, 2, 1, 1, dt, oracle.EPI_GELU)
        assert ends[0, 0] == 30.0 and abs(ends[1, 0]) < 1e-300


ALL_PINS = [pin_bruteforce_tiny, pin_identity_and_permutation, pin_zero_and_ones,
            pin_integer_exact, pin_relu_invariants, pin_linearity_homogeneity,
            pin_fp32_library, pin_row_subset, pin_nan_inf, pin_gelu]


@pytest.mark.parametrize("pin", ALL_PINS, ids=lambda p: p.__name__)
def test_oracle_pin(pin):
    pin(oracle.gemm_epilogue_f64)


# ------------------------------------------------------- decode and rounding pins
def _all_finite_sorted(dt):
    bits = np.arange(65536, dtype=np.uint16)
    vals = lib_decode(bits, dt)
    keep = np.isfinite(vals) & ~((vals == 0) & np.signbit(vals))
    order = np.argsort(vals[keep], kind="stable")
    return vals[keep][order], bits[keep][order]


def brute_round(x: float, dt: int, table) -> int:
    """Nearest representable value by search; ties to the even bit pattern;
    beyond max + half an ulp -> Inf (IEEE overflow rule)."""
    vals, bits = table
    if math.isnan(x):
        return -1
    mbits = 10 if dt == oracle.F16 else 7
    ebits = 5 if dt == oracle.F16 else 8
    sign = 1 << (mbits + ebits)
    inf = ((1 << ebits) - 1) << mbits
    vmax = vals[-1]
    half_ulp = (vmax - vals[-2]) / 2
    if abs(x) >= vmax + half_ulp:
        return inf | (sign if x < 0 else 0)
    if x == 0:
        return sign if math.copysign(1.0, x) < 0 else 0
    i = int(np.searchsorted(vals, x))
    cands = []
    for j in (i - 1, i):
        if 0 <= j < len(vals):
            cands.append((abs(Fraction(float(vals[j])) - Fraction(x)), int(bits[j]) & 1, int(bits[j])))
    cands.sort()
    best = cands[0]
    if len(cands) > 1 and cands[1][0] == best[0]:
        best = min(cands, key=lambda c: c[1])      # even significand wins the tie
    b = best[2]
    if b == 0 and x < 0:
        b = sign                                    # rounds to -0.0
    return b


def test_decode_exhaustive():
    bits = np.arange(65536, dtype=np.uint16)
    for dt in (oracle.F16, oracle.BF16):
        got = oracle.decode(bits, dt)
        want = lib_decode(bits, dt)
        same = (got == want) | (np.isnan(got) & np.isnan(want))
        assert same.all()
        assert np.array_equal(np.signbit(got[~np.isnan(got)]), np.signbit(want[~np.isnan(want)]))


def test_round_against_numpy_f16():
    rng = np.random.default_rng(5)
    x = np.concatenate([
        rng.standard_normal(200000) * 10.0 ** rng.uniform(-9, 5, 200000),
        np.array([65504.0, 65519.99, 65520.0, 65536.0, 2.0 ** -24, 2.0 ** -25,
                  2.0 ** -25 * 1.0000001, 3 * 2.0 ** -26, 2.0 ** -14, -0.0, 0.0,
                  np.inf, -np.inf, 1.0 + 2.0 ** -11, 1.0 + 3 * 2.0 ** -11]),
    ])
    x = np.concatenate([x, -x])
    got = oracle.round_to(x, oracle.F16)
    with np.errstate(over="ignore"):
        want = x.astype(np.float16).view(np.uint16)
    assert np.array_equal(got, want)


def test_round_bruteforce_both():
    rng = np.random.default_rng(6)
    for dt in (oracle.F16, oracle.BF16):
        table = _all_finite_sorted(dt)
        vals = table[0]
        mids = (vals[1:] + vals[:-1]) / 2                       # exact ties
        pick = rng.choice(len(mids), 3000, replace=False)
        x = np.concatenate([mids[pick], np.nextafter(mids[pick], np.inf),
                            np.nextafter(mids[pick], -np.inf),
                            rng.standard_normal(2000) * 10.0 ** rng.uniform(-45, 38, 2000),
                            [vals[-1] * 1.001, vals[0] * 1.001, 1e-300, -1e-300]])
        x = x[np.isfinite(x)]
        got = oracle.round_to(x, dt)
        for xi, gi in zip(x.tolist(), got.tolist()):
            assert gi == brute_round(xi, dt, table), (dt, xi, hex(gi))


def test_round_bf16_against_torch_float32():
    rng = np.random.default_rng(12)
    x32 = (rng.standard_normal(200000) * 10.0 ** rng.uniform(-40, 38, 200000)).astype(np.float32)
    x32 = x32[np.isfinite(x32)]
    got = oracle.round_to(x32.astype(np.float64), oracle.BF16)
    want = torch.from_numpy(x32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got, want)


# --------------------------------------------------------------- mutation tests
def _mut_transpose_b(A, B, bias, M, N, K, dt, epi, rows=None):
    if B is None:
        return oracle.gemm_epilogue_f64(A, B, bias, M, N, K, dt, epi, rows=rows)
    Bb = np.asarray(B)[:K, :N]
    if K == N:
        Bb = np.ascontiguousarray(Bb.T)
    return oracle.gemm_epilogue_f64(A, Bb, bias, M, N, K, dt, epi, rows=rows)


def _mut_drop_bias(A, B, bias, M, N, K, dt, epi, rows=None):
    e = {oracle.EPI_BIAS: oracle.EPI_NONE, oracle.EPI_BIAS_RELU: oracle.EPI_RELU,
         oracle.EPI_BIAS_GELU: oracle.EPI_GELU}.get(epi, epi)
    return oracle.gemm_epilogue_f64(A, B, None, M, N, K, dt, e, rows=rows)


def _mut_bias_by_row(A, B, bias, M, N, K, dt, epi, rows=None):
    if not has_bias(epi):
        return oracle.gemm_epilogue_f64(A, B, bias, M, N, K, dt, epi, rows=rows)
    out = oracle.gemm_epilogue_f64(A, B, None, M, N, K, dt, oracle.EPI_NONE, rows=rows)
    bd = oracle.decode(bias, dt)
    idx = np.arange(M) if rows is None else np.asarray(rows)
    out = out + bd[idx % N][:, None]
    return np.where(out > 0, out, 0.0) if has_relu(epi) else out


def _mut_relu_before_bias(A, B, bias, M, N, K, dt, epi, rows=None):
    if epi != oracle.EPI_BIAS_RELU:
        return oracle.gemm_epilogue_f64(A, B, bias, M, N, K, dt, epi, rows=rows)
    out = oracle.gemm_epilogue_f64(A, B, None, M, N, K, dt, oracle.EPI_RELU, rows=rows)
    return out + oracle.decode(bias, dt)[None, :]


def _mut_drop_last_k(A, B, bias, M, N, K, dt, epi, rows=None):
    if K == 0:
        return oracle.gemm_epilogue_f64(A, B, bias, M, N, K, dt, epi, rows=rows)
    Ak = np.ascontiguousarray(np.asarray(A)[:, : K - 1]) if K > 1 else None
    Bk = np.ascontiguousarray(np.asarray(B)[: K - 1]) if K > 1 else None
    return oracle.gemm_epilogue_f64(Ak, Bk, bias, M, N, K - 1, dt, epi, rows=rows)


def _mut_sign_flip(A, B, bias, M, N, K, dt, epi, rows=None):
    return -oracle.gemm_epilogue_f64(A, B, bias, M, N, K, dt, epi, rows=rows)


def _mut_negative_zero(A, B, bias, M, N, K, dt, epi, rows=None):
    out = oracle.gemm_epilogue_f64(A, B, bias, M, N, K, dt, epi, rows=rows)
    if has_relu(epi):
        out = np.where(out == 0, -0.0, out)
    return out


def _mut_pitch_ignored(A, B, bias, M, N, K, dt, epi, rows=None):
    if A is not None and np.asarray(A).ndim == 2 and np.asarray(A).shape[1] != K and M * K > 0:
        A = np.ascontiguousarray(A).reshape(-1)[: M * K].reshape(M, K)
    return oracle.gemm_epilogue_f64(A, B, bias, M, N, K, dt, epi, rows=rows)


def _gelu_wrong(x, c):
    return x / (1.0 + np.exp(-c * (x + 0.044715 * x * x * x)))


def _mut_gelu_constant(A, B, bias, M, N, K, dt, epi, rows=None):
    """GELU with the tanh-argument constant sqrt(2/pi) in the sigmoid form."""
    if not has_gelu(epi):
        return oracle.gemm_epilogue_f64(A, B, bias, M, N, K, dt, epi, rows=rows)
    pre_epi = oracle.EPI_BIAS if has_bias(epi) else oracle.EPI_NONE
    pre = oracle.gemm_epilogue_f64(A, B, bias, M, N, K, dt, pre_epi, rows=rows)
    with np.errstate(over="ignore"):
        return _gelu_wrong(pre, 0.7978845608)


def _mut_gelu_before_bias(A, B, bias, M, N, K, dt, epi, rows=None):
    if epi != oracle.EPI_BIAS_GELU:
        return oracle.gemm_epilogue_f64(A, B, bias, M, N, K, dt, epi, rows=rows)
    out = oracle.gemm_epilogue_f64(A, B, None, M, N, K, dt, oracle.EPI_GELU, rows=rows)
    return out + oracle.decode(bias, dt)[None, :]


MUTANTS = [_mut_transpose_b, _mut_drop_bias, _mut_bias_by_row, _mut_relu_before_bias,
           _mut_drop_last_k, _mut_sign_flip, _mut_negative_zero, _mut_pitch_ignored,
           _mut_gelu_constant, _mut_gelu_before_bias]


@pytest.mark.parametrize("mutant", MUTANTS, ids=lambda m: m.__name__)
def test_pins_catch_planted_mistake(mutant):
    caught = []
    for pin in ALL_PINS:
        try:
            pin(mutant)
        except (AssertionError, ValueError):
            caught.append(pin.__name__)
    assert caught, f"no pin fails for {mutant.__name__}"
