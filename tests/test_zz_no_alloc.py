"""The allocation-free entry point tgemm_run_noalloc, through the C ABI.

It exists for callers that must not allocate GPU memory: code whose device
memory is reserved up front by another allocator (where a library-side
allocation can fail or fragment that reserve), latency-bound loops that avoid
allocation calls, and deployments that forbid allocation after start-up.
Instead of drawing scratch from a pool, it repacks unaligned operands into a
fixed 64 MiB device array inside the library.

Checked here: two calls in a row whose operands need that scratch agree with
tgemm_run within the tolerance the other tests use (the two entry points may
sum the k products in different orders: tgemm_run may split k across CTAs for
small problems, this variant never does), both agree with the oracle, the
second call is not disturbed by what the first left in the shared array, and a
call that would need more scratch than the array holds is rejected before
anything runs.  This file is collected last so that a failure
here does not hide the rest of the suite; it also passes on its own in a fresh
process.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import seeded_inputs as si
from gpu_helpers import (SENTINEL, TINY, U_OUT, alloc_c, assert_bit_exact, assert_close, c_bits, decode, magnitude,
                         oracle_ref, to_device_pitched)

pytestmark = pytest.mark.gpu

SCRATCH_LIMIT = 7
DT = {"fp16": 0, "bf16": 1}
EPI = {"none": 0, "relu": 1, "bias": 2, "bias_relu": 3}


def prepare(M, N, K, dtype, seed, lda, ldb):
    A, B, bias = si.make_inputs(M, N, K, dtype, seed, lda=lda if lda != K else None,
                                ldb=ldb if ldb != N else None)
    return (A, B, bias), to_device_pitched(A, K), to_device_pitched(B, N), bias.to("cuda")


def call(fn, Ad, Bd, bd, Cd, M, N, K, dtype, epi):
    return fn(Ad.data_ptr(), Bd.data_ptr(), bd.data_ptr(), Cd.data_ptr(), M, N, K,
              Ad.stride(0), Bd.stride(0), Cd.stride(0), DT[dtype], EPI[epi],
              torch.cuda.current_stream().cuda_stream)


# (M, N, K, dtype, epilogue, seed, lda, ldb, ldc): each case repacks at least
# one operand into the fixed scratch.
CASES = [
    (1000, 1001, 520, "fp16", "bias_relu", 31, 520, 1001, 1001),   # B repacked, masked C stores
    (777, 640, 517, "bf16", "relu", 32, 517, 640, 648),            # A repacked, TMA C stores
    (513, 300, 301, "fp16", "bias", 33, 301, 300, 300),            # A and B repacked
]


def test_noalloc_matches_run_on_consecutive_calls(cuda_lib):
    prepared = []
    for (M, N, K, dt, epi, seed, lda, ldb, ldc) in CASES:
        inputs, Ad, Bd, bd = prepare(M, N, K, dt, seed, lda, ldb)
        prepared.append((inputs, Ad, Bd, bd, alloc_c(M, N, ldc, dt), alloc_c(M, N, ldc, dt)))
    # Back-to-back calls of the new entry point, then the existing one.
    for rep in range(2):
        for (M, N, K, dt, epi, *_), (inputs, Ad, Bd, bd, Cn, Cr) in zip(CASES, prepared):
            assert call(cuda_lib.tgemm_run_noalloc, Ad, Bd, bd, Cn, M, N, K, dt, epi) == 0
        torch.cuda.synchronize()
        for (M, N, K, dt, epi, seed, lda, ldb, ldc), (inputs, Ad, Bd, bd, Cn, Cr) in zip(CASES, prepared):
            if rep == 0:
                assert call(cuda_lib.tgemm_run, Ad, Bd, bd, Cr, M, N, K, dt, epi) == 0
            torch.cuda.synchronize()
            got, want = c_bits(Cn, M, ldc), c_bits(Cr, M, ldc)
            if ldc > N:
                assert (got[:, N:] == SENTINEL).all()
            used = (inputs[0], inputs[1], inputs[2] if epi in ("bias", "bias_relu") else None)
            ref = oracle_ref(used, M, N, K, dt, epi)
            mag = magnitude(used, N, K)
            what = f"case {M}x{N}x{K}, call {rep + 1}"
            assert_close(got[:, :N], ref, dt, "noalloc " + what, mag, K)
            assert_close(want[:, :N], ref, dt, "tgemm_run " + what, mag, K)
            # The two entry points against each other: each is within the derived
            # bound of the exact value, so they differ by at most twice that bound.
            gamma = 2.0 * (K + 2) * 2.0 ** -24
            bound = 2 * (U_OUT[dt] * np.abs(ref) + (1 + U_OUT[dt]) * gamma * mag + TINY[dt])
            diff = np.abs(decode(got[:, :N], dt) - decode(want[:, :N], dt))
            assert (diff <= bound).all(), what
    assert cuda_lib.tgemm_last_device_status() == 0


def test_noalloc_integer_inputs_bit_exact_on_a_few_tile_shape(cuda_lib):
    """A decode-like shape (few output tiles, long k loop) with an unaligned
    pitch of A: tgemm_run splits its k loop across CTAs, this variant never
    does, so their summation orders differ; with small-integer inputs every
    partial sum is exact, so both must equal the oracle's rounding bit for bit
    (and hence each other), on two calls in a row."""
    M, N, K, dt, epi, lda = 128, 1024, 4096, "fp16", "bias_relu", 4100
    plan = cuda_lib.tgemm_plan(M, N, K, torch.cuda.get_device_properties(0).multi_processor_count)
    assert plan["split_k"] > 1            # the two entry points really take different plans
    A, B, bias = si.make_inputs(M, N, K, dt, 41, kind="int", lda=lda)
    Ad, Bd, bd = to_device_pitched(A, K), B.to("cuda"), bias.to("cuda")
    want = oracle_ref((A, B, bias), M, N, K, dt, epi)
    Cr = alloc_c(M, N, N, dt)
    assert call(cuda_lib.tgemm_run, Ad, Bd, bd, Cr, M, N, K, dt, epi) == 0
    for rep in range(2):
        Cn = alloc_c(M, N, N, dt)
        assert call(cuda_lib.tgemm_run_noalloc, Ad, Bd, bd, Cn, M, N, K, dt, epi) == 0
        torch.cuda.synchronize()
        got = c_bits(Cn, M, N)
        assert_bit_exact(got, want, dt, f"noalloc int call {rep + 1}")
        assert (got == c_bits(Cr, M, N)).all(), f"noalloc and tgemm_run differ on call {rep + 1}"
    assert cuda_lib.tgemm_last_device_status() == 0


def test_noalloc_rejects_scratch_beyond_its_limit(cuda_lib):
    # lda = 4100 is unaligned, so A would be repacked: 8192 * 4104 * 2 B > 64 MiB.
    M, N, K = 8192, 64, 4100
    assert M * 4104 * 2 > cuda_lib.NOALLOC_SCRATCH_BYTES
    Ad = torch.zeros((M, K), dtype=torch.float16, device="cuda")
    Bd = torch.zeros((K, N), dtype=torch.float16, device="cuda")
    bd = torch.zeros((N,), dtype=torch.float16, device="cuda")
    Cd = alloc_c(M, N, N, "fp16")
    assert call(cuda_lib.tgemm_run_noalloc, Ad, Bd, bd, Cd, M, N, K, "fp16", "bias_relu") == SCRATCH_LIMIT
    torch.cuda.synchronize()
    assert (c_bits(Cd, M, N) == SENTINEL).all()
    assert "SCRATCH_LIMIT" in cuda_lib.tgemm_status_string(SCRATCH_LIMIT)
