"""Calls that consume the previous call's output on the same stream, with no
synchronisation in between.  Every kernel is enqueued as a programmatic
dependent launch (its set-up may overlap the end of the previous kernel), so
these check that nothing is read before the producing kernel has finished:
C1 = epi(A @ B + bias) is the A operand of the next call, through each kind
of plan (whole tiles, a k-split tail, split-K of every tile, the repack of an
unaligned pitch in front of the GEMM) and into the attention kernel.  Each
result is compared bit for bit with the oracle applied to the GPU's own
intermediate (small-integer inputs keep every sum exact)."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import gemm_epilogue_02_gb300 as tg
import oracle
import seeded_inputs as si
from gpu_helpers import alloc_c, assert_bit_exact, c_bits, decode, oracle_ref

pytestmark = pytest.mark.gpu


def int_tensor(shape, seed, lo=-2, hi=3):
    g = torch.Generator("cpu").manual_seed(seed)
    return torch.randint(lo, hi, shape, generator=g).to(torch.float16)


@pytest.mark.parametrize("M,N,K,N2", [
    (1024, 1024, 512, 768),      # whole tiles
    (4096, 4096, 1024, 512),     # pair tiles with a tail
    (16, 2048, 4096, 1024),      # split-K of every tile (few rows)
    (2560, 2048, 2048, 1536),    # k-split tail
])
def test_chained_calls_see_the_previous_result(cuda_lib, M, N, K, N2):
    # Entries in {-1, 0, 1} (bias in {-2..2}): every sum of both steps is an
    # integer far inside fp32's exact range, so each result is the oracle's
    # exact sum rounded once, bit for bit.
    A = int_tensor((M, K), 1, -1, 2)
    B = int_tensor((K, N), 2, -1, 2)
    bias = int_tensor((N,), 3)
    B2 = int_tensor((N, N2), 4, -1, 2)
    Ad, Bd, bd, B2d = A.cuda(), B.cuda(), bias.cuda(), B2.cuda()
    C1, C2, C3 = alloc_c(M, N, N, "fp16"), alloc_c(M, N2, N2, "fp16"), alloc_c(M, N2, N2, "fp16")
    s = torch.cuda.current_stream()
    # C1 -> C2 -> C3 back to back, twice (the second round rewrites C1 while
    # the host waits for nothing).
    for _ in range(2):
        tg.run(Ad, Bd, bd, C1, "bias_relu", stream=s)
        tg.run(C1, B2d, None, C2, "none", stream=s)
        tg.run(C1, B2d, None, C3, "relu", stream=s)
    torch.cuda.synchronize()
    c1 = c_bits(C1, M, N)
    assert_bit_exact(c1, oracle_ref((A, B, bias), M, N, K, "fp16", "bias_relu"), "fp16", f"chain step 1 {M}x{N}x{K}")
    C1h = torch.from_numpy(c1.view(np.int16)).view(torch.float16)
    assert np.isfinite(decode(c1, "fp16")).all()
    ref2 = oracle_ref((C1h, B2, None), M, N2, N, "fp16", "none")
    assert np.abs(ref2).max() < 65504.0   # no overflow: every output is a finite fp16
    assert_bit_exact(c_bits(C2, M, N2), ref2, "fp16", f"chain step 2 {M}x{N2}x{N}")
    ref3 = oracle_ref((C1h, B2, None), M, N2, N, "fp16", "relu")
    assert_bit_exact(c_bits(C3, M, N2), ref3, "fp16", f"chain step 3 {M}x{N2}x{N}")


def test_chain_through_a_repacked_operand(cuda_lib):
    """The second call's A has an unaligned pitch, so a repack kernel runs in
    front of its GEMM; it reads C1 straight after the first call."""
    M, N, K, N2 = 1000, 1003, 256, 640
    A = int_tensor((M, K), 11, -1, 2)
    B = int_tensor((K, N), 12, -1, 2)
    B2 = int_tensor((N, N2), 13, -1, 2)
    C1 = alloc_c(M, N, N, "fp16")   # pitch 1003: not a multiple of 8
    C2 = alloc_c(M, N2, N2, "fp16")
    s = torch.cuda.current_stream()
    tg.run(A.cuda(), B.cuda(), None, C1, "relu", stream=s)
    tg.run(C1, B2.cuda(), None, C2, "none", stream=s)
    torch.cuda.synchronize()
    c1 = c_bits(C1, M, N)
    assert_bit_exact(c1, oracle_ref((A, B, None), M, N, K, "fp16", "relu"), "fp16", "repack chain step 1")
    C1h = torch.from_numpy(c1.view(np.int16)).view(torch.float16)
    assert_bit_exact(c_bits(C2, M, N2), oracle_ref((C1h, B2, None), M, N2, N, "fp16", "none"), "fp16",
                     "repack chain step 2")


def test_attention_after_a_gemm_reads_its_output(cuda_lib):
    """Q is written by a GEMM right before the attention call (no sync): the
    attention output must be the oracle's on the GEMM's Q."""
    w = si.AttnWorkload("chain", 1, 256, 2, 64, "fp16", False, 5)
    _, k, v = si.make_attention_inputs(w)
    M, K = w.B * w.S * w.H, 64
    X = int_tensor((M, K), 21, -1, 2)
    Wm = (int_tensor((K, w.D), 22, -1, 2) * 0.125).to(torch.float16)   # exact products
    Qd = alloc_c(M, w.D, w.D, "fp16")
    O = torch.empty(w.B, w.S, w.H, w.D, dtype=torch.float16, device="cuda")
    kd, vd = k.cuda(), v.cuda()
    s = torch.cuda.current_stream()
    tg.run(X.cuda(), Wm.cuda(), None, Qd, "none", stream=s)
    tg.attention(Qd.view(w.B, w.S, w.H, w.D), kd, vd, O, causal=False, stream=s)
    torch.cuda.synchronize()
    q_bits = c_bits(Qd, M, w.D)
    assert_bit_exact(q_bits, oracle_ref((X, Wm, None), M, w.D, K, "fp16", "none"), "fp16", "Q from the GEMM")
    q = torch.from_numpy(q_bits.view(np.int16)).view(torch.float16).view(w.B, w.S, w.H, w.D)
    ref = oracle.attention_f64(si.bits(q), si.bits(k), si.bits(v), w.B, w.S, w.H, w.D, False, oracle.F16)
    got = O.float().cpu().numpy().astype(np.float64)
    err = np.abs(got - ref.reshape(got.shape)).max()
    assert err < 2e-2, err
