"""GPU parity of the attention forward pass against the fp64 oracle, through the
C ABI (tgemm_attention_fwd).

Bound, per output element, against the unrounded fp64 value ref and the
magnitude mag = sum_j w_ij |V_j| (the oracle with |V|):

    |out - ref| <= (u_out + 1e-4) |ref| + (u_P + 2e-4) mag + 1e-6

u_out is the output rounding (2^-11 fp16, 2^-8 bf16); u_P the rounding of P to
the input format before P.V (the same u); the 1e-4 / 2e-4 terms cover the
fp32 arithmetic: the scores' fp32 dot products (64 terms) move each exponent
by about 1e-5 at these magnitudes, the P.V and row-sum accumulations over up
to 1024 keys add at most 1024 * 2^-24 = 6e-5 relative, exp2 and the rescale
factors a few ulp.  The page's own check (torch SDPA, relative error 3e-2) is
far looser.

Coverage: one block, ragged sequences (1, 129, 200, 255 keys), several heads
and batches, causal and not, both 16-bit formats, the page's workload
(4, 1024, 8, 64) on sampled rows, repeat-run determinism, large-magnitude
scores (softmax near one-hot), and the device status word.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import decode

pytestmark = pytest.mark.gpu

TDT = {"fp16": torch.float16, "bf16": torch.bfloat16}
ODT = {"fp16": oracle.F16, "bf16": oracle.BF16}
U = {"fp16": 2.0 ** -11, "bf16": 2.0 ** -8}


def bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def make_qkv(B, S, H, dtype, seed, scale=1.0):
    g = torch.Generator().manual_seed(seed)
    return [(torch.randn(B, S, H, 64, generator=g) * scale).to(TDT[dtype]) for _ in range(3)]


def run_attention(tg, q, k, v, causal):
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    o = torch.full_like(qd, float("nan"))
    tg.attention(qd, kd, vd, o, causal=causal)
    torch.cuda.synchronize()
    return o


def check(tg, B, S, H, dtype, causal, seed, rows=None, scale=1.0, what=""):
    q, k, v = make_qkv(B, S, H, dtype, seed, scale)
    o = run_attention(tg, q, k, v, causal)
    got = decode(bits(o).reshape(-1, 64), dtype)
    if rows is not None:
        got = got[rows]
    ref = oracle.attention_f64(bits(q), bits(k), bits(v), B, S, H, 64, causal, ODT[dtype], rows=rows)
    mag = oracle.attention_f64(bits(q), bits(k), bits(v), B, S, H, 64, causal, ODT[dtype], rows=rows, abs_v=True)
    assert np.isfinite(got).all(), what
    bound = (U[dtype] + 1e-4) * np.abs(ref) + (U[dtype] + 2e-4) * mag + 1e-6
    bad = np.abs(got - ref) > bound
    assert not bad.any(), (f"{what}: {int(bad.sum())} of {bad.size} outside the bound, "
                           f"worst excess {(np.abs(got - ref) - bound).max():.3e}")
    return o


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("B,S,H", [(1, 128, 1), (1, 1, 1), (2, 129, 3), (1, 200, 2), (3, 255, 1), (1, 384, 2)])
def test_attention_shapes(cuda_lib, B, S, H, dtype, causal):
    check(cuda_lib, B, S, H, dtype, causal, seed=B * 1000 + S + H, what=f"{B}x{S}x{H} {dtype} causal={causal}")


@pytest.mark.parametrize("causal", [False, True])
def test_attention_page_workload_sampled(cuda_lib, causal):
    """(batch, seq, heads, dim) = (4, 1024, 8, 64) fp16, randn inputs (the page's
    workload), rows sampled across batches, heads and query positions."""
    B, S, H = 4, 1024, 8
    rng = np.random.default_rng(3)
    fixed = [0, H - 1, (S - 1) * H, ((B - 1) * S + S - 1) * H + H - 1, (2 * S + 127) * H + 3, (S + 128) * H]
    rows = sorted(set(fixed) | set(rng.choice(B * S * H, size=400, replace=False).tolist()))
    check(cuda_lib, B, S, H, "fp16", causal, seed=21, rows=rows, what=f"page workload causal={causal}")


def test_attention_peaked_softmax(cuda_lib):
    """Scores of magnitude ~50: the running maximum changes often and the
    softmax is close to one-hot, which exercises the rescaling."""
    for causal in (False, True):
        check(cuda_lib, 1, 300, 2, "fp16", causal, seed=7, scale=3.0, what=f"peaked causal={causal}")


def test_attention_deterministic(cuda_lib):
    q, k, v = make_qkv(2, 300, 2, "bf16", 9)
    a = run_attention(cuda_lib, q, k, v, True)
    b = run_attention(cuda_lib, q, k, v, True)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_attention_leaves_status_ok(cuda_lib):
    check(cuda_lib, 1, 256, 1, "fp16", False, seed=5)
    assert cuda_lib.tgemm_last_device_status() == 0
