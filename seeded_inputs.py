"""Seeded synthetic inputs for the fused GEMM epilogue, shared by the tests,
the smoke check and the benchmark.

This module holds no arithmetic of the method itself: it only draws random
numbers and casts them to the 16-bit input dtype.  Both the CUDA path and the
CPU oracle read the very same quantised host arrays, so input quantisation is
never counted as error.

Recipe (the workloads' own description: A ~ N(0,1), B ~ N(0,1)/sqrt(K),
bias ~ N(0, 0.1), seeded):
  * torch.Generator('cpu').manual_seed(seed); fp32 draws in the order A, B, bias;
  * B is scaled by 1/sqrt(K) and bias by 0.1 (taken as the standard deviation)
    in fp32, then everything is cast to fp16/bf16 (round to nearest even);
  * the integer-exact variant draws every entry of A, B and bias uniformly from
    {-2, -1, 0, 1, 2} (torch.randint(-2, 3)), same order;
  * the GELU workload follows its page's recipe ("TileLang で GPU カーネル設計を
    解説" §4): A and B ~ N(0,1) / K^(1/4), bias ~ N(0,1), same order.
Padded leading dimensions fill the pad with NaN so a read of the pad shows up.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import torch

EPILOGUES = {"none": 0, "relu": 1, "bias": 2, "bias_relu": 3, "gelu": 4, "bias_gelu": 5}
DTYPES = {"fp16": torch.float16, "bf16": torch.bfloat16}


@dataclass(frozen=True)
class Workload:
    name: str
    M: int
    N: int
    K: int
    dtype: str
    epilogue: str
    seed: int
    kind: str = "normal"          # "normal" or "int"
    lda: int | None = None
    ldb: int | None = None
    ldc: int | None = None

    @property
    def flops(self) -> int:
        return 2 * self.M * self.N * self.K


# The five workloads of the method's evaluation, plus the integer-exact variant,
# the padded-pitch twin of the ragged case, the GELU page's workload and a
# decode shape.
WORKLOADS = {
    "c0": Workload("gemm_relu_256_fp16", 256, 256, 256, "fp16", "relu", 0),
    "c1": Workload("gemm_bias_relu_4096_fp16", 4096, 4096, 4096, "fp16", "bias_relu", 1),
    "c1x": Workload("gemm_bias_relu_4096_fp16_int", 4096, 4096, 4096, "fp16", "bias_relu", 1, kind="int"),
    "c2": Workload("gemm_bias_relu_8192_bf16", 8192, 8192, 8192, "bf16", "bias_relu", 2),
    "c3": Workload("gemm_bias_relu_skinny_128x28672x8192_fp16", 128, 28672, 8192, "fp16", "bias_relu", 3),
    "c4": Workload("gemm_bias_relu_ragged_8191x6143x4104_fp16", 8191, 6143, 4104, "fp16", "bias_relu", 4),
    "c4p": Workload("gemm_bias_relu_ragged_8191x6143x4104_fp16_ld6144", 8191, 6143, 4104, "fp16",
                    "bias_relu", 4, ldb=6144, ldc=6144),
    "c5": Workload("gemm_bias_gelu_4096x4096x1024_fp16", 4096, 4096, 1024, "fp16", "bias_gelu", 5,
                   kind="gelu"),
    # A decode shape (few rows, long k): the small-M case split in k.
    "d16": Workload("gemm_bias_relu_decode_16x4096x8192_fp16", 16, 4096, 8192, "fp16", "bias_relu", 6),
}


def _pad_cols(x: torch.Tensor, ld: int | None) -> torch.Tensor:
    if ld is None or ld == x.shape[1]:
        return x.contiguous()
    assert ld > x.shape[1]
    out = torch.full((x.shape[0], ld), float("nan"), dtype=x.dtype)
    out[:, : x.shape[1]] = x
    return out


def make_inputs(M: int, N: int, K: int, dtype: str = "fp16", seed: int = 0,
                kind: str = "normal", with_bias: bool = True,
                lda: int | None = None, ldb: int | None = None):
    """Return CPU tensors (A [M, lda], B [K, ldb], bias [N] or None) in `dtype`.

    Only the first K columns of A and N columns of B are the operands; a wider
    pitch leaves NaN in the pad.  The bias is always drawn (after A and B) so
    that A and B do not depend on `with_bias`.
    """
    tdt = DTYPES[dtype]
    g = torch.Generator("cpu").manual_seed(int(seed))
    if kind == "normal":
        a = torch.randn(M, K, generator=g, dtype=torch.float32)
        b = torch.randn(K, N, generator=g, dtype=torch.float32) * (1.0 / math.sqrt(max(K, 1)))
        bias = torch.randn(N, generator=g, dtype=torch.float32) * 0.1
    elif kind == "gelu":
        s = 1.0 / math.sqrt(math.sqrt(max(K, 1)))
        a = torch.randn(M, K, generator=g, dtype=torch.float32) * s
        b = torch.randn(K, N, generator=g, dtype=torch.float32) * s
        bias = torch.randn(N, generator=g, dtype=torch.float32)
    elif kind == "int":
        a = torch.randint(-2, 3, (M, K), generator=g).to(torch.float32)
        b = torch.randint(-2, 3, (K, N), generator=g).to(torch.float32)
        bias = torch.randint(-2, 3, (N,), generator=g).to(torch.float32)
    else:
        raise ValueError(kind)
    A = _pad_cols(a.to(tdt), lda)
    B = _pad_cols(b.to(tdt), ldb)
    return A, B, (bias.to(tdt).contiguous() if with_bias else None)


def make_workload(w: Workload):
    """Inputs of a named workload: (A, B, bias or None)."""
    with_bias = w.epilogue in ("bias", "bias_relu", "bias_gelu")
    return make_inputs(w.M, w.N, w.K, w.dtype, w.seed, w.kind, with_bias, w.lda, w.ldb)


def bits(x: torch.Tensor):
    """uint16 numpy view of a CPU fp16/bf16 tensor (the oracle's input form)."""
    return x.contiguous().view(torch.int16).numpy().view("uint16")


@dataclass(frozen=True)
class AttnWorkload:
    """Attention forward pass over [batch, seq, heads, dim] tensors."""
    name: str
    B: int
    S: int
    H: int
    D: int
    dtype: str
    causal: bool
    seed: int

    @property
    def flops(self) -> float:
        # 4 * B * H * S^2 * D (two GEMMs), half of it when causal, as the page counts.
        return 4.0 * self.B * self.H * self.S * self.S * self.D * (0.5 if self.causal else 1.0)


# The FlashAttention workload of "TileLang で GPU カーネル設計を解説" §6:
# (B, H, S, D) = (4, 8, 1024, 64), fp16, Q, K, V ~ N(0, 1); full and causal.
ATTN_WORKLOADS = {
    "fa": AttnWorkload("attention_fwd_4x1024x8x64_fp16", 4, 1024, 8, 64, "fp16", False, 22),
    "fa_causal": AttnWorkload("attention_fwd_causal_4x1024x8x64_fp16", 4, 1024, 8, 64, "fp16", True, 23),
}


def make_attention_inputs(w: AttnWorkload):
    """CPU tensors Q, K, V [B, S, H, D] in w.dtype: fp32 N(0, 1) draws in the
    order Q, K, V from one seeded generator, rounded to the 16-bit format."""
    g = torch.Generator("cpu").manual_seed(int(w.seed))
    return [torch.randn(w.B, w.S, w.H, w.D, generator=g, dtype=torch.float32).to(DTYPES[w.dtype])
            for _ in range(3)]
