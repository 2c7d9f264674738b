"""Plain fp64 CPU oracles for C = act(A.B + bias) and for attention's output
O = softmax(scale * Q.K^T) V.

TEST INFRASTRUCTURE ONLY: the test suite, the smoke check and the benchmark's
CPU-baseline leg are the only callers.  The product library never imports,
links or calls anything under this directory, and this directory imports
nothing from the product package.

Parity pins (see tests/test_oracle_pins.py): brute force in exact rational
arithmetic on tiny shapes, identity / permutation / all-ones / zero special
cases, exact small-integer products against numpy int64 matmul, ReLU
invariants, linearity in A, power-of-two homogeneity, an fp32 library matmul
cross-check, and exhaustive decode / rounding checks against numpy, torch
and a brute-force nearest-value search.  Attention pins (see
tests/test_oracle_attention.py): torch's float64 scaled-dot-product attention,
closed forms for zero queries and single keys, key-permutation and score-shift
invariances.
"""
from .oracle import (  # noqa: F401
    F16, BF16, EPI_NONE, EPI_RELU, EPI_BIAS, EPI_BIAS_RELU, EPI_GELU, EPI_BIAS_GELU,
    build, gemm_epilogue_f64, round_to, decode, max_threads, set_threads,
    dtype_code, attention_f64,
)
