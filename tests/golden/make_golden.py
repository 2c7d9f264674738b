"""Writes the stored expected values under tests/golden/ by calling only the oracle.

Fixture: the M=2, N=8, K=4 debugging shape that "从零开始学习 TileLang…" §16.1
recommends starting from, with small-integer fp16 inputs (seed 1) and every
epilogue.  Products and sums of such inputs are exact, so the stored values
are exact integers.  Run from the repository root:  python tests/golden/make_golden.py
"""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
import seeded_inputs as si  # noqa: E402

M, N, K = 2, 8, 4


def main():
    A, B, bias = si.make_inputs(M, N, K, "fp16", seed=1, kind="int")
    a, b, c = si.bits(A), si.bits(B), si.bits(bias)
    lines = ["# debugging shape M=2 N=8 K=4 of the TileLang tutorial, section 16.1;",
             "# fp16 small-integer inputs from seeded_inputs.make_inputs(2, 8, 4, 'fp16', seed=1, kind='int');",
             "# expected values written by tests/golden/make_golden.py (oracle only).",
             "A " + " ".join(f"{v:g}" for v in A.float().flatten().tolist()),
             "B " + " ".join(f"{v:g}" for v in B.float().flatten().tolist()),
             "bias " + " ".join(f"{v:g}" for v in bias.float().flatten().tolist())]
    for name, epi in (("none", 0), ("relu", 1), ("bias", 2), ("bias_relu", 3)):
        ref = oracle.gemm_epilogue_f64(a, b, c if epi >= 2 else None, M, N, K, oracle.F16, epi)
        lines.append(f"C_{name} " + " ".join(f"{v:g}" for v in ref.flatten().tolist()))
    with open(os.path.join(os.path.dirname(os.path.abspath(__file__)), "debug_shape_2x8x4.txt"), "w") as f:
        f.write("\n".join(lines) + "\n")


if __name__ == "__main__":
    main()
