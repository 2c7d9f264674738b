"""Golden fixture (oracle regression on the tutorial's M=2, N=8, K=4 debugging
shape) and properties of the seeded input generator."""
import math
import os

import numpy as np
import torch

import oracle
import seeded_inputs as si

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "debug_shape_2x8x4.txt")


def read_golden():
    out = {}
    for line in open(GOLDEN):
        if line.startswith("#") or not line.strip():
            continue
        key, *vals = line.split()
        out[key] = np.array([float(v) for v in vals])
    return out


def test_golden_matches_oracle_and_inputs():
    g = read_golden()
    A, B, bias = si.make_inputs(2, 8, 4, "fp16", seed=1, kind="int")
    assert np.array_equal(A.double().flatten().numpy(), g["A"])
    assert np.array_equal(B.double().flatten().numpy(), g["B"])
    assert np.array_equal(bias.double().numpy(), g["bias"])
    for name, epi in (("none", 0), ("relu", 1), ("bias", 2), ("bias_relu", 3)):
        ref = oracle.gemm_epilogue_f64(si.bits(A), si.bits(B), si.bits(bias) if epi >= 2 else None,
                                       2, 8, 4, oracle.F16, epi)
        assert np.array_equal(ref.flatten(), g[f"C_{name}"])
    # An entry checked by hand: row 0 of A is (-2, 2, 2, 1), column 7 of B is (-2, 2, -1, -2).
    assert g["C_none"][7] == (-2) * (-2) + 2 * 2 + 2 * (-1) + 1 * (-2)


def test_inputs_deterministic_and_ordered():
    a1, b1, c1 = si.make_inputs(64, 48, 32, "bf16", seed=5)
    a2, b2, c2 = si.make_inputs(64, 48, 32, "bf16", seed=5)
    assert torch.equal(a1, a2) and torch.equal(b1, b2) and torch.equal(c1, c2)
    a3, b3, _ = si.make_inputs(64, 48, 32, "bf16", seed=6)
    assert not torch.equal(a1, a3)
    # The bias is drawn last: A and B do not depend on with_bias.
    a4, b4, c4 = si.make_inputs(64, 48, 32, "bf16", seed=5, with_bias=False)
    assert torch.equal(a1, a4) and torch.equal(b1, b4) and c4 is None


def test_inputs_distribution_and_padding():
    K = 1024
    A, B, bias = si.make_inputs(512, 256, K, "fp16", seed=3, ldb=264)
    assert A.shape == (512, K) and B.shape == (K, 264) and bias.shape == (256,)
    assert torch.isnan(B[:, 256:]).all() and not torch.isnan(B[:, :256]).any()
    assert abs(A.float().std().item() - 1.0) < 0.02
    assert abs(B[:, :256].float().std().item() * math.sqrt(K) - 1.0) < 0.02
    assert abs(bias.float().std().item() - 0.1) < 0.02
    Ai, Bi, bi = si.make_inputs(64, 64, 64, "fp16", seed=1, kind="int")
    for t in (Ai, Bi, bi):
        vals = set(t.float().unique().tolist())
        assert vals <= {-2.0, -1.0, 0.0, 1.0, 2.0}


def test_workload_table():
    w = si.WORKLOADS
    assert (w["c2"].M, w["c2"].N, w["c2"].K, w["c2"].dtype) == (8192, 8192, 8192, "bf16")
    assert (w["c3"].M, w["c3"].N, w["c3"].K) == (128, 28672, 8192)
    assert (w["c4"].M, w["c4"].N, w["c4"].K) == (8191, 6143, 4104)
    assert w["c0"].epilogue == "relu" and w["c1"].epilogue == "bias_relu"
    assert w["c1"].flops == 2 * 4096 ** 3
