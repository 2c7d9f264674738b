"""GPU parity of the fused GEMM epilogue against the fp64 CPU oracle, through
the C ABI.  Bit-exact on small-integer inputs; otherwise relative Frobenius
<= 2e-3 and |err| <= 1e-2 + 1e-2 |ref| per element (against unrounded fp64).

Coverage: the five workloads of the method's evaluation at their full sizes
(sampled rows, every column), the integer-exact variant, a tiny / odd shape
sweep (the tutorial's start-small advice and edge-case list), every epilogue x
dtype, each tile configuration, wider pitches with guarded padding, K = 0 and
empty problems, repeat-run determinism, the host-buffer entry point, and the
device pointer check."""
from __future__ import annotations

import os

import numpy as np
import pytest
import torch

import oracle
import seeded_inputs as si
from gpu_helpers import (EPI, assert_bit_exact, assert_close, assert_pad_untouched, c_bits,
                         check_epilogue, magnitude, oracle_ref, run_tgemm, run_tgemm_layout)

pytestmark = pytest.mark.gpu


def sample_rows(M, n=48, seed=0):
    """Fixed edge rows, n random rows, and one row of every 128-row block (a
    different offset in each), so that every output tile has a checked row."""
    rng = np.random.default_rng(seed)
    fixed = [0, 1, 127, 128, 129, M // 2, M - 129, M - 128, M - 2, M - 1]
    rows = set(r for r in fixed if 0 <= r < M)
    rows |= set(rng.choice(M, size=min(n, M), replace=False).tolist())
    rows |= {min(M - 1, b * 128 + int(rng.integers(128))) for b in range((M + 127) // 128)}
    return sorted(rows)


@pytest.fixture(autouse=True)
def _lib(cuda_lib):
    yield cuda_lib


# ------------------------------------------------------------------ workloads
@pytest.mark.parametrize("name", ["c0", "c1", "c2", "c3", "c4", "c4p", "c5", "d16"])
def test_workload_full_size(cuda_lib, name):
    w = si.WORKLOADS[name]
    inputs, got = run_tgemm(cuda_lib, w.M, w.N, w.K, w.dtype, w.epilogue, w.seed, w.kind,
                            w.lda, w.ldb, w.ldc)
    assert_pad_untouched(got, w.N, name)
    rows = list(range(w.M)) if w.M * w.N * w.K <= 2 ** 26 else sample_rows(w.M, seed=w.seed)
    check_epilogue(got[rows, : w.N], inputs, w.M, w.N, w.K, w.dtype, w.epilogue, name, rows=rows)


def test_gelu_workload_page_check(cuda_lib):
    """The GELU workload's own acceptance test on its page (relative Frobenius
    against the unfused GELU(a@b + bias) below 3e-2), on top of the oracle bounds."""
    w = si.WORKLOADS["c5"]
    inputs, got = run_tgemm(cuda_lib, w.M, w.N, w.K, w.dtype, w.epilogue, w.seed, w.kind)
    rows = sample_rows(w.M, n=32, seed=9)
    A, B, bias = inputs
    pre = (A[rows].double() @ B.double()) + bias.double()
    ref = torch.nn.functional.gelu(pre, approximate="tanh").numpy()
    out = torch.from_numpy(got[rows].view(np.int16)).view(torch.float16).double().numpy()
    assert np.linalg.norm(out - ref) / np.linalg.norm(ref) < 3e-2


def test_integer_exact_4096(cuda_lib):
    w = si.WORKLOADS["c1x"]
    for epi in ("bias_relu", "none"):
        inputs, got = run_tgemm(cuda_lib, w.M, w.N, w.K, w.dtype, epi, w.seed, "int")
        rows = sample_rows(w.M, n=40, seed=11)
        ref = oracle_ref(inputs, w.M, w.N, w.K, w.dtype, epi, rows=rows)
        assert_bit_exact(got[rows], ref, w.dtype, f"c1x {epi}")


# ------------------------------------------------------------------ shapes
SWEEP = [1, 2, 7, 8, 9, 63, 64, 65, 127, 128, 129, 255, 257]


def sweep_cases(n=120):
    rng = np.random.default_rng(2024)
    cases = {(2, 8, 4), (1, 1, 1), (257, 257, 257), (1, 257, 257), (257, 1, 257), (257, 257, 1)}
    while len(cases) < n:
        cases.add(tuple(int(rng.choice(SWEEP)) for _ in range(3)))
    return sorted(cases)


@pytest.mark.parametrize("M,N,K", sweep_cases())
def test_small_and_odd_shapes(cuda_lib, M, N, K):
    idx = M * 7 + N * 3 + K
    epi = ["none", "relu", "bias", "bias_relu"][idx % 4]
    dtype = ["fp16", "bf16"][(idx // 4) % 2]
    inputs, got = run_tgemm(cuda_lib, M, N, K, dtype, epi, seed=idx, kind="int")
    ref = oracle_ref(inputs, M, N, K, dtype, epi)
    assert_bit_exact(got, ref, dtype, f"{M}x{N}x{K} {epi} {dtype}")
    inputs, got = run_tgemm(cuda_lib, M, N, K, dtype, epi, seed=idx)
    ref = oracle_ref(inputs, M, N, K, dtype, epi)
    assert_close(got, ref, dtype, f"{M}x{N}x{K} {epi} {dtype}", magnitude(inputs, N, K), K)


CONFIGS = ["64", "128", "192", "256", "128x2", "224x2", "256x2", "256x4"]


@pytest.mark.parametrize("bn", CONFIGS)
@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
@pytest.mark.parametrize("epi", ["none", "relu", "bias", "bias_relu", "gelu", "bias_gelu"])
def test_each_tile_config_epilogue_dtype(cuda_lib, monkeypatch, bn, dtype, epi):
    """Several tiles in both directions, a ragged tail on M, N and K, and a k
    loop longer than the ring (so stages wrap) for each kernel configuration
    (C tile width, and 1 CTA or a CTA pair per tile); bit-exact on integer
    inputs for the piecewise-linear epilogues."""
    monkeypatch.setenv("TGEMM_FORCE_CFG", bn)
    M, N, K = 333, 700, 1000
    if "gelu" not in epi:
        inputs, got = run_tgemm(cuda_lib, M, N, K, dtype, epi, seed=5, kind="int")
        assert_bit_exact(got, oracle_ref(inputs, M, N, K, dtype, epi), dtype, f"int bn={bn}")
    inputs, got = run_tgemm(cuda_lib, M, N, K, dtype, epi, seed=6, kind="gelu" if "gelu" in epi else "normal")
    check_epilogue(got, inputs, M, N, K, dtype, epi, f"bn={bn}")


@pytest.mark.parametrize("bn", CONFIGS)
def test_persistent_loop_many_tiles(cuda_lib, monkeypatch, bn):
    """More tiles than SMs: each CTA runs several tiles and both TMEM buffers."""
    monkeypatch.setenv("TGEMM_FORCE_CFG", bn)
    M, N, K = 2560, 3072, 192
    inputs, got = run_tgemm(cuda_lib, M, N, K, "bf16", "bias_relu", seed=9, kind="int")
    assert_bit_exact(got, oracle_ref(inputs, M, N, K, "bf16", "bias_relu"), "bf16", f"bn={bn}")


@pytest.mark.parametrize("lda,ldb,ldc", [(72, 136, 136), (75, 133, 131), (64, 129, 128),
                                         (80, 128, 130)])
def test_pitches_and_guarded_padding(cuda_lib, lda, ldb, ldc):
    """Wider row pitches, aligned (TMA paths) and unaligned (repack / masked-store
    paths); C's padding columns must keep their sentinel."""
    M, N, K = 200, 128, 64
    inputs, got = run_tgemm(cuda_lib, M, N, K, "fp16", "bias_relu", seed=3, kind="int",
                            lda=lda, ldb=ldb, ldc=ldc)
    assert_pad_untouched(got, N, "pad")
    assert_bit_exact(got[:, :N], oracle_ref(inputs, M, N, K, "fp16", "bias_relu"), "fp16", "pitch")


@pytest.mark.parametrize("cfg", CONFIGS)
def test_pair_rows_beyond_m(cuda_lib, monkeypatch, cfg):
    """M that leaves the second CTA of a pair without rows, and tiny M / N."""
    monkeypatch.setenv("TGEMM_FORCE_CFG", cfg)
    for (M, N, K) in [(128, 520, 300), (100, 64, 64), (300, 100, 130), (1, 1, 1)]:
        inputs, got = run_tgemm(cuda_lib, M, N, K, "fp16", "bias_relu", seed=M + N, kind="int")
        assert_bit_exact(got, oracle_ref(inputs, M, N, K, "fp16", "bias_relu"), "fp16", f"{cfg} {M}x{N}x{K}")


# ------------------------------------------------------------------ split-K
@pytest.mark.parametrize("cfg", CONFIGS)
@pytest.mark.parametrize("split", ["2", "3", "5"])
def test_split_k_forced(cuda_lib, monkeypatch, cfg, split):
    """k ranges of a tile computed by different CTAs, fp32 partials summed by the
    last arriving warp of each region, then the epilogue (bit-exact on integers)."""
    monkeypatch.setenv("TGEMM_FORCE_CFG", cfg)
    monkeypatch.setenv("TGEMM_SPLIT_K", split)
    M, N, K = 333, 700, 1000
    inputs, got = run_tgemm(cuda_lib, M, N, K, "fp16", "bias_relu", seed=41, kind="int")
    assert_bit_exact(got, oracle_ref(inputs, M, N, K, "fp16", "bias_relu"), "fp16", f"{cfg} split={split}")
    inputs, got = run_tgemm(cuda_lib, M, N, K, "bf16", "bias_gelu", seed=42, kind="gelu")
    check_epilogue(got, inputs, M, N, K, "bf16", "bias_gelu", f"{cfg} split={split}")


@pytest.mark.parametrize("M", [1, 16, 64, 128])
def test_decode_shapes_split_automatically(cuda_lib, M):
    """Few-row (decode-like) shapes: too few tiles for the GPU, so the k loop is
    split; the result must not depend on the split (deterministic order)."""
    N, K = 4096, 8192
    inputs, got = run_tgemm(cuda_lib, M, N, K, "fp16", "bias_relu", seed=43 + M)
    check_epilogue(got, inputs, M, N, K, "fp16", "bias_relu", f"M={M}")
    _, again = run_tgemm(cuda_lib, M, N, K, "fp16", "bias_relu", seed=43 + M)
    assert np.array_equal(got, again)


# ------------------------------------------------------------------ narrow tail
# (cfg, M, N, K, parts expected on a 152-SM GB300): the last, partial wave's
# tiles are cut into column parts that run as narrower MMAs.
NARROW_CASES = [
    ("256x2", 2048, 2560, 320, 2),     # 8 x 10 = 80 pair tiles: 4 cut in two
    ("256x4", 2048, 2560, 320, 2),     # 4 x 10 = 40 shared-B tiles on 38 clusters: 2 cut in two
    ("256x2", 2048, 2404, 200, 2),     # last column block has 100 columns: one part lies past N
    ("256", 2560, 2048, 256, 4),       # 20 x 8 = 160 tiles on 152 SMs: 8 cut in four (64 columns)
    ("128", 2560, 1088, 130, 2),       # 20 x 9 = 180 tiles: 28 cut in two
]


@pytest.mark.parametrize("cfg,M,N,K,parts", NARROW_CASES)
def test_narrow_tail(cuda_lib, monkeypatch, cfg, M, N, K, parts):
    """Column parts of the last wave's tiles: exact on integers, within the
    bound on normal inputs, and the same bits as whole tiles (each output is
    still one k loop in the same order)."""
    monkeypatch.setenv("TGEMM_FORCE_CFG", cfg)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    plan = cuda_lib.tgemm_plan(M, N, K, sms)
    assert plan["narrow_parts"] == parts and plan["narrow_first"] < plan["tiles"], plan
    inputs, got = run_tgemm(cuda_lib, M, N, K, "fp16", "bias_relu", seed=51, kind="int")
    assert_bit_exact(got, oracle_ref(inputs, M, N, K, "fp16", "bias_relu"), "fp16", f"{cfg} narrow int")
    inputs, got = run_tgemm(cuda_lib, M, N, K, "bf16", "bias_gelu", seed=52, kind="gelu")
    rows = sample_rows(M, n=64, seed=52)
    check_epilogue(got[rows], inputs, M, N, K, "bf16", "bias_gelu", f"{cfg} narrow gelu", rows=rows)
    monkeypatch.setenv("TGEMM_TAIL_SPLIT", "0")
    assert cuda_lib.tgemm_plan(M, N, K, sms)["narrow_parts"] == 1
    _, whole = run_tgemm(cuda_lib, M, N, K, "bf16", "bias_gelu", seed=52, kind="gelu")
    assert np.array_equal(got, whole), "narrow parts changed the result bits"


# ------------------------------------------------------------------ k-split tail
# (cfg, M, N, K, ranges expected on a 152-SM GB300): the last, partial wave's
# tiles have their k loops cut into ranges that run first; the last range to
# finish adds the fp32 partials in range order before the epilogue.
TAIL_SPLIT_CASES = [
    ("256x2", 2048, 2560, 4096, 4),    # 8 x 10 = 80 pair tiles: 4 left, 64 k-blocks in 4 ranges
    ("256x4", 2048, 2560, 4096, 4),    # 4 x 10 = 40 shared-B tiles: 2 left, 64 k-blocks in 4 ranges
    ("256x4", 2560, 2404, 2000, 2),    # 5 x 10 = 50 tiles: 12 left in 2 ranges, ragged k-block and columns
    ("224x2", 2048, 2240, 3072, 3),    # 80 tiles of 224 columns: 4 left, 48 k-blocks in 3 ranges
    ("256x2", 2048, 2404, 2000, 2),    # ragged k-block and a last column block of 100 columns
    ("256", 2560, 2048, 4096, 4),      # 160 single-CTA tiles: 8 left over
    ("128", 2560, 1088, 2070, 2),      # 180 tiles: 28 left; 33 k-blocks as 17 + 16
]


@pytest.mark.parametrize("cfg,M,N,K,ranges", TAIL_SPLIT_CASES)
def test_k_split_tail(cuda_lib, monkeypatch, cfg, M, N, K, ranges):
    """k ranges of the last wave's tiles: exact on integers, within the bound
    on normal inputs, the same bits on every run, and within the bound of the
    whole-tile result (only the summation order of those tiles changes)."""
    monkeypatch.setenv("TGEMM_FORCE_CFG", cfg)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    plan = cuda_lib.tgemm_plan(M, N, K, sms)
    if sms == 152:
        assert plan["split_k"] == ranges and plan["split_first"] == plan["tiles"] - plan["tiles"] % plan["groups"], plan
    # One row of every 128-row block (every column is checked): each tile is sampled.
    rows = sorted(set(sample_rows(M, n=32, seed=72)) | set(range(5, M, 128)) | set(range(M - 8, M)))
    inputs, got = run_tgemm(cuda_lib, M, N, K, "fp16", "bias_relu", seed=71, kind="int")
    ref = oracle_ref(inputs, M, N, K, "fp16", "bias_relu", rows=rows)
    assert_bit_exact(got[rows], ref, "fp16", f"{cfg} k tail int")
    inputs, got = run_tgemm(cuda_lib, M, N, K, "bf16", "bias_gelu", seed=72, kind="gelu")
    check_epilogue(got[rows], inputs, M, N, K, "bf16", "bias_gelu", f"{cfg} k tail gelu", rows=rows)
    _, again = run_tgemm(cuda_lib, M, N, K, "bf16", "bias_gelu", seed=72, kind="gelu")
    assert np.array_equal(got, again), "k-split tail is not deterministic"
    monkeypatch.setenv("TGEMM_TAIL_SPLIT", "0")
    assert cuda_lib.tgemm_plan(M, N, K, sms)["split_k"] == 1
    _, whole = run_tgemm(cuda_lib, M, N, K, "bf16", "bias_gelu", seed=72, kind="gelu")
    check_epilogue(whole[rows], inputs, M, N, K, "bf16", "bias_gelu", f"{cfg} whole tiles gelu", rows=rows)


@pytest.mark.parametrize("cfg", ["256x4", "256x2", "128x2", "256", "192", "128", "64"])
@pytest.mark.parametrize("M,N,K,ldb", [(700, 1024, 300, None),     # N a multiple of 64: one 3-D box per k-block
                                       (700, 1000, 300, 1024),     # last chunk past N inside the pitch
                                       (700, 1000, 300, None)])    # ... outside it: 2-D copies
def test_b_sub_tiles_in_one_copy(cuda_lib, monkeypatch, cfg, M, N, K, ldb):
    """B [K, N] loaded as one 3-D box per k-block (all 64-column sub-tiles of a
    CTA) gives the same bits as one 2-D copy per sub-tile, and exact integers."""
    monkeypatch.setenv("TGEMM_FORCE_CFG", cfg)
    inputs, got = run_tgemm(cuda_lib, M, N, K, "fp16", "bias_relu", seed=61, kind="int", ldb=ldb)
    assert_bit_exact(got[:, :N], oracle_ref(inputs, M, N, K, "fp16", "bias_relu"), "fp16", f"{cfg} b3d")
    monkeypatch.setenv("TGEMM_NO_B3D", "1")
    _, two_d = run_tgemm(cuda_lib, M, N, K, "fp16", "bias_relu", seed=61, kind="int", ldb=ldb)
    assert np.array_equal(got, two_d)
    inputs, got = run_tgemm(cuda_lib, M, N, K, "bf16", "bias_gelu", seed=62, kind="gelu", ldb=ldb)
    monkeypatch.delenv("TGEMM_NO_B3D")
    _, three_d = run_tgemm(cuda_lib, M, N, K, "bf16", "bias_gelu", seed=62, kind="gelu", ldb=ldb)
    assert np.array_equal(got, three_d)
    check_epilogue(three_d[:, :N], inputs, M, N, K, "bf16", "bias_gelu", f"{cfg} b3d gelu")


@pytest.mark.parametrize("ta,tb", [(0, 1), (1, 0)])
def test_narrow_tail_transposed(cuda_lib, monkeypatch, ta, tb):
    """Narrow parts with B stored [N, K] (the whole n box is loaded, the MMA
    reads its first part) and with A stored [K, M]."""
    monkeypatch.setenv("TGEMM_FORCE_CFG", "256x2")
    M, N, K = 2048, 2404, 200
    inputs, got = run_tgemm_layout(cuda_lib, M, N, K, "fp16", "bias_relu", seed=53, kind="int",
                                   transpose_a=bool(ta), transpose_b=bool(tb))
    assert_bit_exact(got, oracle_ref(inputs, M, N, K, "fp16", "bias_relu"), "fp16", f"narrow ta={ta} tb={tb}")


# ------------------------------------------------------------------ layouts
@pytest.mark.parametrize("ta,tb", [(0, 1), (1, 0), (1, 1)])
@pytest.mark.parametrize("cfg", CONFIGS)
def test_transposed_operands(cuda_lib, monkeypatch, cfg, ta, tb):
    """A stored [K, M] and/or B stored [N, K] (the T.gemm transpose options,
    the nn.Linear weight layout): ragged M / N / K, every tile configuration."""
    monkeypatch.setenv("TGEMM_FORCE_CFG", cfg)
    M, N, K = 333, 700, 1000
    inputs, got = run_tgemm_layout(cuda_lib, M, N, K, "bf16", "bias_relu", seed=31, kind="int",
                                   transpose_a=bool(ta), transpose_b=bool(tb))
    assert_bit_exact(got, oracle_ref(inputs, M, N, K, "bf16", "bias_relu"), "bf16", f"{cfg} ta={ta} tb={tb}")
    inputs, got = run_tgemm_layout(cuda_lib, M, N, K, "fp16", "bias_gelu", seed=32, kind="gelu",
                                   transpose_a=bool(ta), transpose_b=bool(tb))
    check_epilogue(got, inputs, M, N, K, "fp16", "bias_gelu", f"{cfg} ta={ta} tb={tb}")


@pytest.mark.parametrize("ta,tb,pad_a,pad_b", [(1, 1, 3, 5), (0, 1, 0, 1), (1, 0, 7, 0)])
def test_transposed_operands_unaligned_pitch(cuda_lib, ta, tb, pad_a, pad_b):
    """Transposed storage whose pitch is not a multiple of 8 goes through the repack."""
    M, N, K = 257, 300, 129
    inputs, got = run_tgemm_layout(cuda_lib, M, N, K, "fp16", "bias", seed=33, kind="int",
                                   transpose_a=bool(ta), transpose_b=bool(tb), pad_a=pad_a, pad_b=pad_b)
    assert_bit_exact(got, oracle_ref(inputs, M, N, K, "fp16", "bias"), "fp16", "pitch")


def test_linear_layout_4096(cuda_lib):
    """The 4096^3 workload with B in the [out_features, in_features] layout."""
    w = si.WORKLOADS["c1"]
    inputs, got = run_tgemm_layout(cuda_lib, w.M, w.N, w.K, w.dtype, w.epilogue, w.seed,
                                   transpose_b=True)
    rows = sample_rows(w.M, n=16, seed=3)
    check_epilogue(got[rows], inputs, w.M, w.N, w.K, w.dtype, w.epilogue, "c1 B^T", rows=rows)


# ------------------------------------------------------------------ degenerate
@pytest.mark.parametrize("epi", ["none", "relu", "bias", "bias_relu", "gelu", "bias_gelu"])
def test_k_zero_writes_epilogue_of_bias(cuda_lib, epi):
    M, N = 70, 90
    inputs, got = run_tgemm(cuda_lib, M, N, 0, "bf16", epi, seed=4, kind="gelu" if "gelu" in epi else "normal")
    if "gelu" in epi:
        check_epilogue(got, inputs, M, N, 0, "bf16", epi, "K=0")
    else:
        assert_bit_exact(got, oracle_ref(inputs, M, N, 0, "bf16", epi), "bf16", "K=0")


def test_empty_problems_are_noops(cuda_lib):
    for (M, N) in [(0, 64), (64, 0), (0, 0)]:
        C = torch.full((max(M, 1), max(N, 1)), 7.0, dtype=torch.float16, device="cuda")
        A = torch.ones((max(M, 1), 64), dtype=torch.float16, device="cuda")
        B = torch.ones((64, max(N, 1)), dtype=torch.float16, device="cuda")
        st = cuda_lib.tgemm_run(A.data_ptr(), B.data_ptr(), 0, C.data_ptr(), M, N, 64, 64,
                                max(N, 1), max(N, 1), 0, 1, 0)
        torch.cuda.synchronize()
        assert st == 0 and (C == 7.0).all()


# ------------------------------------------------------------------ invariants
def test_relu_equals_max_of_none_bit_exact(cuda_lib):
    M, N, K = 512, 768, 320
    _, none = run_tgemm(cuda_lib, M, N, K, "bf16", "none", seed=8)
    _, relu = run_tgemm(cuda_lib, M, N, K, "bf16", "relu", seed=8)
    v = torch.from_numpy(none.view(np.int16)).view(torch.bfloat16).float()
    want = torch.where(v > 0, v, torch.zeros_like(v)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(relu, want)
    assert not (relu == 0x8000).any()


def test_repeat_runs_are_deterministic(cuda_lib):
    M, N, K = 1024, 1536, 2048
    _, first = run_tgemm(cuda_lib, M, N, K, "fp16", "bias_relu", seed=12)
    for _ in range(5):
        _, again = run_tgemm(cuda_lib, M, N, K, "fp16", "bias_relu", seed=12)
        assert np.array_equal(first, again)


# ------------------------------------------------------------------ entry points
def test_host_entry_point_matches_device_entry_point(cuda_lib):
    M, N, K = 777, 1000, 520
    (A, B, bias), dev = run_tgemm(cuda_lib, M, N, K, "fp16", "bias_relu", seed=21)
    Ah, Bh, bh = A.pin_memory(), B.pin_memory(), bias.pin_memory()
    Ch = torch.full((M, N + 8), float("nan"), dtype=torch.float16).pin_memory()
    Cv = Ch[:, :N]
    cuda_lib.run_host(Ah, Bh, bh, Cv, "bias_relu")
    torch.cuda.synchronize()
    got = Ch.view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got[:, :N], dev)
    assert np.isnan(Ch[:, N:].float().numpy()).all()


@pytest.mark.parametrize("M,N,K,lda,ldb,ldc", [
    (4096, 4096, 1024, 1027, 4096, 4100),     # chunks of rows of A / C, unaligned host pitches
    (128, 16384, 8192, 8192, 16389, 16384),   # B dominates: one chunk, unaligned B pitch
])
def test_host_entry_point_pipelined_chunks(cuda_lib, M, N, K, lda, ldb, ldc):
    """The host path splits large problems into chunks whose copies and GEMMs
    overlap on separate streams.  Chunks are separate GEMMs whose k loops may be
    split differently from one whole-problem call, so the two agree within twice
    the derived error bound rather than bit for bit; both match the oracle."""
    A, B, bias = si.make_inputs(M, N, K, "fp16", seed=23, lda=lda if lda != K else None,
                                ldb=ldb if ldb != N else None)
    dev = torch.empty((M, N), dtype=torch.float16, device="cuda")
    cuda_lib.run(A.cuda()[:, :K], B.cuda()[:, :N], bias.cuda(), dev, "bias_relu")
    Ah, Bh, bh = A.pin_memory(), B.pin_memory(), bias.pin_memory()
    Ch = torch.full((M, ldc), float("nan"), dtype=torch.float16).pin_memory()
    cuda_lib.run_host(Ah[:, :K], Bh[:, :N], bh, Ch[:, :N], "bias_relu")
    torch.cuda.synchronize()
    got = Ch.view(torch.int16).numpy().view(np.uint16)
    devb = dev.cpu().view(torch.int16).numpy().view(np.uint16)
    if ldc > N:
        assert np.isnan(Ch[:, N:].float().numpy()).all()
    rows = sample_rows(M, n=8, seed=5)
    ref = oracle_ref((A, B, bias), M, N, K, "fp16", "bias_relu", rows=rows)
    mag = magnitude((A, B, bias), N, K, rows)
    assert_close(got[rows, :N], ref, "fp16", "host path", mag, K)
    assert_close(devb[rows], ref, "fp16", "device path", mag, K)
    gamma = 2.0 * (K + 2) * 2.0 ** -24
    bound = 2 * (2.0 ** -11 * np.abs(ref) + (1 + 2.0 ** -11) * gamma * mag + 2.0 ** -25)
    diff = np.abs(got[rows, :N].view(np.float16).astype(np.float64) - devb[rows].view(np.float16).astype(np.float64))
    assert (diff <= bound).all()


def test_host_memory_passed_to_device_entry_point_is_rejected(cuda_lib):
    A = torch.ones((64, 64), dtype=torch.float16)
    Cd = torch.empty((64, 64), dtype=torch.float16, device="cuda")
    st = cuda_lib.tgemm_run(A.data_ptr(), A.data_ptr() + 64 * 64 * 2 * 4, 0, Cd.data_ptr(),
                            64, 64, 64, 64, 64, 64, 0, 1, 0)
    assert st == 1


def test_no_kernel_timed_out(cuda_lib):
    assert cuda_lib.tgemm_last_device_status() == 0
