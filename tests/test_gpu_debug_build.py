"""The debug build (libtgemm_debug.so: -DTGEMM_DEBUG, device-side bounds and
alignment checks at every computed global access, a failed check recorded in
the status word and the access skipped).

* On every path (each tile configuration with split-K, the k-split and
  column-part tails, the decode shapes, transposed operands, unaligned
  pitches through the repack and the masked stores, the no-allocation and
  host-buffer entry points, attention full and causal with a ragged
  sequence) no check fires and the output is bit-identical to the release
  build's on the same inputs.
* A planted violation (TGEMM_DEBUG_PLANT=c_store: the checks' bound for C one
  row short) is caught: TGEMM_ERR_DEBUG_CHECK, check id 4, C's last row left
  untouched and every other row as in the release build.  Nothing faults:
  the checks skip the stores they refuse.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import gemm_epilogue_02_gb300 as tg
import seeded_inputs as si
from gpu_helpers import EPI, SENTINEL, alloc_c, c_bits, to_device_pitched

pytestmark = pytest.mark.gpu

DEBUG_CHECK = 8


@pytest.fixture(scope="module")
def libs(cuda_lib):
    rel, dbg = tg.load(), tg.load_debug()
    assert rel.tgemm_debug_last_check() == -1 and dbg.tgemm_debug_last_check() == 0
    return rel, dbg


def gemm_inputs(M, N, K, dtype, seed, kind, lda=None, ldb=None, ldc=None):
    A, B, bias = si.make_inputs(M, N, K, dtype, seed, kind, lda=lda, ldb=ldb)
    return (to_device_pitched(A, K), to_device_pitched(B, N), bias.to("cuda"), ldc or N)


def run_both(libs, fn, *args, ldc, M, N, dtype="fp16"):
    """Run the same call through the release and the debug library; return
    both C's bits and the debug library's status and check id."""
    outs = []
    for lib in libs:
        C = alloc_c(M, N, ldc, dtype)
        st = fn(lib, C, *args)
        assert st == 0, tg.tgemm_status_string(st)
        torch.cuda.synchronize()
        outs.append(c_bits(C, M, ldc))
    dbg = libs[1]
    return outs[0], outs[1], dbg.tgemm_last_device_status(), dbg.tgemm_debug_last_check()


def call_run(lib, C, A, B, bias, M, N, K, dtype, epi):
    return lib.tgemm_run(A.data_ptr(), B.data_ptr(), bias.data_ptr(), C.data_ptr(), M, N, K, A.stride(0),
                         B.stride(0), C.stride(0), 1 if dtype == "bf16" else 0, EPI[epi],
                         torch.cuda.current_stream().cuda_stream)


def assert_same_and_clean(rel, dbg, status, check, what):
    assert status == 0 and check == 0, f"{what}: status {status}, check {check}"
    assert np.array_equal(rel, dbg), f"{what}: debug build differs from the release build"


@pytest.mark.parametrize("cfg", ["256x2", "224x2", "128x2", "256x4", "256", "192", "128", "64"])
@pytest.mark.parametrize("split", ["1", "3"])
def test_every_config_without_a_failed_check(libs, monkeypatch, cfg, split):
    monkeypatch.setenv("TGEMM_FORCE_CFG", cfg)
    monkeypatch.setenv("TGEMM_SPLIT_K", split)
    M, N, K = 600, 900, 400
    A, B, bias, ldc = gemm_inputs(M, N, K, "fp16", 3, "normal")
    rel, dbg, st, chk = run_both(libs, call_run, A, B, bias, M, N, K, "fp16", "bias_relu", ldc=ldc, M=M, N=N)
    assert_same_and_clean(rel, dbg, st, chk, f"{cfg} split {split}")


@pytest.mark.parametrize("M,N,K,lda,ldb,ldc,dtype,epi", [
    (2560, 2048, 2048, None, None, None, "bf16", "bias_relu"),     # k-split tail
    (2048, 2404, 200, None, None, None, "fp16", "bias_gelu"),      # column-part tail
    (16, 2048, 4096, None, None, None, "fp16", "bias_relu"),       # split-K of every tile
    (1, 1000, 3000, None, None, None, "bf16", "relu"),             # one row
    (1000, 1003, 300, 301, 1005, 1007, "fp16", "bias_relu"),       # repack of A and B, masked stores
    (8191, 6143, 4104, None, None, None, "fp16", "bias_relu"),     # the ragged workload (dense pitches)
])
def test_paths_without_a_failed_check(libs, M, N, K, lda, ldb, ldc, dtype, epi):
    kind = "gelu" if "gelu" in epi else "normal"
    A, B, bias, ldc = gemm_inputs(M, N, K, dtype, 5, kind, lda, ldb, ldc)
    rel, dbg, st, chk = run_both(libs, call_run, A, B, bias, M, N, K, dtype, epi, ldc=ldc, M=M, N=N, dtype=dtype)
    assert_same_and_clean(rel, dbg, st, chk, f"{M}x{N}x{K}")


@pytest.mark.parametrize("ta,tb", [(1, 0), (0, 1), (1, 1)])
def test_transposed_layouts_without_a_failed_check(libs, ta, tb):
    M, N, K = 333, 700, 1000
    A, B, bias = si.make_inputs(M, N, K, "bf16", 7, "normal")
    Ad = (A.t().contiguous() if ta else A).cuda()
    Bd = (B.t().contiguous() if tb else B).cuda()
    bd = bias.cuda()

    def call(lib, C):
        return lib.tgemm_run_ex(Ad.data_ptr(), Bd.data_ptr(), bd.data_ptr(), C.data_ptr(), M, N, K, Ad.stride(0),
                                Bd.stride(0), C.stride(0), 1, EPI["bias_relu"], ta, tb,
                                torch.cuda.current_stream().cuda_stream)
    rel, dbg, st, chk = run_both(libs, call, ldc=N, M=M, N=N, dtype="bf16")
    assert_same_and_clean(rel, dbg, st, chk, f"ta={ta} tb={tb}")


def test_noalloc_and_host_entry_points_without_a_failed_check(libs):
    M, N, K = 700, 1001, 500
    A, B, bias, ldc = gemm_inputs(M, N, K, "fp16", 9, "normal", ldb=1003)
    rel, dbg, st, chk = run_both(libs, lambda lib, C: lib.tgemm_run_noalloc(
        A.data_ptr(), B.data_ptr(), bias.data_ptr(), C.data_ptr(), M, N, K, A.stride(0), B.stride(0), C.stride(0), 0,
        EPI["bias_relu"], torch.cuda.current_stream().cuda_stream), ldc=ldc, M=M, N=N)
    assert_same_and_clean(rel, dbg, st, chk, "noalloc")
    Ah, Bh, bh = A.cpu().contiguous(), B.cpu().contiguous(), bias.cpu()
    outs = []
    for lib in libs:
        Ch = torch.empty(M, N, dtype=torch.float16)
        st = lib.tgemm_run_host(Ah.data_ptr(), Bh.data_ptr(), bh.data_ptr(), Ch.data_ptr(), M, N, K, K, N, N, 0,
                                EPI["bias_relu"], None)
        assert st == 0
        torch.cuda.synchronize()
        outs.append(Ch.view(torch.int16).numpy().copy())
    assert libs[1].tgemm_last_device_status() == 0 and libs[1].tgemm_debug_last_check() == 0
    assert np.array_equal(outs[0], outs[1])


@pytest.mark.parametrize("causal", [0, 1])
def test_attention_without_a_failed_check(libs, causal):
    w = si.AttnWorkload("dbg", 2, 200, 3, 64, "fp16", bool(causal), 11)
    q, k, v = [t.cuda() for t in si.make_attention_inputs(w)]
    outs = []
    for lib in libs:
        o = torch.empty_like(q)
        st = lib.tgemm_attention_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), w.B, w.S, w.H, w.D,
                                     causal, 0, torch.cuda.current_stream().cuda_stream)
        assert st == 0
        torch.cuda.synchronize()
        outs.append(o.view(torch.int16).cpu().numpy())
    assert libs[1].tgemm_last_device_status() == 0 and libs[1].tgemm_debug_last_check() == 0
    assert np.array_equal(outs[0], outs[1])


def test_planted_violation_is_caught_and_skipped(libs, monkeypatch):
    """TGEMM_DEBUG_PLANT=c_store: the debug build's bound for C ends one row
    early, so every plain store of C's last row fails its check and is
    skipped; the release build does not read the variable."""
    monkeypatch.setenv("TGEMM_DEBUG_PLANT", "c_store")
    M, N, K, ldc = 300, 260, 128, 263           # pitch not a multiple of 8: plain (masked) stores
    A, B, bias, ldc = gemm_inputs(M, N, K, "fp16", 13, "int", ldc=ldc)
    rel, dbg, st, chk = run_both(libs, call_run, A, B, bias, M, N, K, "fp16", "bias_relu", ldc=ldc, M=M, N=N)
    assert st == DEBUG_CHECK and chk == 4, (st, chk)
    assert np.array_equal(rel[: M - 1], dbg[: M - 1])
    assert (dbg[M - 1] == SENTINEL).all()          # the refused stores were skipped
    assert not (rel[M - 1, :N] == SENTINEL).any()   # the release build wrote the row
    monkeypatch.delenv("TGEMM_DEBUG_PLANT")
    rel2, dbg2, st2, chk2 = run_both(libs, call_run, A, B, bias, M, N, K, "fp16", "bias_relu", ldc=ldc, M=M, N=N)
    assert_same_and_clean(rel2, dbg2, st2, chk2, "after the planted run")
