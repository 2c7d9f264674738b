"""Failure path of the fused GEMM kernel on the GPU: a bounded wait that runs
out.  With TGEMM_TEST_STALL=1 the kernel announces 16 bytes more for its first
operand slot than its copies deliver, so that slot never completes; every wait
in the kernel is bounded (2 s), so the kernel records TGEMM_ERR_TIMEOUT in the
device status word, lets its copies land, frees its TMEM and returns.  The
test reads that status on the host and then checks that the context is still
usable: the next call (without the stall) is bit-exact and reports no error.
Nothing here faults, traps or hangs the GPU."""
from __future__ import annotations

import time

import pytest
import torch

from gpu_helpers import assert_bit_exact, oracle_ref, run_tgemm

pytestmark = pytest.mark.gpu

TIMEOUT = 6   # TGEMM_ERR_TIMEOUT


@pytest.mark.parametrize("cfg", ["256x4", "256x2", "128"])
def test_operand_wait_runs_out_and_context_stays_usable(cuda_lib, monkeypatch, cfg):
    monkeypatch.setenv("TGEMM_FORCE_CFG", cfg)
    M, N, K = 512, 512, 512
    assert cuda_lib.tgemm_last_device_status() == 0
    monkeypatch.setenv("TGEMM_TEST_STALL", "1")
    t0 = time.monotonic()
    run_tgemm(cuda_lib, M, N, K, "fp16", "bias_relu", seed=3, kind="int")   # synchronizes
    waited = time.monotonic() - t0
    assert cuda_lib.tgemm_last_device_status() == TIMEOUT
    assert 1.5 < waited < 30.0, waited
    # The status word was cleared by the read; the next launch runs normally.
    monkeypatch.delenv("TGEMM_TEST_STALL")
    inputs, got = run_tgemm(cuda_lib, M, N, K, "fp16", "bias_relu", seed=3, kind="int")
    assert_bit_exact(got, oracle_ref(inputs, M, N, K, "fp16", "bias_relu"), "fp16", f"after stall cfg={cfg}")
    assert cuda_lib.tgemm_last_device_status() == 0
    torch.cuda.synchronize()
