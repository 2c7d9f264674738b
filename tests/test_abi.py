"""The C-ABI library loads and exports every function include/tgemm.h declares,
and the host-side argument validation returns the documented status codes
before touching any device (runs without a GPU)."""
import ctypes
import os
import re

import pytest
import torch

import gemm_epilogue_02_gb300 as tg

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "tgemm.h")

OK, INVALID, ALIGN, UNSUPPORTED, ALIAS = 0, 1, 2, 3, 4


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*[\w\s\*]*?\b(tgemm_\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_abi():
    names = declared_functions()
    assert set(names) == set(tg.EXPORTED), names


def test_library_exports_every_declared_symbol():
    lib = tg.load()
    for name in declared_functions():
        assert hasattr(lib, name), name
    assert tg.tgemm_version() == 0x000100


def test_debug_build_exports_the_same_abi():
    """libtgemm_debug.so (the device-side checks compiled in) has the same
    C ABI; the release build says it compiles no checks."""
    dbg = tg.load_debug()
    for name in declared_functions():
        assert hasattr(dbg, name), name
    assert dbg.tgemm_version() == tg.tgemm_version()
    assert tg.load().tgemm_debug_last_check() == -1   # release build: no checks, no device access
    assert dbg.tgemm_status_string(8).decode().startswith("TGEMM_ERR_DEBUG_CHECK")


def test_header_documents_every_environment_variable_the_library_reads():
    src_dir = os.path.join(ROOT, "gemm_epilogue_02_gb300", "csrc")
    names = set()
    for f in os.listdir(src_dir):
        if f.endswith((".cu", ".cuh")):
            names |= set(re.findall(r'getenv\("(\w+)"\)', open(os.path.join(src_dir, f)).read()))
    assert names, "no environment variables found"
    header = open(HEADER).read()
    missing = sorted(n for n in names if n not in header)
    assert not missing, missing


def test_status_strings():
    for code, name in tg.STATUS.items():
        assert tg.tgemm_status_string(code).startswith(name)
    assert "UNKNOWN" in tg.tgemm_status_string(99)


# Fake, 16-byte-aligned, disjoint addresses: validation reads addresses only.
A, B, BIAS, C = 0x100000, 0x200000, 0x300000, 0x400000


def call(**kw):
    args = dict(A=A, B=B, bias=BIAS, C=C, M=64, N=64, K=64, lda=64, ldb=64, ldc=64, dtype=0, epi=3)
    args.update(kw)
    return tg.tgemm_run(args["A"], args["B"], args["bias"], args["C"], args["M"], args["N"],
                        args["K"], args["lda"], args["ldb"], args["ldc"], args["dtype"], args["epi"], 0)


@pytest.mark.parametrize("kw,code", [
    (dict(M=-1), INVALID), (dict(N=-1), INVALID), (dict(K=-1), INVALID),
    (dict(lda=63), INVALID), (dict(ldb=63), INVALID), (dict(ldc=63), INVALID),
    (dict(dtype=2), INVALID), (dict(epi=6), INVALID), (dict(epi=-1), INVALID),
    (dict(A=0), INVALID), (dict(B=0), INVALID), (dict(C=0), INVALID),
    (dict(bias=0, epi=2), INVALID), (dict(bias=0, epi=3), INVALID), (dict(bias=0, epi=5), INVALID),
    (dict(M=2 ** 31), INVALID),
    (dict(A=A + 2), ALIGN), (dict(B=B + 8), ALIGN), (dict(C=C + 2), ALIGN), (dict(bias=BIAS + 4), ALIGN),
    (dict(C=A + 64), ALIAS), (dict(C=B), ALIAS), (dict(C=BIAS - 64 * 2 + 16), ALIAS),
])
def test_invalid_arguments_rejected_before_any_launch(kw, code):
    assert call(**kw) == code


def test_pointer_rules_that_depend_on_the_problem():
    # Empty problems are valid with NULL pointers (nothing is read or written)...
    assert call(A=0, B=0, bias=0, C=0, M=0) in (OK, UNSUPPORTED)
    # ...K == 0 does not read A or B, and NONE/RELU do not read the bias.
    assert call(A=0, B=0, K=0, lda=0, ldb=64) in (OK, UNSUPPORTED)
    assert call(bias=0, epi=1) in (OK, UNSUPPORTED)
    assert call(bias=BIAS + 2, epi=0) in (OK, UNSUPPORTED)
    # A pitch wider than the width, unaligned or not, is accepted.
    assert call(lda=67, ldb=65, ldc=99) in (OK, UNSUPPORTED)


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-GPU path")
def test_valid_call_without_gpu_reports_unsupported_device():
    assert call() == UNSUPPORTED
    assert tg.tgemm_last_device_status() == UNSUPPORTED
    buf = (ctypes.c_uint16 * 64)()
    p = ctypes.addressof(buf)
    assert tg.tgemm_run_host(p, p + 32, 0, p + 64, 4, 4, 4, 4, 4, 4, 0, 1, 0) in (UNSUPPORTED, ALIAS)


def call_ex(ta, tb, **kw):
    args = dict(A=A, B=B, bias=BIAS, C=C, M=64, N=32, K=48, lda=64, ldb=48, ldc=32)
    args.update(kw)
    return tg.tgemm_run_ex(args["A"], args["B"], args["bias"], args["C"], args["M"], args["N"], args["K"],
                           args["lda"], args["ldb"], args["ldc"], 0, 3, ta, tb, 0)


def test_transposed_layout_validation():
    # Stored [K, M] A needs lda >= M; stored [N, K] B needs ldb >= K.
    assert call_ex(1, 1, lda=63) == INVALID
    assert call_ex(1, 1, ldb=47) == INVALID
    assert call_ex(2, 0) == INVALID
    assert call_ex(0, -1, lda=48, ldb=32) == INVALID
    assert call_ex(1, 1) in (OK, UNSUPPORTED)
    assert call_ex(0, 0, lda=48, ldb=32) in (OK, UNSUPPORTED)


def call_attn(**kw):
    args = dict(Q=0x100000, K=0x200000, V=0x300000, O=0x400000, B=2, S=128, H=2, D=64, causal=0, dtype=0)
    args.update(kw)
    return tg.tgemm_attention_fwd(args["Q"], args["K"], args["V"], args["O"], args["B"], args["S"], args["H"],
                                  args["D"], args["causal"], args["dtype"], 0)


@pytest.mark.parametrize("kw,code", [
    (dict(D=128), INVALID), (dict(D=32), INVALID), (dict(B=-1), INVALID), (dict(S=-1), INVALID),
    (dict(H=-1), INVALID), (dict(causal=2), INVALID), (dict(dtype=2), INVALID), (dict(H=70000), INVALID),
    (dict(Q=0), INVALID), (dict(O=0), INVALID), (dict(K=0x200008), ALIGN), (dict(O=0x400002), ALIGN),
    (dict(O=0x300000 + 1024), ALIAS), (dict(O=0x100000), ALIAS),
])
def test_attention_arguments_rejected_before_any_launch(kw, code):
    assert call_attn(**kw) == code


def test_attention_empty_problems_and_valid_call():
    assert call_attn(B=0, Q=0, K=0, V=0, O=0) == OK
    assert call_attn(S=0) == OK
    assert call_attn() in (OK, UNSUPPORTED, INVALID)   # no GPU here (or host pointers on one)
