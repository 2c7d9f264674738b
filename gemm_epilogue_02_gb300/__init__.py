"""Fused tensor-core GEMM epilogue for GB300 (sm_103a):  C = act(A.B + bias).

The computation lives in the CUDA library (csrc/, C ABI in include/tgemm.h);
this package only marshals torch tensors (device memory and the current
stream) into that ABI.
"""
from __future__ import annotations

import torch

from ._binding import (  # noqa: F401
    TGEMM_BF16, TGEMM_EPI_BIAS, TGEMM_EPI_BIAS_GELU, TGEMM_EPI_BIAS_RELU, TGEMM_EPI_GELU,
    TGEMM_EPI_NONE, TGEMM_EPI_RELU, TGEMM_F16,
    EXPORTED, NOALLOC_SCRATCH_BYTES, PLAN_FIELDS, STATUS, TgemmError, library_path, load, load_debug,
    tgemm_attention_fwd, tgemm_debug_last_check, tgemm_last_device_status, tgemm_plan, tgemm_run,
    tgemm_run_ex, tgemm_run_host, tgemm_run_noalloc,
    tgemm_status_string, tgemm_version,
)
from .build import build  # noqa: F401

EPILOGUES = {"none": TGEMM_EPI_NONE, "relu": TGEMM_EPI_RELU, "bias": TGEMM_EPI_BIAS,
             "bias_relu": TGEMM_EPI_BIAS_RELU, "gelu": TGEMM_EPI_GELU, "bias_gelu": TGEMM_EPI_BIAS_GELU}
_DT = {torch.float16: TGEMM_F16, torch.bfloat16: TGEMM_BF16}


def _epi(epilogue) -> int:
    return EPILOGUES[epilogue] if isinstance(epilogue, str) else int(epilogue)


def _check_2d(name, t):
    if t.dim() != 2 or t.stride(1) != 1:
        raise ValueError(f"{name} must be a 2-D tensor with unit column stride")


def run(A: torch.Tensor, B: torch.Tensor, bias, C: torch.Tensor, epilogue="bias_relu",
        stream=None, transpose_a: bool = False, transpose_b: bool = False) -> torch.Tensor:
    """C = epi(A @ B + bias) on CUDA tensors, enqueued on the current (or given) stream.

    A is [M, K] (or, with transpose_a, the stored [K, M] = A^T), B is [K, N]
    (or, with transpose_b, the stored [N, K] = B^T, the nn.Linear weight
    layout), C is [M, N]; each may have a row pitch wider than its width
    (stride(0) >= width); bias is [N] or None.  Raises TgemmError on a status
    other than TGEMM_OK.
    """
    # Each tensor attribute read costs a trip into torch, so every one is read once.
    sa, sb, sc = A.stride(), B.stride(), C.stride()
    if len(sa) != 2 or len(sb) != 2 or len(sc) != 2 or sa[1] != 1 or sb[1] != 1 or sc[1] != 1:
        for name, t in (("A", A), ("B", B), ("C", C)):
            _check_2d(name, t)
    (a0, a1), (b0, b1), (M, N) = A.shape, B.shape, C.shape
    M2, K = (a1, a0) if transpose_a else (a0, a1)
    K2, N2 = (b1, b0) if transpose_b else (b0, b1)
    if K2 != K or M2 != M or N2 != N:
        raise ValueError(f"shape mismatch A{tuple(A.shape)} B{tuple(B.shape)} C{tuple(C.shape)}")
    dt = A.dtype
    code = _DT.get(dt)
    if code is None or B.dtype != dt or C.dtype != dt:
        raise ValueError("A, B and C must share dtype float16 or bfloat16")
    bptr = 0
    if bias is not None:
        if bias.dtype != dt or bias.dim() != 1 or bias.numel() != N or bias.stride(0) != 1:
            raise ValueError("bias must be a contiguous [N] tensor of the same dtype")
        bptr = bias.data_ptr()
    dev = A.device
    s = stream if stream is not None else torch.cuda.current_stream(dev)
    args = (A.data_ptr(), B.data_ptr(), bptr, C.data_ptr(), M, N, K, sa[0], sb[0], sc[0], code, _epi(epilogue))
    # The library works on the current device: switch only when A is elsewhere.
    if dev.index == torch.cuda.current_device():
        st = _call(args, transpose_a, transpose_b, s.cuda_stream)
    else:
        with torch.cuda.device(dev):
            st = _call(args, transpose_a, transpose_b, s.cuda_stream)
    if st != 0:
        raise TgemmError(st)
    return C


def _call(args, transpose_a, transpose_b, stream) -> int:
    if transpose_a or transpose_b:
        return tgemm_run_ex(*args, int(transpose_a), int(transpose_b), stream)
    return tgemm_run(*args, stream)


def run_host(A: torch.Tensor, B: torch.Tensor, bias, C: torch.Tensor, epilogue="bias_relu",
             stream=None, device=None) -> torch.Tensor:
    """The same on CPU tensors (ideally pinned): copies in, computes and copies C
    back inside the library, on `stream` of `device`.  The caller synchronises."""
    _check_2d("A", A), _check_2d("B", B), _check_2d("C", C)
    M, K = A.shape
    N = B.shape[1]
    dev = torch.device(device) if device is not None else torch.device("cuda", torch.cuda.current_device())
    s = stream if stream is not None else torch.cuda.current_stream(dev)
    with torch.cuda.device(dev):
        st = tgemm_run_host(A.data_ptr(), B.data_ptr(), bias.data_ptr() if bias is not None else 0,
                            C.data_ptr(), M, N, K, A.stride(0), B.stride(0), C.stride(0),
                            _DT[A.dtype], _epi(epilogue), s.cuda_stream)
    if st != 0:
        raise TgemmError(st, "tgemm_run_host")
    return C


def attention(Q: torch.Tensor, K: torch.Tensor, V: torch.Tensor, O: torch.Tensor, causal: bool = False,
              stream=None) -> torch.Tensor:
    """O = softmax(Q K^T / sqrt(dim)) V (causal: keys up to the query) on CUDA
    tensors of shape [batch, seq, heads, 64], contiguous, float16 or bfloat16,
    enqueued on the current (or given) stream.  Raises TgemmError on a status
    other than TGEMM_OK."""
    for name, t in (("Q", Q), ("K", K), ("V", V), ("O", O)):
        if t.dim() != 4 or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous [batch, seq, heads, dim] tensor")
    if not (Q.shape == K.shape == V.shape == O.shape):
        raise ValueError("Q, K, V and O must have one shape")
    if not (Q.dtype == K.dtype == V.dtype == O.dtype) or Q.dtype not in _DT:
        raise ValueError("Q, K, V and O must share dtype float16 or bfloat16")
    batch, seq, heads, dim = Q.shape
    s = stream if stream is not None else torch.cuda.current_stream(Q.device)
    with torch.cuda.device(Q.device):
        st = tgemm_attention_fwd(Q.data_ptr(), K.data_ptr(), V.data_ptr(), O.data_ptr(), batch, seq, heads, dim,
                                 int(causal), _DT[Q.dtype], s.cuda_stream)
    if st != 0:
        raise TgemmError(st, "tgemm_attention_fwd")
    return O
