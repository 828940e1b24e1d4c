"""Torch-tensor front end of the one-shot ``hgemm`` entry point.

Only argument marshalling: shapes, strides and dtypes are read from the
tensors, the output is allocated with torch (device memory is torch's job),
and the product itself is computed by libhgemm's kernels.  There is no CPU or
library fallback: a missing library or a non-CUDA tensor raises.
"""
from __future__ import annotations

import torch

from . import hgemm as _h

_IN = {torch.float16: _h.HGEMM_F16, torch.bfloat16: _h.HGEMM_BF16}
_OUT = {torch.float16: _h.HGEMM_F16, torch.bfloat16: _h.HGEMM_BF16, torch.float32: _h.HGEMM_F32}


def matmul(A: torch.Tensor, B: torch.Tensor, out_dtype: torch.dtype | None = None,
           out: torch.Tensor | None = None, stream: torch.cuda.Stream | None = None) -> torch.Tensor:
    """C = A @ B for row-major fp16/bf16 CUDA tensors, fp32 accumulation.

    ``A`` is ``(M, K)`` or ``(batch, M, K)``, ``B`` is ``(K, N)`` or
    ``(batch, K, N)``; the last dimension of each must be contiguous (any
    leading-dimension / batch stride is passed through).  ``out_dtype``
    defaults to the input dtype; ``out`` may be given with a contiguous last
    dimension."""
    if A.dtype not in _IN or B.dtype != A.dtype:
        raise TypeError(f"A and B must both be float16 or both bfloat16 (got {A.dtype}, {B.dtype})")
    if not (A.is_cuda and B.is_cuda) or A.device != B.device:
        raise ValueError("A and B must be CUDA tensors on the same device")
    if A.dim() != B.dim() or A.dim() not in (2, 3):
        raise ValueError("A and B must both be 2-D or both 3-D")
    batched = A.dim() == 3
    if batched and A.shape[0] != B.shape[0]:
        raise ValueError("batch sizes differ")
    M, K = A.shape[-2], A.shape[-1]
    if B.shape[-2] != K:
        raise ValueError(f"inner dimensions differ: {K} vs {B.shape[-2]}")
    N = B.shape[-1]
    batch = A.shape[0] if batched else 1
    if (K > 1 and A.stride(-1) != 1) or (N > 1 and B.stride(-1) != 1):
        raise ValueError("the last dimension of A and B must be contiguous")
    out_dtype = out_dtype or A.dtype
    if out_dtype not in _OUT:
        raise TypeError(f"unsupported output dtype {out_dtype}")
    shape = (batch, M, N) if batched else (M, N)
    if out is None:
        out = torch.empty(shape, dtype=out_dtype, device=A.device)
    elif tuple(out.shape) != shape or out.dtype != out_dtype or out.device != A.device:
        raise ValueError("out has the wrong shape, dtype or device")
    elif N > 1 and out.stride(-1) != 1:
        raise ValueError("the last dimension of out must be contiguous")
    lda = A.stride(-2) if M > 1 else max(K, 1)
    ldb = B.stride(-2) if K > 1 else max(N, 1)
    ldc = out.stride(-2) if M > 1 else max(N, 1)
    sA = A.stride(0) if batched else 0
    sB = B.stride(0) if batched else 0
    sC = out.stride(0) if batched else 0
    with torch.cuda.device(A.device):
        _h.hgemm(A, B, out, M, N, K, lda, ldb, ldc, batch, sA, sB, sC, _IN[A.dtype], _OUT[out_dtype],
                 stream if stream is not None else torch.cuda.current_stream(A.device))
    return out
