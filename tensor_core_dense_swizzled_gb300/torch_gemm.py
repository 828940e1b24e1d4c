"""Torch-tensor front end of libhgemm.

Only argument marshalling: shapes, strides and dtypes are read from the
tensors, the output is allocated with torch (device memory is torch's job),
and the product itself is computed by libhgemm's kernels.  There is no CPU or
library fallback: a missing library or a non-CUDA tensor raises.

Plain products go through the one-shot ``hgemm`` entry point (its plan cache
lives in the library).  Products with B given as the transpose of a row-major
N x K tensor (``B = W.t()``), 8-bit inputs or a fused epilogue go through
plans created with ``hgemm_plan_create_ex`` and kept in a cache here
(:func:`matmul_cache_clear` frees them).  Both caches hold one plan per
stream (a plan's workspace must not serve two streams at once), and a plan's
host-side run is serialised, so matmul may be called from several threads
and streams at once.
"""
from __future__ import annotations

import threading
import types

import torch

from . import hgemm as _h

_IN = {torch.float16: _h.HGEMM_F16, torch.bfloat16: _h.HGEMM_BF16,
       torch.float8_e4m3fn: _h.HGEMM_E4M3, torch.float8_e5m2: _h.HGEMM_E5M2}
_F8 = (torch.float8_e4m3fn, torch.float8_e5m2)
_OUT = {torch.float16: _h.HGEMM_F16, torch.bfloat16: _h.HGEMM_BF16, torch.float32: _h.HGEMM_F32}
_ACT = {None: _h.HGEMM_ACT_NONE, "none": _h.HGEMM_ACT_NONE, "relu": _h.HGEMM_ACT_RELU,
        "gelu": _h.HGEMM_ACT_GELU, "gelu_tanh": _h.HGEMM_ACT_GELU_TANH}

_plans: dict = {}  # key (arguments, stream) -> (plan handle, lock held while it runs)
_plans_lock = threading.Lock()


def _plan(key, M, N, K, lda, ldb, ldc, batch, sA, sB, sC, din, dout, trans_b):
    with _plans_lock:
        entry = _plans.get(key)
        if entry is None:
            h = _h.hgemm_plan_create_ex(M, N, K, lda, ldb, ldc, batch, sA, sB, sC, din, dout,
                                        _h.Options(trans_b=int(trans_b)))
            entry = (h, threading.Lock())
            _plans[key] = entry
        return entry


def matmul_cache_clear() -> None:
    """Destroys the plans :func:`matmul` created (none may still be running)."""
    with _plans_lock:
        for h, _ in _plans.values():
            _h.hgemm_plan_destroy(h)
        _plans.clear()


def matmul(A: torch.Tensor, B: torch.Tensor, out_dtype: torch.dtype | None = None,
           out: torch.Tensor | None = None, stream: torch.cuda.Stream | None = None, *,
           alpha: float = 1.0, beta: float = 0.0, bias: torch.Tensor | None = None,
           row_scale: torch.Tensor | None = None, col_scale: torch.Tensor | None = None,
           activation: str | None = None) -> torch.Tensor:
    """C = act(alpha * rs[i] * cs[j] * (A @ B) + beta * C + bias[j]) for CUDA
    tensors, fp32 accumulation.

    ``A`` is ``(M, K)`` or ``(batch, M, K)`` with a contiguous last dimension.
    ``B`` is ``(K, N)`` or ``(batch, K, N)``, either with a contiguous last
    dimension, or the transpose of a tensor stored N x K (``W.t()``: stride 1
    along K), which runs the transposed-B path.  Inputs float16 / bfloat16, or
    float8_e4m3fn / float8_e5m2 (both the same type; 8-bit inputs need B in
    the transposed form and 16-byte aligned rows).  ``out_dtype`` defaults to
    the input dtype (bfloat16 for 8-bit inputs); ``out`` may be given with a
    contiguous last dimension (its values are C above when beta != 0).
    ``bias``, ``row_scale``, ``col_scale``: fp32 CUDA vectors of N, M, N values;
    ``activation``: None, "relu", "gelu" (erf form) or "gelu_tanh"."""
    if A.dtype not in _IN or B.dtype != A.dtype:
        raise TypeError(f"A and B must have the same input dtype among {list(_IN)} "
                        f"(got {A.dtype}, {B.dtype})")
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
    if K > 1 and A.stride(-1) != 1:
        raise ValueError("the last dimension of A must be contiguous")
    # B given as W.t() with W stored N x K: stride 1 along K
    trans_b = N > 1 and B.stride(-1) != 1 and (K <= 1 or B.stride(-2) == 1)
    if N > 1 and B.stride(-1) != 1 and not trans_b:
        raise ValueError("B must have a contiguous last dimension or be the transpose of one")
    f8 = A.dtype in _F8
    if f8 and not trans_b:
        raise ValueError("8-bit inputs take B as the transpose of an N x K tensor (W.t())")
    out_dtype = out_dtype or (torch.bfloat16 if f8 else A.dtype)
    if out_dtype not in _OUT:
        raise TypeError(f"unsupported output dtype {out_dtype}")
    if activation not in _ACT:
        raise ValueError(f"unknown activation {activation!r}")
    shape = (batch, M, N) if batched else (M, N)
    if out is None:
        if beta != 0.0:
            raise ValueError("beta != 0 reads C: pass out")
        out = torch.empty(shape, dtype=out_dtype, device=A.device)
    elif tuple(out.shape) != shape or out.dtype != out_dtype or out.device != A.device:
        raise ValueError("out has the wrong shape, dtype or device")
    elif N > 1 and out.stride(-1) != 1:
        raise ValueError("the last dimension of out must be contiguous")
    for name, vec, n in (("bias", bias, N), ("row_scale", row_scale, M), ("col_scale", col_scale, N)):
        if vec is not None and (vec.dtype != torch.float32 or not vec.is_cuda or vec.numel() != n
                                or not vec.is_contiguous() or vec.device != A.device):
            raise ValueError(f"{name} must be a contiguous fp32 CUDA tensor of {n} values")
    lda = A.stride(-2) if M > 1 else max(K, 1)
    if trans_b:
        ldb = B.stride(-1) if N > 1 else max(K, 1)
    else:
        ldb = B.stride(-2) if K > 1 else max(N, 1)
    ldc = out.stride(-2) if M > 1 else max(N, 1)
    sA = A.stride(0) if batched else 0
    sB = B.stride(0) if batched else 0
    sC = out.stride(0) if batched else 0
    din, dout = _IN[A.dtype], _OUT[out_dtype]
    stream = stream if stream is not None else torch.cuda.current_stream(A.device)
    epi = (alpha != 1.0 or beta != 0.0 or bias is not None or row_scale is not None
           or col_scale is not None or _ACT[activation] != _h.HGEMM_ACT_NONE)
    with torch.cuda.device(A.device):
        if not trans_b and not epi:
            _h.hgemm(A, B, out, M, N, K, lda, ldb, ldc, batch, sA, sB, sC, din, dout, stream)
            return out
        key = (A.device.index, M, N, K, lda, ldb, ldc, batch, sA, sB, sC, din, dout, trans_b,
               stream.cuda_stream)
        plan, lock = _plan(key, M, N, K, lda, ldb, ldc, batch, sA, sB, sC, din, dout, trans_b)
        with lock:
            if epi:
                ep = types.SimpleNamespace(alpha=float(alpha), beta=float(beta), bias=bias,
                                           row_scale=row_scale, col_scale=col_scale,
                                           activation=_ACT[activation])
                _h.hgemm_run_ex(plan, A, B, out, ep, stream)
            else:
                _h.hgemm_run(plan, A, B, out, stream)
    return out
