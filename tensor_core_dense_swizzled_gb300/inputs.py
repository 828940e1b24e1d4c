"""Seeded synthetic inputs for the GEMM workloads.

This module holds no GEMM arithmetic: it only draws the operands, so that the
CUDA path and the CPU oracle can be fed the very same bits.  Every draw runs on
the CPU from ``torch.Generator().manual_seed(seed)`` in fp32, A first and then
B, and is rounded to the input type with round-to-nearest-even by ``.to()``.

The workloads are the five shapes the GEMM is judged on (all row-major, fp32
accumulation):

==========================  =========================================================
name                        shape / values
==========================  =========================================================
``int512``                  512^3 fp16, integers uniform in [-4, 4], seed 0, fp32 out
``square4096``              4096^3 bf16, N(0,1), seed 1, bf16 out
``square8192``              8192^3 fp16, U[-1,1], seed 2, fp16 out
``batched_qk``              64 x (1024x128)(128x1024) bf16, N(0,1)/sqrt(128), seed 3,
                            fp32 out -- the attention S = Q K^T shape, K^T stored
                            row-major (128 x 1024)
``ragged4095``              4095^3 fp16, U[-1,1], seed 3, fp32 out (lda=ldb=ldc=4095)
``ragged4095_h``            the same inputs, fp16 out
``skinny``                  M=8, N=28672, K=4096 bf16; A N(0,1), B N(0,0.02), seed 4,
                            bf16 out
``*_tn``                    the same draws with B stored N x K
``square4096_fp8``          4096^3 E4M3, N(0,1), seed 1, B stored N x K, bf16 out
``skinny_fp8``              8 x 28672 x 4096 E4M3; A N(0,1), B N(0,1), seed 4, B
                            stored N x K, bf16 out
==========================  =========================================================

Attention workloads (``ATTENTION_WORKLOADS``): ``attn`` is 64 heads x
(1024 queries, 1024 keys, head dimension 128) bf16 -- the batched S = Q K^T
shape above, followed by the softmax and O = P V -- with Q, K, V drawn
N(0, 1) in that order from seed 5 and scale 1/sqrt(128); ``attn_causal`` the
same with the causal mask.

8-bit draws are rounded by ``.to(torch.float8_e4m3fn / float8_e5m2)``; the
distributions stay far inside both formats' ranges (448 and 57344), so no
value saturates or overflows.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import torch

__all__ = ["Workload", "WORKLOADS", "make_inputs", "make_random", "torch_dtype",
           "AttentionWorkload", "ATTENTION_WORKLOADS", "make_attention_inputs"]

_TD = {"f16": torch.float16, "bf16": torch.bfloat16, "f32": torch.float32,
       "e4m3": torch.float8_e4m3fn, "e5m2": torch.float8_e5m2}


def torch_dtype(name: str) -> torch.dtype:
    return _TD[name]


@dataclass(frozen=True)
class Workload:
    name: str
    M: int
    N: int
    K: int
    batch: int
    dtype_in: str   # "f16" | "bf16" | "e4m3" | "e5m2"
    dtype_out: str  # "f32" | "f16" | "bf16"
    dist_a: str     # "int4" | "normal" | "uniform"
    dist_b: str
    scale_a: float
    scale_b: float
    seed: int
    trans_b: bool = False  # B stored N x K (C = A . B_stored^T), same values as the K x N draw

    @property
    def lda(self) -> int:
        return self.K

    @property
    def ldb(self) -> int:
        return self.K if self.trans_b else self.N

    @property
    def ldc(self) -> int:
        return self.N

    @property
    def strideA(self) -> int:
        return self.M * self.K if self.batch > 1 else 0

    @property
    def strideB(self) -> int:
        return self.K * self.N if self.batch > 1 else 0  # K x N or N x K: the same size

    @property
    def strideC(self) -> int:
        return self.M * self.N if self.batch > 1 else 0


WORKLOADS = {
    w.name: w
    for w in [
        Workload("int512", 512, 512, 512, 1, "f16", "f32", "int4", "int4", 1.0, 1.0, 0),
        Workload("square4096", 4096, 4096, 4096, 1, "bf16", "bf16", "normal", "normal", 1.0, 1.0, 1),
        Workload("square8192", 8192, 8192, 8192, 1, "f16", "f16", "uniform", "uniform", 1.0, 1.0, 2),
        Workload("batched_qk", 1024, 1024, 128, 64, "bf16", "f32", "normal", "normal",
                 1.0 / math.sqrt(128.0), 1.0 / math.sqrt(128.0), 3),
        Workload("ragged4095", 4095, 4095, 4095, 1, "f16", "f32", "uniform", "uniform", 1.0, 1.0, 3),
        Workload("ragged4095_h", 4095, 4095, 4095, 1, "f16", "f16", "uniform", "uniform", 1.0, 1.0, 3),
        Workload("skinny", 8, 28672, 4096, 1, "bf16", "bf16", "normal", "normal", 1.0, 0.02, 4),
        # the same products with B stored N x K: a linear layer's [out][in]
        # weight, attention's K stored [seq][dim], and the square product
        Workload("skinny_tn", 8, 28672, 4096, 1, "bf16", "bf16", "normal", "normal", 1.0, 0.02, 4,
                 trans_b=True),
        Workload("batched_qk_tn", 1024, 1024, 128, 64, "bf16", "f32", "normal", "normal",
                 1.0 / math.sqrt(128.0), 1.0 / math.sqrt(128.0), 3, trans_b=True),
        Workload("square4096_tn", 4096, 4096, 4096, 1, "bf16", "bf16", "normal", "normal", 1.0, 1.0, 1,
                 trans_b=True),
        # 8-bit inputs (B stored N x K, the layout 8-bit tensor-core operands take)
        Workload("square4096_fp8", 4096, 4096, 4096, 1, "e4m3", "bf16", "normal", "normal", 1.0, 1.0,
                 1, trans_b=True),
        Workload("skinny_fp8", 8, 28672, 4096, 1, "e4m3", "bf16", "normal", "normal", 1.0, 1.0, 4,
                 trans_b=True),
    ]
}


def _draw(gen: torch.Generator, shape, dist: str, scale: float) -> torch.Tensor:
    if dist == "int4":  # integers uniform on {-4, ..., 4}
        return torch.randint(-4, 5, shape, generator=gen, dtype=torch.int32).to(torch.float32)
    if dist == "normal":
        return torch.randn(shape, generator=gen, dtype=torch.float32) * scale
    if dist == "uniform":  # U[-1, 1]
        return (torch.rand(shape, generator=gen, dtype=torch.float32) * 2.0 - 1.0) * scale
    raise ValueError(f"unknown distribution {dist!r}")


def make_inputs(w: Workload):
    """Returns CPU tensors ``(A, B)`` in the workload's input dtype, shaped
    ``(batch, M, K)`` / ``(batch, K, N)`` when ``batch > 1`` and ``(M, K)`` /
    ``(K, N)`` otherwise (B ``(..., N, K)`` for ``trans_b`` workloads); all
    contiguous row-major."""
    gen = torch.Generator().manual_seed(w.seed)
    sa = (w.batch, w.M, w.K) if w.batch > 1 else (w.M, w.K)
    sb = (w.batch, w.K, w.N) if w.batch > 1 else (w.K, w.N)
    A = _draw(gen, sa, w.dist_a, w.scale_a).to(_TD[w.dtype_in])
    B = _draw(gen, sb, w.dist_b, w.scale_b).to(_TD[w.dtype_in])
    if w.trans_b:  # stored N x K, the same values
        B = B.transpose(-1, -2).contiguous()
    return A, B


def make_random(shape, dtype_in: str, seed: int, dist: str = "normal", scale: float = 1.0):
    """One seeded tensor of the given shape (for the small parity cases)."""
    gen = torch.Generator().manual_seed(seed)
    return _draw(gen, tuple(shape), dist, scale).to(_TD[dtype_in])


@dataclass(frozen=True)
class AttentionWorkload:
    name: str
    bh: int      # batch x heads
    sq: int      # query rows per head
    skv: int     # key / value rows per head
    dtype: str   # "bf16" | "f16" (inputs and output)
    causal: bool
    seed: int

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(128.0)


ATTENTION_WORKLOADS = {
    w.name: w
    for w in [
        AttentionWorkload("attn", 64, 1024, 1024, "bf16", False, 5),
        AttentionWorkload("attn_causal", 64, 1024, 1024, "bf16", True, 5),
    ]
}


def make_attention_inputs(w: AttentionWorkload):
    """CPU tensors ``(Q, K, V)`` shaped (bh, seq, 128), contiguous, N(0, 1)."""
    gen = torch.Generator().manual_seed(w.seed)
    Q = _draw(gen, (w.bh, w.sq, 128), "normal", 1.0).to(_TD[w.dtype])
    K = _draw(gen, (w.bh, w.skv, 128), "normal", 1.0).to(_TD[w.dtype])
    V = _draw(gen, (w.bh, w.skv, 128), "normal", 1.0).to(_TD[w.dtype])
    return Q, K, V
