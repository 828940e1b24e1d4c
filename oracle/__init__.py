"""CPU oracle for the half-precision GEMM C = A.B -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may import this package.  The CUDA
library never loads it and shares no code with it.

The arithmetic lives in ``hgemm_oracle.c`` (plain C, fp64, k ascending), built
into ``liboracle.so`` by :func:`build`.  This module only marshals numpy
arrays of raw 16-bit patterns into it, and states the acceptance measure:

* ``Cref = sum_k dec(A[i,k]) * dec(B[k,j])`` and
  ``Den = sum_k |dec(A[i,k])| * |dec(B[k,j])|`` -- the matrix product with both
  operands row-major ("hgemm_mma_m16n8k16_mma2x4_warp4x4_kernel", section 1.1)
  accumulated wider than the inputs ("tensor-cores-cutlass-and-cute",
  section 四.1, and the "post_1787550000" experiment, section 3: wide
  accumulation is the floor);
* the normalised error ``max |C - Cref| / Den`` (entries with ``Den == 0``
  must be exactly zero).

Parity is pinned in ``tests/test_oracle_pins.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "hgemm_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

F16, BF16, E4M3, E5M2 = 0, 1, 2, 3


def build(force: bool = False) -> str:
    """Compiles ``hgemm_oracle.c`` with the host C compiler; returns the path."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
             "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            i64, p = ctypes.c_int64, ctypes.c_void_p
            lib.oracle_gemm.argtypes = [p, p, ctypes.c_int, i64, i64, i64, i64, i64,
                                        i64, i64, i64, p, p, ctypes.c_int]
            lib.oracle_gemm.restype = ctypes.c_int
            lib.oracle_gemm_entries.argtypes = [p, p, ctypes.c_int, i64, i64, i64, i64, i64,
                                                i64, p, p, p, p, p]
            lib.oracle_gemm_entries.restype = ctypes.c_int
            lib.oracle_decode_f16.argtypes = [ctypes.c_uint16]
            lib.oracle_decode_f16.restype = ctypes.c_double
            lib.oracle_decode_bf16.argtypes = [ctypes.c_uint16]
            lib.oracle_decode_bf16.restype = ctypes.c_double
            lib.oracle_decode_e4m3.argtypes = [ctypes.c_uint16]
            lib.oracle_decode_e4m3.restype = ctypes.c_double
            lib.oracle_decode_e5m2.argtypes = [ctypes.c_uint16]
            lib.oracle_decode_e5m2.restype = ctypes.c_double
            lib.oracle_decode_array.argtypes = [p, ctypes.c_int, i64, p]
            lib.oracle_decode_array.restype = None
            lib.oracle_attention.argtypes = [p, p, p, ctypes.c_int, i64, i64, i64, ctypes.c_double,
                                             ctypes.c_int, i64, p, p, p, p, p, p, ctypes.c_int]
            lib.oracle_attention.restype = ctypes.c_int
            _lib = lib
    return _lib


def _u16(x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x)
    if x.dtype != np.uint16:
        raise TypeError("oracle inputs are raw 16-bit patterns (numpy uint16)")
    return x


def _ptr(x: np.ndarray) -> int:
    return x.ctypes.data


def gemm(A: np.ndarray, B: np.ndarray, dtype_in: int, M: int, N: int, K: int,
         lda: int, ldb: int, batch: int = 1, strideA: int = 0, strideB: int = 0,
         threads: int | None = None):
    """Full product.  ``A``/``B`` are flat uint16 buffers read with the given
    leading dimensions and batch strides (in elements).  Returns ``(Cref, Den)``
    as fp64 arrays of shape ``(batch, M, N)``."""
    lib = _load()
    A, B = _u16(A), _u16(B)
    _check_extent(A, M, K, lda, batch, strideA)
    _check_extent(B, K, N, ldb, batch, strideB)
    Cref = np.empty((batch, M, N), dtype=np.float64)
    Den = np.empty((batch, M, N), dtype=np.float64)
    if threads is None:
        threads = os.cpu_count() or 1
    rc = lib.oracle_gemm(_ptr(A), _ptr(B), dtype_in, M, N, K, lda, ldb, batch,
                         strideA, strideB, _ptr(Cref), _ptr(Den), int(threads))
    if rc != 0:
        raise ValueError("oracle_gemm rejected its arguments")
    return Cref, Den


def gemm_bt(A: np.ndarray, Bs: np.ndarray, dtype_in: int, M: int, N: int, K: int,
            lda: int, ldb: int, batch: int = 1, strideA: int = 0, strideB: int = 0):
    """C = A . Bs^T with ``Bs`` stored N x K (element (j, k) of batch b at
    b*strideB + j*ldb + k): the product with B[k][j] = Bs[j][k].  The stored
    matrix is transposed into a dense K x N copy (data movement only) and the
    product is :func:`gemm`'s."""
    Bs = _u16(Bs)
    _check_extent(Bs, N, K, ldb, batch, strideB)
    Bt = np.empty((batch, K, N), dtype=np.uint16)
    for b in range(batch):
        if N and K:
            rows = np.lib.stride_tricks.as_strided(Bs[b * strideB:], shape=(N, K), strides=(ldb * 2, 2))
            Bt[b] = rows.T
    return gemm(A, Bt.reshape(-1), dtype_in, M, N, K, lda, N, batch, strideA, K * N)


def gemm_entries(A: np.ndarray, B: np.ndarray, dtype_in: int, K: int, lda: int, ldb: int,
                 eb, ei, ej, strideA: int = 0, strideB: int = 0):
    """The same definition for the entries ``(eb[e], ei[e], ej[e])`` only."""
    lib = _load()
    A, B = _u16(A), _u16(B)
    eb = np.ascontiguousarray(eb, dtype=np.int64)
    ei = np.ascontiguousarray(ei, dtype=np.int64)
    ej = np.ascontiguousarray(ej, dtype=np.int64)
    n = eb.size
    if not (ei.size == n and ej.size == n):
        raise ValueError("entry index arrays differ in length")
    if n:
        # every element the sums touch must lie inside the buffers
        amax = int(eb.max()) * strideA + int(ei.max()) * lda + max(K - 1, 0)
        bmax = int(eb.max()) * strideB + max(K - 1, 0) * ldb + int(ej.max())
        if K > 0 and (amax >= A.size or bmax >= B.size):
            raise ValueError("entry indices reach outside the operand buffers")
    Cref = np.empty(n, dtype=np.float64)
    Den = np.empty(n, dtype=np.float64)
    rc = lib.oracle_gemm_entries(_ptr(A), _ptr(B), dtype_in, K, lda, ldb, strideA, strideB,
                                 n, _ptr(eb), _ptr(ei), _ptr(ej), _ptr(Cref), _ptr(Den))
    if rc != 0:
        raise ValueError("oracle_gemm_entries rejected its arguments")
    return Cref, Den


def widen8(b: np.ndarray) -> np.ndarray:
    """8-bit patterns (E4M3 / E5M2) as the 16-bit pattern arrays the oracle
    reads (the byte in the low half)."""
    return np.ascontiguousarray(np.asarray(b, dtype=np.uint8).astype(np.uint16))


def decode(bits: np.ndarray, dtype: int) -> np.ndarray:
    """Reads raw fp16 (dtype 0), bf16 (1), E4M3 (2) or E5M2 (3) patterns
    (16-bit arrays; 8-bit patterns widened) with the oracle's own decoders;
    returns fp64 of the same shape."""
    lib = _load()
    bits = _u16(bits)
    out = np.empty(bits.shape, dtype=np.float64)
    lib.oracle_decode_array(_ptr(bits), int(dtype), bits.size, _ptr(out))
    return out


def decode_one(h: int, dtype: int) -> float:
    lib = _load()
    return [lib.oracle_decode_f16, lib.oracle_decode_bf16, lib.oracle_decode_e4m3,
            lib.oracle_decode_e5m2][dtype](h)


def normalized_error(C: np.ndarray, Cref: np.ndarray, Den: np.ndarray) -> float:
    """``max |C - Cref| / Den`` over entries with ``Den > 0``; an entry with
    ``Den == 0`` (an empty sum or a zero row/column) that is not exactly zero
    counts as an infinite error, and a NaN anywhere in C where Cref is finite
    does too."""
    C = np.asarray(C, dtype=np.float64)
    if C.shape != Cref.shape:
        raise ValueError(f"shape mismatch {C.shape} vs {Cref.shape}")
    if C.size == 0:
        return 0.0
    bad_nan = np.isnan(C) & ~np.isnan(Cref)
    if bad_nan.any():
        return float("inf")
    zero = Den == 0
    if (C[zero] != 0).any():
        return float("inf")
    nz = ~zero
    if not nz.any():
        return 0.0
    return float(np.max(np.abs(C[nz] - Cref[nz]) / Den[nz]))


def flops(M: int, N: int, K: int, batch: int = 1) -> int:
    """2*M*N*K per product: one multiply and one add per term
    ("tensor-cores-cutlass-and-cute", section 四.1)."""
    return 2 * M * N * K * batch


def min_bytes(M: int, N: int, K: int, in_bytes: int, out_bytes: int, batch: int = 1) -> int:
    """Each of A, B read once and C written once
    ("tensor-cores-cutlass-and-cute", section 四.1)."""
    return batch * (M * K * in_bytes + K * N * in_bytes + M * N * out_bytes)


def _check_extent(X: np.ndarray, rows: int, cols: int, ld: int, batch: int, stride: int):
    if rows == 0 or cols == 0:
        return
    if ld < cols:
        raise ValueError("leading dimension shorter than a row")
    last = (batch - 1) * stride + (rows - 1) * ld + cols - 1
    if last >= X.size:
        raise ValueError("operand buffer too small for its shape")


# ---------------------------------------------------------------- fused epilogue

ACT_NONE, ACT_RELU, ACT_GELU, ACT_GELU_TANH = 0, 1, 2, 3

# Largest slope of GELU(x) = x * Phi(x): its derivative Phi(x) + x * phi(x)
# has derivative phi(x) * (2 - x^2), so it peaks at x = sqrt(2) at
# Phi(sqrt 2) + sqrt(2) * phi(sqrt 2) = 1.1289...  An error e in GELU's
# argument moves its value by at most this times e.
GELU_MAX_SLOPE = (0.5 * (1.0 + __import__("math").erf(1.0))
                  + np.sqrt(2.0) * np.exp(-1.0) / np.sqrt(2.0 * np.pi))


def _phi_cdf(x: np.ndarray) -> np.ndarray:
    """Standard normal CDF, 0.5 * (1 + erf(x / sqrt 2)), in fp64."""
    try:
        from scipy.special import erf  # library routine for erf
        return 0.5 * (1.0 + erf(x / np.sqrt(2.0)))
    except ImportError:  # pragma: no cover - scipy is on both machines
        import math
        return 0.5 * (1.0 + np.vectorize(math.erf)(x / np.sqrt(2.0)))


def activation(x: np.ndarray, act: int) -> np.ndarray:
    """ReLU max(x, 0), GELU x * Phi(x) (the erf form of the Gaussian error
    linear unit: cuBLASLt's BIAS / RELU / GELU epilogues that
    "tensor-cores-cutlass-and-cute" lists in its comparison with cuBLAS), or
    its tanh form."""
    x = np.asarray(x, dtype=np.float64)
    if act == ACT_NONE:
        return x
    if act == ACT_RELU:
        return np.maximum(x, 0.0)
    if act == ACT_GELU:
        return x * _phi_cdf(x)
    if act == ACT_GELU_TANH:
        # the tanh form of GELU: 0.5 x (1 + tanh(sqrt(2/pi) (x + 0.044715 x^3)))
        return 0.5 * x * (1.0 + np.tanh(np.sqrt(2.0 / np.pi) * (x + 0.044715 * x ** 3)))
    raise ValueError("unknown activation")


def epilogue(Cref: np.ndarray, Den: np.ndarray, *, alpha: float = 1.0, beta: float = 0.0,
             C_prev: np.ndarray | None = None, bias: np.ndarray | None = None,
             row_scale: np.ndarray | None = None, col_scale: np.ndarray | None = None,
             act: int = ACT_NONE):
    """The fused epilogue in fp64 on the oracle's product (shape (batch,) M x N):

        D[i][j] = act(alpha * rs[i] * cs[j] * Cref[i][j] + beta * C_prev[i][j] + bias[j])

    (rs, cs, bias default to 1, 1, 0; the vectors are shared by every batch
    entry).  Returns (D, DenD), DenD the acceptance denominator: the bound on
    |D - D_gpu| that the product's own bound Den carries through the affine
    part, plus the magnitudes of the added terms (each rounded once in fp32),
    times GELU's largest slope when GELU is applied."""
    Cref = np.asarray(Cref, dtype=np.float64)
    Den = np.asarray(Den, dtype=np.float64)
    M, N = Cref.shape[-2], Cref.shape[-1]
    rs = np.ones(M) if row_scale is None else np.asarray(row_scale, dtype=np.float64)
    cs = np.ones(N) if col_scale is None else np.asarray(col_scale, dtype=np.float64)
    scale = alpha * rs[:, None] * cs[None, :]
    t = scale * Cref
    den = np.abs(scale) * Den
    if beta != 0.0:
        Cp = np.asarray(C_prev, dtype=np.float64)
        t = t + beta * Cp
        den = den + np.abs(beta * Cp)
    if bias is not None:
        bv = np.asarray(bias, dtype=np.float64)[None, :]
        t = t + bv
        den = den + np.abs(bv)
    if act in (ACT_GELU, ACT_GELU_TANH):
        den = den * GELU_MAX_SLOPE
    return activation(t, act), den


# ---------------------------------------------------------------- attention

def attention(Q: np.ndarray, K: np.ndarray, V: np.ndarray, dtype_in: int, BH: int, SQ: int,
              SKV: int, D: int, scale: float, causal: bool = False, rows=None,
              threads: int | None = None):
    """Attention forward, the plain definition (``oracle_attention`` in
    ``hgemm_oracle.c``): O = softmax(scale * Q K^T [causal mask]) V per
    (bh, query row), in fp64.  ``Q`` is a flat uint16 buffer [BH][SQ][D],
    ``K`` and ``V`` [BH][SKV][D].  Causal: key j is allowed for query i when
    j <= i + SKV - SQ.

    ``rows``: None for every row, else a pair of index arrays ``(b, i)``.
    Returns ``(O, Den, lse, sden)``: O and Den shaped (BH, SQ, D) or (n, D);
    lse and sden (BH, SQ) or (n,).  ``Den[c] = sum_j p_j |v_j[c]| / l`` is the
    error normaliser; ``sden`` bounds |scale * q.k| by the sum of magnitudes."""
    lib = _load()
    Q, K, V = _u16(Q), _u16(K), _u16(V)
    if Q.size < BH * SQ * D or K.size < BH * SKV * D or V.size < BH * SKV * D:
        raise ValueError("attention operands are smaller than [BH][seq][D]")
    if rows is None:
        rb = np.repeat(np.arange(BH, dtype=np.int64), SQ)
        ri = np.tile(np.arange(SQ, dtype=np.int64), BH)
        shape = (BH, SQ)
    else:
        rb = np.ascontiguousarray(rows[0], dtype=np.int64)
        ri = np.ascontiguousarray(rows[1], dtype=np.int64)
        if rb.size != ri.size:
            raise ValueError("row index arrays differ in length")
        if rb.size and (rb.min() < 0 or rb.max() >= BH or ri.min() < 0 or ri.max() >= SQ):
            raise ValueError("row indices out of range")
        shape = (rb.size,)
    n = rb.size
    O = np.empty((n, D), dtype=np.float64)
    Den = np.empty((n, D), dtype=np.float64)
    lse = np.empty(n, dtype=np.float64)
    sden = np.empty(n, dtype=np.float64)
    if threads is None:
        threads = os.cpu_count() or 1
    rc = lib.oracle_attention(_ptr(Q), _ptr(K), _ptr(V), dtype_in, SQ, SKV, D, float(scale),
                              int(bool(causal)), n, _ptr(rb), _ptr(ri), _ptr(O), _ptr(Den),
                              _ptr(lse), _ptr(sden), int(threads))
    if rc != 0:
        raise ValueError("oracle_attention rejected its arguments")
    return (O.reshape(*shape, D), Den.reshape(*shape, D), lse.reshape(shape), sden.reshape(shape))
