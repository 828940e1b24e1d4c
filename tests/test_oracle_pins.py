"""Pins of the CPU oracle to facts that do not come from the oracle itself.

* the worked example of the single-warp layout experiment
  (dandandamowang.xyz "post_1787550000", section 6.1), stored in
  ``tests/golden/worked_example_16x8x16.txt``;
* the printed work / traffic counts of the 4096^3 GEMM
  ("tensor-cores-cutlass-and-cute", section 四.1), in
  ``tests/golden/gemm_counts_4096.txt``;
* exact sums on small shapes: products of two 16-bit floats are exact in
  binary64, so ``math.fsum`` of them is the exact sum correctly rounded, and
  Python ``Fraction`` gives the exact rational;
* special cases with a textbook answer (identity, one-hot rows, zeros) and
  integer data, where numpy's int64 matmul is exact;
* the decoders against numpy's binary16 and binary32 decoders over all
  65536 patterns;
* mutations (a transposed operand, a dropped term, a sign flip, a shifted
  index) fed through the oracle's arguments must break a pin.
"""
import math
import os
from fractions import Fraction

import numpy as np
import pytest

from tensor_core_dense_swizzled_gb300 import inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def bits(t):
    """Raw uint16 patterns of a CPU fp16/bf16 tensor."""
    import torch
    return t.contiguous().view(torch.int16).numpy().view(np.uint16).reshape(-1)


def lib_decode(b, dtype):
    """Library decoders, independent of the oracle's: numpy binary16, and
    bf16 as the upper half of a binary32."""
    b = np.asarray(b, dtype=np.uint16)
    if dtype == 0:
        return b.view(np.float16).astype(np.float64)
    with np.errstate(invalid="ignore"):
        return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def encode_exact(values, dtype):
    """Patterns of values that are exact in the format (checked)."""
    v = np.asarray(values, dtype=np.float64)
    if dtype == 0:
        b = v.astype(np.float16).view(np.uint16)
    else:
        f = v.astype(np.float32).view(np.uint32)
        assert np.all((f & 0xFFFF) == 0), "value not exact in bf16"
        b = (f >> 16).astype(np.uint16)
    assert np.array_equal(lib_decode(b, dtype), v)
    return b


def load_worked_example():
    spots, rows = [], []
    with open(os.path.join(GOLDEN, "worked_example_16x8x16.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            tok = line.split()
            if tok[0] == "spot":
                spots.append(tuple(int(x) for x in tok[1:]))
            elif tok[0] == "row":
                rows.append([int(x) for x in tok[1:]])
    return spots, np.array(rows, dtype=np.float64)


def worked_example_operands(dtype):
    A = np.array([[i for k in range(16)] for i in range(16)], dtype=np.float64)
    B = np.array([[j for j in range(8)] for k in range(16)], dtype=np.float64)
    return encode_exact(A, dtype).reshape(-1), encode_exact(B, dtype).reshape(-1)


# ---------------------------------------------------------------- worked example

@pytest.mark.parametrize("dtype", [0, 1])
def test_worked_example(oracle_mod, dtype):
    spots, table = load_worked_example()
    assert table.shape == (16, 8)
    assert (3, 5, 240) in spots and (15, 7, 1680) in spots
    A, B = worked_example_operands(dtype)
    Cref, Den = oracle_mod.gemm(A, B, dtype, 16, 8, 16, 16, 8)
    assert np.array_equal(Cref[0], table)
    for i, j, v in spots:
        assert Cref[0, i, j] == v
    # all inputs are non-negative, so the normaliser equals the sum itself
    assert np.array_equal(Den[0], table)


def test_worked_example_transposed_operand_is_caught(oracle_mod):
    """A transposed B (reading B[j][k] for B[k][j]) must break the pin:
    the pages point out that such layout slips change values silently."""
    _, table = load_worked_example()
    A, B = worked_example_operands(0)
    Bt = np.ascontiguousarray(B.reshape(16, 8).T).reshape(-1)  # 8 x 16
    # read the 8x16 buffer as if it were 16x8 with ld 8
    Cbad, _ = oracle_mod.gemm(A, Bt, 0, 16, 8, 16, 16, 8)
    assert not np.array_equal(Cbad[0], table)


def test_worked_example_shifted_row_is_caught(oracle_mod):
    _, table = load_worked_example()
    A, B = worked_example_operands(0)
    # an off-by-one row index: start A one row later (rows 1..16, 16 wraps to 0)
    A2 = np.concatenate([A[16:], A[:16]])
    Cbad, _ = oracle_mod.gemm(A2, B, 0, 16, 8, 16, 16, 8)
    assert not np.array_equal(Cbad[0], table)


# ---------------------------------------------------------------- counts

def load_counts():
    d = {}
    with open(os.path.join(GOLDEN, "gemm_counts_4096.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            k, v = line.split()
            d[k] = float(v)
    return d


def test_printed_counts(oracle_mod):
    c = load_counts()
    M, N, K = int(c["M"]), int(c["N"]), int(c["K"])
    fl = oracle_mod.flops(M, N, K)
    assert fl == 137438953472
    assert round(fl / 1e9, 1) == c["flops_gflop_printed"]
    by = oracle_mod.min_bytes(M, N, K, 2, 2)
    assert by == 100663296
    assert by / 2**20 == c["min_bytes_mib_printed"]
    assert round(by / 1e6, 1) == c["min_bytes_mb_printed"]
    assert round(fl / by) == c["intensity_printed"]
    assert oracle_mod.flops(16, 8, 16) == c["mma_m16n8k16_flop"]
    assert oracle_mod.flops(16, 8, 16) // 2 == c["mma_m16n8k16_fma"]


# ---------------------------------------------------------------- decoders

@pytest.mark.parametrize("dtype", [0, 1])
def test_decoder_all_patterns(oracle_mod, dtype):
    allb = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    mine = oracle_mod.decode(allb, dtype)
    ref = lib_decode(allb, dtype)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(mine), nan)
    assert np.array_equal(mine[~nan], ref[~nan])
    # signed zeros decode with their sign
    assert np.array_equal(np.signbit(mine[~nan]), np.signbit(ref[~nan]))


def test_decoder_special_values(oracle_mod):
    d = oracle_mod.decode_one
    assert d(0x0001, 0) == 2.0 ** -24          # smallest fp16 subnormal
    assert d(0x03FF, 0) == 1023 * 2.0 ** -24   # largest fp16 subnormal
    assert d(0x0400, 0) == 2.0 ** -14          # smallest fp16 normal
    assert d(0x7BFF, 0) == 65504.0             # largest fp16
    assert d(0x3C00, 0) == 1.0 and d(0xBC00, 0) == -1.0
    assert d(0x0001, 1) == 2.0 ** -133         # smallest bf16 subnormal
    assert d(0x3F80, 1) == 1.0 and d(0xC000, 1) == -2.0
    assert d(0x7F7F, 1) == float.fromhex("0x1.fep127")
    assert math.isinf(d(0x7C00, 0)) and math.isinf(d(0x7F80, 1))


# ---------------------------------------------------------------- exact sums

SHAPES = [(1, 1, 1), (2, 7, 8), (7, 2, 15), (8, 16, 17), (15, 8, 31), (16, 17, 33),
          (17, 31, 16), (31, 33, 7), (33, 15, 2), (127, 1, 128), (1, 129, 255), (128, 127, 1)]


def exact_fsum(Ad, Bd):
    """Correctly rounded exact product: each product is exact in binary64."""
    M, K = Ad.shape
    N = Bd.shape[1]
    out = np.empty((M, N))
    for i in range(M):
        prods = Ad[i][:, None] * Bd  # K x N, every entry exact
        for j in range(N):
            out[i, j] = math.fsum(prods[:, j])
    return out


@pytest.mark.parametrize("dtype", [0, 1])
@pytest.mark.parametrize("shape", SHAPES)
def test_bruteforce_fsum(oracle_mod, dtype, shape):
    M, N, K = shape
    seed = 1000 + M * 7 + N * 13 + K
    dname = "f16" if dtype == 0 else "bf16"
    A = bits(inputs.make_random((M, K), dname, seed, "normal"))
    B = bits(inputs.make_random((K, N), dname, seed + 1, "uniform"))
    Cref, Den = oracle_mod.gemm(A, B, dtype, M, N, K, K, N)
    ex = exact_fsum(lib_decode(A, dtype).reshape(M, K), lib_decode(B, dtype).reshape(K, N))
    bound = K * 2.0 ** -53 * Den[0] * 1.0001 + 1e-300
    assert np.all(np.abs(Cref[0] - ex) <= bound)
    # Den is the sum of |products|: compare with numpy on the absolute values
    Ad, Bd = lib_decode(A, dtype).reshape(M, K), lib_decode(B, dtype).reshape(K, N)
    dref = np.abs(Ad) @ np.abs(Bd)
    assert np.allclose(Den[0], dref, rtol=1e-13, atol=0)
    assert np.all(np.abs(Cref[0]) <= Den[0] * (1 + 1e-12))


@pytest.mark.parametrize("dtype", [0, 1])
def test_bruteforce_fraction(oracle_mod, dtype):
    """Exact rationals on a tiny product with odd leading dimensions and a
    batch stride: every stride and offset is exercised."""
    M, N, K, batch = 3, 5, 7, 2
    lda, ldb, sA, sB = K + 3, N + 2, 40, 60
    rng = np.random.default_rng(7 + dtype)
    dname = "f16" if dtype == 0 else "bf16"
    A = bits(inputs.make_random((batch * sA,), dname, 11 + dtype, "normal"))
    B = bits(inputs.make_random((batch * sB,), dname, 12 + dtype, "normal"))
    Cref, Den = oracle_mod.gemm(A, B, dtype, M, N, K, lda, ldb, batch, sA, sB)
    Ad, Bd = lib_decode(A, dtype), lib_decode(B, dtype)
    for b in range(batch):
        for i in range(M):
            for j in range(N):
                s = sum(Fraction(Ad[b * sA + i * lda + k]) * Fraction(Bd[b * sB + k * ldb + j])
                        for k in range(K))
                d = sum(abs(Fraction(Ad[b * sA + i * lda + k]) * Fraction(Bd[b * sB + k * ldb + j]))
                        for k in range(K))
                assert abs(Fraction(Cref[b, i, j]) - s) <= Fraction(K) * Fraction(2) ** -53 * d
                assert abs(Fraction(Den[b, i, j]) - d) <= Fraction(K) * Fraction(2) ** -53 * d
    del rng


def test_dropped_term_is_caught(oracle_mod):
    """Summing one term fewer (K-1) must disagree with the exact sum."""
    M, N, K = 8, 8, 17
    A = bits(inputs.make_random((M, K), "f16", 5, "uniform"))
    B = bits(inputs.make_random((K, N), "f16", 6, "uniform"))
    ex = exact_fsum(lib_decode(A, 0).reshape(M, K), lib_decode(B, 0).reshape(K, N))
    Cbad, Dbad = oracle_mod.gemm(A, B, 0, M, N, K - 1, K, N)
    assert np.any(np.abs(Cbad[0] - ex) > K * 2.0 ** -53 * Dbad[0] + 1e-300)


def test_sign_flip_is_caught(oracle_mod):
    """A sign slip in one operand changes every non-zero entry."""
    M, N, K = 4, 4, 9
    A = bits(inputs.make_random((M, K), "bf16", 8, "normal"))
    B = bits(inputs.make_random((K, N), "bf16", 9, "normal"))
    Cref, _ = oracle_mod.gemm(A, B, 1, M, N, K, K, N)
    An = A ^ np.uint16(0x8000)
    Cneg, _ = oracle_mod.gemm(An, B, 1, M, N, K, K, N)
    assert np.array_equal(Cneg, -Cref)
    ex = exact_fsum(lib_decode(A, 1).reshape(M, K), lib_decode(B, 1).reshape(K, N))
    assert not np.allclose(Cneg[0], ex)


# ---------------------------------------------------------------- textbook cases

@pytest.mark.parametrize("dtype", [0, 1])
def test_identity(oracle_mod, dtype):
    M = K = N = 33
    dname = "f16" if dtype == 0 else "bf16"
    A = bits(inputs.make_random((M, K), dname, 21, "normal"))
    I = encode_exact(np.eye(K), dtype).reshape(-1)
    Cref, Den = oracle_mod.gemm(A, I, dtype, M, N, K, K, N)
    assert np.array_equal(Cref[0], lib_decode(A, dtype).reshape(M, K))
    assert np.array_equal(Den[0], np.abs(lib_decode(A, dtype).reshape(M, K)))


@pytest.mark.parametrize("dtype", [0, 1])
def test_one_hot_rows(oracle_mod, dtype):
    """A[i][k] = [k == i mod K]  =>  C[i][:] = B[i mod K][:] exactly."""
    M, N, K = 40, 24, 16
    dname = "f16" if dtype == 0 else "bf16"
    Av = np.zeros((M, K))
    for i in range(M):
        Av[i, i % K] = 1.0
    A = encode_exact(Av, dtype).reshape(-1)
    B = bits(inputs.make_random((K, N), dname, 22, "normal"))
    Cref, _ = oracle_mod.gemm(A, B, dtype, M, N, K, K, N)
    Bd = lib_decode(B, dtype).reshape(K, N)
    for i in range(M):
        assert np.array_equal(Cref[0, i], Bd[i % K])


def test_zeros_and_empty_sum(oracle_mod):
    A = np.zeros(6 * 5, dtype=np.uint16)
    B = bits(inputs.make_random((5, 4), "f16", 3, "normal"))
    Cref, Den = oracle_mod.gemm(A, B, 0, 6, 4, 5, 5, 4)
    assert np.all(Cref == 0) and np.all(Den == 0)
    # K = 0: the empty sum is zero
    Cref, Den = oracle_mod.gemm(np.zeros(1, np.uint16), np.zeros(1, np.uint16), 0, 3, 2, 0, 1, 2)
    assert Cref.shape == (1, 3, 2) and np.all(Cref == 0) and np.all(Den == 0)


def test_integer_data_is_exact(oracle_mod):
    """The 512^3 integer workload recipe on a smaller shape: integers in
    [-4, 4] give exact sums in any order, equal to numpy's int64 matmul."""
    M, N, K = 64, 48, 512
    A = inputs.make_random((M, K), "f16", 0, "int4")
    B = inputs.make_random((K, N), "f16", 1, "int4")
    Cref, Den = oracle_mod.gemm(bits(A), bits(B), 0, M, N, K, K, N)
    Ai = A.float().numpy().astype(np.int64)
    Bi = B.float().numpy().astype(np.int64)
    assert Ai.min() >= -4 and Ai.max() <= 4 and len(np.unique(Ai)) == 9
    assert np.array_equal(Cref[0], (Ai @ Bi).astype(np.float64))
    assert np.array_equal(Den[0], (np.abs(Ai) @ np.abs(Bi)).astype(np.float64))


# ---------------------------------------------------------------- entries / threads

def test_entries_match_full(oracle_mod):
    M, N, K, batch = 37, 29, 45, 3
    sA, sB = M * K + 5, K * N + 3
    A = bits(inputs.make_random((batch * sA,), "bf16", 31, "normal"))
    B = bits(inputs.make_random((batch * sB,), "bf16", 32, "normal"))
    Cref, Den = oracle_mod.gemm(A, B, 1, M, N, K, K, N, batch, sA, sB)
    rng = np.random.default_rng(0)
    eb = rng.integers(0, batch, 200)
    ei = rng.integers(0, M, 200)
    ej = rng.integers(0, N, 200)
    c, d = oracle_mod.gemm_entries(A, B, 1, K, K, N, eb, ei, ej, sA, sB)
    assert np.array_equal(c, Cref[eb, ei, ej])
    assert np.array_equal(d, Den[eb, ei, ej])


def test_thread_count_does_not_change_result(oracle_mod):
    M, N, K = 50, 20, 300
    A = bits(inputs.make_random((M, K), "f16", 41, "uniform"))
    B = bits(inputs.make_random((K, N), "f16", 42, "uniform"))
    c1, d1 = oracle_mod.gemm(A, B, 0, M, N, K, K, N, threads=1)
    c8, d8 = oracle_mod.gemm(A, B, 0, M, N, K, K, N, threads=8)
    assert np.array_equal(c1, c8) and np.array_equal(d1, d8)


def test_fp16_uniform_exact_in_int64(oracle_mod):
    """U[-1,1] fp16 values are multiples of 2^-24 with |v| <= 1, so
    v * 2^24 are integers below 2^25: an int64 matmul of them is the exact
    product scaled by 2^48 for K up to 2^13."""
    M, N, K = 96, 80, 257
    A = bits(inputs.make_random((M, K), "f16", 51, "uniform"))
    B = bits(inputs.make_random((K, N), "f16", 52, "uniform"))
    Cref, Den = oracle_mod.gemm(A, B, 0, M, N, K, K, N)
    Ai = np.rint(lib_decode(A, 0) * 2.0 ** 24).astype(np.int64).reshape(M, K)
    Bi = np.rint(lib_decode(B, 0) * 2.0 ** 24).astype(np.int64).reshape(K, N)
    exact = (Ai @ Bi).astype(np.float64) * 2.0 ** -48  # int64 -> fp64 rounds once
    assert np.all(np.abs(Cref[0] - exact) <= (K + 1) * 2.0 ** -53 * Den[0])


# ---------------------------------------------------------------- acceptance measure

def test_normalized_error_semantics(oracle_mod):
    Cref = np.array([[[1.0, 0.0, -2.0]]])
    Den = np.array([[[2.0, 0.0, 4.0]]])
    assert oracle_mod.normalized_error(Cref.copy(), Cref, Den) == 0.0
    C = np.array([[[1.002, 0.0, -2.0]]])
    assert abs(oracle_mod.normalized_error(C, Cref, Den) - 0.001) < 1e-12
    C = np.array([[[1.0, 1e-30, -2.0]]])   # Den == 0 entry must be exactly zero
    assert oracle_mod.normalized_error(C, Cref, Den) == float("inf")
    C = np.array([[[float("nan"), 0.0, -2.0]]])
    assert oracle_mod.normalized_error(C, Cref, Den) == float("inf")


# ---------------------------------------------------------------- transposed B

@pytest.mark.parametrize("dtype", [0, 1])
def test_worked_example_with_b_stored_transposed(oracle_mod, dtype):
    """B given as its N x K transpose (B^T[j][k] = j) with a padded leading
    dimension still gives the worked example's D = 16 i j."""
    _, table = load_worked_example()
    A, B = worked_example_operands(dtype)
    Bkn = lib_decode(B, dtype).reshape(16, 8)
    ldb = 20
    Bs = np.zeros(8 * ldb, dtype=np.float64)
    for j in range(8):
        Bs[j * ldb:j * ldb + 16] = Bkn[:, j]
    Cref, Den = oracle_mod.gemm_bt(A, encode_exact(Bs, dtype), dtype, 16, 8, 16, 16, ldb)
    assert np.array_equal(Cref[0], table)


def test_transposed_b_batched_against_fsum(oracle_mod):
    """Batched C = A . Bs^T against math.fsum of the products read straight
    from the stored N x K layout."""
    rng = np.random.default_rng(11)
    M, N, K, batch, ldb, sB = 3, 5, 7, 2, 9, 50
    A = encode_exact(rng.integers(-4, 5, size=batch * M * K).astype(np.float64), 0)
    Bs = encode_exact(rng.integers(-4, 5, size=(batch - 1) * sB + N * ldb).astype(np.float64), 0)
    Cref, _ = oracle_mod.gemm_bt(A, Bs, 0, M, N, K, K, ldb, batch, M * K, sB)
    a, bs = lib_decode(A, 0), lib_decode(Bs, 0)
    for b in range(batch):
        for i in range(M):
            for j in range(N):
                want = math.fsum(a[b * M * K + i * K + k] * bs[b * sB + j * ldb + k] for k in range(K))
                assert Cref[b, i, j] == want


# ---------------------------------------------------------------- 8-bit inputs

FP8_TORCH = {2: "float8_e4m3fn", 3: "float8_e5m2"}


@pytest.mark.parametrize("dtype", [2, 3])
def test_fp8_decoder_all_patterns(oracle_mod, dtype):
    """The oracle's E4M3 / E5M2 decoders against PyTorch's float8 dtypes
    (an independent library decoder) on all 256 patterns; NaNs agree."""
    import torch
    b = np.arange(256, dtype=np.uint8)
    lib = torch.from_numpy(b).view(getattr(torch, FP8_TORCH[dtype])).float().double().numpy()
    got = oracle_mod.decode(oracle_mod.widen8(b), dtype)
    assert np.array_equal(np.isnan(got), np.isnan(lib))
    ok = ~np.isnan(lib)
    assert np.array_equal(got[ok], lib[ok])


def test_fp8_special_values(oracle_mod):
    """Extremes of the two formats: E4M3 has no infinity, max 448, smallest
    subnormal 2^-9; E5M2 max 57344, infinity at 0x7c, smallest subnormal
    2^-16."""
    d = oracle_mod.decode_one
    assert d(0x7E, 2) == 448.0 and d(0xFE, 2) == -448.0 and math.isnan(d(0x7F, 2))
    assert d(0x01, 2) == 2.0 ** -9 and d(0x08, 2) == 2.0 ** -6 and d(0x38, 2) == 1.0
    assert d(0x7B, 3) == 57344.0 and d(0x7C, 3) == math.inf and math.isnan(d(0x7D, 3))
    assert d(0x01, 3) == 2.0 ** -16 and d(0x3C, 3) == 1.0 and d(0xFC, 3) == -math.inf
    assert math.isnan(d(0x100, 2))  # not an 8-bit pattern


def test_worked_example_e4m3(oracle_mod):
    """The worked example (integers 0..15 are exact in E4M3) read as 8-bit
    inputs: D = 16 i j exactly."""
    import torch
    _, table = load_worked_example()
    A = torch.tensor([[float(i)] * 16 for i in range(16)]).to(torch.float8_e4m3fn)
    B = torch.tensor([[float(j) for j in range(8)] for _ in range(16)]).to(torch.float8_e4m3fn)
    a8 = A.view(torch.uint8).numpy().reshape(-1)
    b8 = B.view(torch.uint8).numpy().reshape(-1)
    Cref, Den = oracle_mod.gemm(oracle_mod.widen8(a8), oracle_mod.widen8(b8), 2, 16, 8, 16, 16, 8)
    assert np.array_equal(Cref[0], table) and np.array_equal(Den[0], table)


def test_fp8_product_against_fsum(oracle_mod):
    """A small E5M2 x E5M2 product against math.fsum of library-decoded values."""
    import torch
    g = torch.Generator().manual_seed(5)
    M, N, K = 4, 6, 9
    A = (torch.randn(M, K, generator=g) * 3).to(torch.float8_e5m2)
    B = (torch.randn(K, N, generator=g) * 3).to(torch.float8_e5m2)
    Cref, _ = oracle_mod.gemm(oracle_mod.widen8(A.view(torch.uint8).numpy().reshape(-1)),
                              oracle_mod.widen8(B.view(torch.uint8).numpy().reshape(-1)), 3, M, N, K, K, N)
    a, b = A.float().double().numpy(), B.float().double().numpy()
    for i in range(M):
        for j in range(N):
            assert Cref[0, i, j] == math.fsum(a[i, k] * b[k, j] for k in range(K))
