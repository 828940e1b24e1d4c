"""Parity of the CUDA path against the CPU oracle, through the C ABI.

Acceptance (fixed by the method's statement of the target):
  * integer-valued inputs whose sums are exact in fp32: bit-exact;
  * otherwise ``max |C - Cref| / Den <= 1e-3`` for fp32 output, ``<= 4e-3``
    for fp16 and ``<= 5e-3`` for bf16 output, with
    ``Den = sum_k |A_ik||B_kj|`` (entries with ``Den == 0`` must be exactly
    zero).
These are bounds, not fudge: fp32 accumulation of K products in any order is
within K * 2^-24 * Den (K * 2^-23 * Den if the hardware truncates; 9.8e-4 at
K = 8192) and rounding the result to fp16 / bf16 adds at most its unit
roundoff, 2^-11 / 2^-8 (11 / 8 significant bits), relative to |C| <= Den.

Small cases are compared element by element with the full oracle product;
the full-size workloads, in the launch configuration the bench times, are
compared on sampled entries the oracle computes one by one.
"""
import numpy as np
import pytest
import torch

import oracle
from tensor_core_dense_swizzled_gb300 import hgemm as H
from tensor_core_dense_swizzled_gb300 import inputs

pytestmark = pytest.mark.gpu

DT = {"f16": H.HGEMM_F16, "bf16": H.HGEMM_BF16, "f32": H.HGEMM_F32}
ORACLE_DT = {"f16": 0, "bf16": 1}
TOL = {"f32": 1e-3, "f16": 4e-3, "bf16": 5e-3}
# The target states 4e-3 for every 16-bit output.  For bf16 the arithmetic
# guarantees only 5e-3 at any K (its unit roundoff is 2^-8), so TOL keeps the
# provable bound; on the full-size workloads with 16-bit output the stated
# 4e-3 is asserted as well.
STATED_16BIT = 4e-3
TORCH = {"f16": torch.float16, "bf16": torch.bfloat16, "f32": torch.float32}


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    oracle.build()
    d = torch.device("cuda:0")
    torch.cuda.set_device(d)
    return d


def bits(t):
    return t.contiguous().cpu().view(torch.int16).numpy().view(np.uint16).reshape(-1)


def span(rows, cols, ld, batch, stride):
    if rows == 0 or cols == 0:
        return 0
    return (batch - 1) * stride + (rows - 1) * ld + cols


def read_c(flat_dev, dout, M, N, ldc, batch, sC, off):
    """Logical (batch, M, N) view of the device C buffer, as fp64 numpy read
    with the oracle's decoder for 16-bit outputs."""
    flat = flat_dev.cpu()
    view = torch.as_strided(flat, (batch, M, N), (sC, ldc, 1), off)
    if dout == "f32":
        return view.double().numpy()
    return oracle.decode(bits(view), ORACLE_DT[dout]).reshape(batch, M, N)


SENTINEL = {"f32": 12345.0, "f16": 1234.0, "bf16": 1234.0}


def run_case(dev, M, N, K, din, dout, *, lda=None, ldb=None, ldc=None, batch=1, sA=None,
             sB=None, sC=None, seed=0, dist_a="normal", dist_b="normal", scale_b=1.0,
             off_a=0, off_b=0, off_c=0, options=None, A_flat=None, B_flat=None, runs=1):
    lda = K if lda is None else lda
    ldb = N if ldb is None else ldb
    ldc = N if ldc is None else ldc
    sA = (M * lda if batch > 1 else 0) if sA is None else sA
    sB = (K * ldb if batch > 1 else 0) if sB is None else sB
    sC = (M * ldc if batch > 1 else 0) if sC is None else sC
    nA = off_a + max(span(M, K, lda, batch, sA), 1)
    nB = off_b + max(span(K, N, ldb, batch, sB), 1)
    nC = off_c + max(span(M, N, ldc, batch, sC), 1)
    if A_flat is None:
        A_flat = inputs.make_random((nA,), din, seed, dist_a)
    if B_flat is None:
        B_flat = inputs.make_random((nB,), din, seed + 1, dist_b, scale_b)
    dA = A_flat.to(dev)
    dB = B_flat.to(dev)
    tail = 64  # elements after the last row: must stay untouched too
    dC_full = torch.full((nC + tail,), SENTINEL[dout], dtype=TORCH[dout], device=dev)
    dC = dC_full[:nC]
    esz_in, esz_out = 2, dC.element_size()
    plan = H.hgemm_plan_create_ex(M, N, K, lda, ldb, ldc, batch, sA, sB, sC, DT[din], DT[dout],
                                  options)
    try:
        info = H.hgemm_plan_get_info(plan)
        outs = []
        for _ in range(runs):
            H.hgemm_run(plan, dA.data_ptr() + off_a * esz_in, dB.data_ptr() + off_b * esz_in,
                        dC.data_ptr() + off_c * esz_out)
            st = H.hgemm_check(plan)
            assert st == 0, f"hgemm_check: {H.STATUS.get(st)} {H.hgemm_last_error_detail()}"
            outs.append(dC.clone())
    finally:
        H.hgemm_plan_destroy(plan)
    Cref, Den = oracle.gemm(bits(A_flat)[off_a:], bits(B_flat)[off_b:], ORACLE_DT[din], M, N, K,
                            lda, ldb, batch, sA, sB)
    got = read_c(dC, dout, M, N, ldc, batch, sC, off_c)
    # elements of the C buffer outside the logical matrices are untouched
    mask = torch.ones(nC, dtype=torch.bool)
    if M and N:
        idx = torch.as_strided(torch.arange(nC), (batch, M, N), (sC, ldc, 1), off_c).reshape(-1)
        mask[idx] = False
    outside = dC.cpu()[mask]
    assert torch.all(outside == SENTINEL[dout]), "kernel wrote outside C"
    assert torch.all(dC_full[nC:].cpu() == SENTINEL[dout]), "kernel wrote past the end of C"
    for o in outs[1:]:
        assert torch.equal(o, outs[0]), "repeated runs differ"
    return got, Cref, Den, info


def check(got, Cref, Den, dout, exact=False):
    if exact:
        assert np.array_equal(got, Cref), f"max |diff| {np.max(np.abs(got - Cref))}"
        return 0.0
    err = oracle.normalized_error(got, Cref, Den)
    assert err <= TOL[dout], f"normalised error {err:.3e} > {TOL[dout]}"
    return err


# ---------------------------------------------------------------- worked example

@pytest.mark.parametrize("din", ["f16", "bf16"])
@pytest.mark.parametrize("dout", ["f32", "f16", "bf16"])
def test_worked_example(dev, din, dout):
    """A[i][k] = i, B[k][j] = j on a 16 x 8 x 16 tile gives D[i][j] = 16*i*j
    ("post_1787550000", section 6.1); every value is exact in every output
    type, so the result must match bit for bit."""
    A = torch.arange(16, dtype=torch.float32).repeat_interleave(16).to(TORCH[din])
    B = torch.arange(8, dtype=torch.float32).repeat(16).to(TORCH[din])
    got, Cref, Den, _ = run_case(dev, 16, 8, 16, din, dout, A_flat=A, B_flat=B)
    check(got, Cref, Den, dout, exact=True)
    assert got[0, 3, 5] == 240 and got[0, 15, 7] == 1680


@pytest.mark.parametrize("path", [H.HGEMM_PATH_TILED, H.HGEMM_PATH_SKINNY])
def test_worked_example_both_paths(dev, path):
    A = torch.arange(16, dtype=torch.float32).repeat_interleave(16).to(torch.float16)
    B = torch.arange(8, dtype=torch.float32).repeat(16).to(torch.float16)
    got, Cref, Den, info = run_case(dev, 16, 8, 16, "f16", "f32", A_flat=A, B_flat=B,
                                    options=H.Options(force_path=path))
    assert info["path"] == path
    check(got, Cref, Den, "f32", exact=True)


# ---------------------------------------------------------------- layout locators

@pytest.mark.parametrize("din", ["f16", "bf16"])
@pytest.mark.parametrize("tile_n", [128, 192, 224, 256])
def test_identity_B_returns_A(dev, din, tile_n):
    """B = I: C must equal A exactly (fp32 out).  A wrong descriptor stride,
    swizzle or major-ness scrambles rows or columns of C."""
    M = K = N = 320
    A = inputs.make_random((M * K,), din, 3)
    B = torch.eye(K, dtype=torch.float32).reshape(-1).to(TORCH[din])
    got, Cref, Den, _ = run_case(dev, M, N, K, din, "f32", A_flat=A, B_flat=B,
                                 options=H.Options(tile_n=tile_n))
    check(got, Cref, Den, "f32", exact=True)


@pytest.mark.parametrize("din", ["f16", "bf16"])
@pytest.mark.parametrize("dout", ["f32", "bf16"])
@pytest.mark.parametrize("pn", [256, 224])
def test_identity_B_returns_A_on_cta_pairs(dev, din, dout, pn):
    """The same locator on 256 x 256 tiles computed by CTA pairs: each CTA
    holds half of B's columns and half of the accumulator rows, so a wrong
    half split shows up as swapped or zeroed column/row blocks."""
    M, K, N = 640, 320, 576
    A = inputs.make_random((M * K,), din, 23)
    B = torch.eye(K, N, dtype=torch.float32).reshape(-1).to(TORCH[din])
    got, Cref, Den, info = run_case(dev, M, N, K, din, dout, A_flat=A, B_flat=B,
                                    options=H.Options(cta_pair=1, tile_n=pn))
    assert info["tile_m"] == 256 and info["tile_n"] == pn
    check(got, Cref, Den, dout, exact=(dout == "f32"))


@pytest.mark.parametrize("shape", [(256, 256, 64), (300, 520, 200), (513, 700, 1000), (1024, 768, 2048),
                                   (2560, 2304, 256), (130, 260, 70), (384, 512, 130), (512, 512, 320)])
@pytest.mark.parametrize("din,dout", [("bf16", "bf16"), ("f16", "f32"), ("f16", "f16")])
@pytest.mark.parametrize("pn", [256, 224])
@pytest.mark.parametrize("ks", [1, 2])
def test_cta_pair_random_shapes(dev, shape, din, dout, pn, ks):
    """ks = K blocks per pipeline stage; with 2, an odd number of 64-wide K
    blocks leaves the last stage with one (130 and 320 have 3 and 5)."""
    M, N, K = shape
    got, Cref, Den, info = run_case(dev, M, N, K, din, dout, seed=M + 2 * N + K,
                                    options=H.Options(cta_pair=1, tile_n=pn, pair_k_blocks=ks))
    assert info["tile_m"] == 256 and info["grid"] % 2 == 0 and info["tile_k"] == 64 * ks
    # one TMA copy per operand per stage exactly when the 4-D views apply: K
    # and N multiples of 64, or the operand read from its zero-padded copy
    assert info["wide_boxes"] == int(pn == 256 and (K % 64 == 0 or info["repack_a"] == 1)
                                     and (N % 64 == 0 or info["repack_b"] == 1))
    check(got, Cref, Den, dout)


@pytest.mark.parametrize("shape", [(600, 333, 333, 2, 0), (1100, 777, 1023, 1, 0), (520, 640, 200, 1, 3),
                                   (300, 4095, 130, 1, 0)])
@pytest.mark.parametrize("din,dout", [("f16", "f32"), ("bf16", "bf16")])
def test_cta_pair_views_over_padded_copies(dev, shape, din, dout):
    """Operands read from their aligned copies: the copies' rows are padded
    with zeros to whole 64-element blocks, and the pair kernel views them over
    the padded extent (one TMA copy per operand per stage) even though K or N
    is not a multiple of 64.  off_a > 0 puts A's base off the 16-byte grid
    (a copy made at run time)."""
    M, N, K, batch, off_a = shape
    got, Cref, Den, info = run_case(dev, M, N, K, din, dout, batch=batch, off_a=off_a,
                                    seed=M + N + K, options=H.Options(cta_pair=1), runs=2)
    assert info["tile_m"] == 256
    check(got, Cref, Den, dout)


@pytest.mark.parametrize("opt", [H.Options(cta_pair=1, force_generic_store=1),
                                 H.Options(cta_pair=1, force_repack=1)])
def test_cta_pair_fallback_paths(dev, opt):
    M, N, K = 333, 444, 222
    got, Cref, Den, _ = run_case(dev, M, N, K, "bf16", "f32", seed=24, options=opt, runs=2)
    check(got, Cref, Den, "f32")


@pytest.mark.parametrize("shape", [(2560, 2048, 256, 1), (4096, 2048, 192, 1), (2304, 2304, 130, 1),
                                   (1280, 2048, 256, 2), (2560, 2000, 320, 1)])
@pytest.mark.parametrize("dout", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("ks", [1, 2])
def test_cta_pair_stream_k(dev, shape, dout, ks):
    """At least one full wave of pair tiles but not a whole number of waves:
    the tiles' K steps are dealt to the pairs in equal contiguous ranges, so
    some tiles are cut between two pairs (one spills its partial first, the
    other adds it and stores).  80, 128 and 81 tiles of 256 x 256 on about 76
    pairs; K = 130 leaves an odd number of 64-wide K blocks; the batched case
    cuts tiles across batch entries; N = 2000 is not a multiple of 64 (box-by-
    box loads).  Three runs in a row must agree bit for bit."""
    M, N, K, batch = shape
    got, Cref, Den, info = run_case(dev, M, N, K, "bf16", dout, batch=batch, seed=M + N + K + 11,
                                    options=H.Options(cta_pair=1, pair_k_blocks=ks, tail_mode=3),
                                    runs=3)
    assert info["tile_m"] == 256 and info["stream_k"] == 1 and info["tail_split"] == 1
    check(got, Cref, Den, dout)


@pytest.mark.parametrize("shape", [(1536, 2560, 512, 1), (1536, 2048, 320, 1), (2048, 2048, 256, 1),
                                   (1500, 2000, 700, 1), (768, 2048, 512, 2)])
@pytest.mark.parametrize("dout", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("ks", [1, 2])
def test_cta_pair_first_wave_dealing(dev, shape, dout, ks):
    """tail_mode 4: the K steps of the tiles that do not fill a wave (here
    all 48 to 64 tiles) are dealt to all pairs first; a tile cut into up to
    four pieces on consecutive pairs is summed, in piece order, by the piece
    that arrives last.  K = 320 and 700 leave a last stage of one K block;
    N = 2000 is not a multiple of 64 (box-by-box loads); the batched case
    deals across batch entries.  Three runs must agree bit for bit (the
    counters reset, the sum order is fixed)."""
    M, N, K, batch = shape
    got, Cref, Den, info = run_case(dev, M, N, K, "bf16", dout, batch=batch, seed=M + N + K + 13,
                                    options=H.Options(cta_pair=1, pair_k_blocks=ks, tail_mode=4),
                                    runs=3)
    assert info["tile_m"] == 256 and info["stream_k"] == 2
    check(got, Cref, Den, dout)


@pytest.mark.parametrize("shape", [(512, 1024, 512), (300, 520, 200), (1024, 768, 96), (640, 1000, 333),
                                   (512, 768, 130), (256, 512, 192), (2560, 2048, 256), (4096, 4096, 128)])
@pytest.mark.parametrize("dout", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("ks", [1, 2])
def test_cta_pair_split_tail(dev, shape, dout, ks):
    """Fewer pair tiles than half the pairs: every tile is a tail tile whose two
    K halves run on two pairs and meet in the two-arriver fixup.  Three runs
    in a row must agree bit for bit (counters and flags reset, and the
    two-term sum does not depend on which half arrives first).  The halves
    split the tile's pipeline stages (ks K blocks each); a tile of one stage
    is not split.  With more tiles than pairs (80 and 256 tiles on about 76
    pairs) the halves of the few left-over tiles run first, whole tiles after."""
    M, N, K = shape
    got, Cref, Den, info = run_case(dev, M, N, K, "bf16", dout, seed=M + N + K + 7,
                                    options=H.Options(cta_pair=1, pair_k_blocks=ks), runs=3)
    steps = -(-(-(-K // 64)) // ks)
    assert info["tile_m"] == 256 and info["tail_split"] == (2 if steps >= 2 else 1)
    check(got, Cref, Den, dout)


@pytest.mark.parametrize("opt", [H.Options(cta_pair=1, force_generic_store=1),
                                 H.Options(cta_pair=1, no_tail_split=1)])
def test_cta_pair_split_tail_variants(dev, opt):
    M, N, K = 520, 700, 300
    got, Cref, Den, info = run_case(dev, M, N, K, "f16", "f16", seed=31, options=opt, runs=2)
    assert info["tail_split"] == (1 if opt.no_tail_split else 2)
    check(got, Cref, Den, "f16")


def test_cta_pair_single_k_block_is_not_split(dev):
    got, Cref, Den, info = run_case(dev, 512, 512, 64, "bf16", "f32", seed=32,
                                    options=H.Options(cta_pair=1))
    assert info["tail_split"] == 1
    check(got, Cref, Den, "f32")


def test_cta_pair_batched(dev):
    M, N, K, batch = 300, 260, 96, 3
    got, Cref, Den, info = run_case(dev, M, N, K, "bf16", "f32", batch=batch, seed=25,
                                    options=H.Options(cta_pair=1))
    check(got, Cref, Den, "f32")


def test_cta_pair_int_exact(dev):
    M, N, K = 512, 512, 512
    A = inputs.make_random((M * K,), "f16", 0, "int4")
    B = inputs.make_random((K * N,), "f16", 1, "int4")
    got, Cref, Den, _ = run_case(dev, M, N, K, "f16", "f32", A_flat=A, B_flat=B,
                                 options=H.Options(cta_pair=1))
    check(got, Cref, Den, "f32", exact=True)


@pytest.mark.parametrize("din", ["f16", "bf16"])
def test_one_hot_rows(dev, din):
    """A[i][k] = [k == i mod K]: row i of C is row (i mod K) of B exactly."""
    M, N, K = 256, 384, 192
    A = torch.zeros(M, K)
    A[torch.arange(M), torch.arange(M) % K] = 1.0
    B = inputs.make_random((K * N,), din, 4)
    got, Cref, Den, _ = run_case(dev, M, N, K, din, "f32", A_flat=A.reshape(-1).to(TORCH[din]),
                                 B_flat=B)
    check(got, Cref, Den, "f32", exact=True)


# ---------------------------------------------------------------- integer workload

def test_int512_bit_exact(dev):
    """512^3 fp16 integers in [-4, 4] (seed 0), fp32 out: every partial sum is
    an integer below 2^24, so any summation order is exact."""
    w = inputs.WORKLOADS["int512"]
    A, B = inputs.make_inputs(w)
    got, Cref, Den, info = run_case(dev, w.M, w.N, w.K, w.dtype_in, w.dtype_out,
                                    A_flat=A.reshape(-1), B_flat=B.reshape(-1))
    assert info["path"] == H.HGEMM_PATH_TILED
    check(got, Cref, Den, "f32", exact=True)


@pytest.mark.parametrize("dout", ["f16", "bf16"])
def test_int_small_exact_16bit_out(dev, dout):
    """Small integer products whose results fit the output format exactly."""
    M, N, K = 200, 136, 24  # |C| <= 24*16 = 384: an integer, exact in fp16 (not always in bf16)
    A = inputs.make_random((M * K,), "f16", 9, "int4")
    B = inputs.make_random((K * N,), "f16", 10, "int4")
    got, Cref, Den, _ = run_case(dev, M, N, K, "f16", dout, A_flat=A, B_flat=B)
    if dout == "f16":
        check(got, Cref, Den, dout, exact=True)
    else:
        check(got, Cref, Den, dout)


# ---------------------------------------------------------------- random ragged shapes

SHAPES = [(33, 40, 17), (128, 256, 64), (129, 257, 65), (300, 520, 200), (511, 383, 130),
          (256, 512, 1024), (640, 1000, 333), (1024, 768, 2048)]


@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("din,dout", [("bf16", "bf16"), ("f16", "f32"), ("bf16", "f32"),
                                      ("f16", "f16")])
def test_random_shapes(dev, shape, din, dout):
    M, N, K = shape
    got, Cref, Den, info = run_case(dev, M, N, K, din, dout, seed=M + N + K)
    assert info["path"] == H.HGEMM_PATH_TILED
    check(got, Cref, Den, dout)


@pytest.mark.parametrize("tile_n", [128, 192, 224, 256])
@pytest.mark.parametrize("dout", ["f32", "bf16", "f16"])
def test_tile_variants(dev, tile_n, dout):
    M, N, K = 390, 700, 300
    got, Cref, Den, info = run_case(dev, M, N, K, "bf16", dout, seed=5,
                                    options=H.Options(tile_n=tile_n))
    assert info["tile_n"] == tile_n
    check(got, Cref, Den, dout)


@pytest.mark.parametrize("ew", [4, 8])
@pytest.mark.parametrize("tile_n", [128, 256])
@pytest.mark.parametrize("dout,generic", [("f32", False), ("bf16", False), ("f16", True), ("f32", True)])
def test_tiled_epilogue_warps(dev, ew, tile_n, dout, generic):
    """Four or eight epilogue warps on the single-CTA kernel (eight: two warps
    per TMEM lane quarter, each storing half of a tile's 32-column chunks).
    More tiles than SMs, so both accumulators and the stage ring wrap; ragged
    M and N edges; TMA or predicated stores."""
    M, N, K = 2900, 1904, 200  # rows of 16-bit C end on 16 bytes (TMA stores apply)
    got, Cref, Den, info = run_case(dev, M, N, K, "bf16", dout, seed=ew + tile_n,
                                    options=H.Options(cta_pair=2, tile_n=tile_n, tiled_epi_warps=ew,
                                                      force_generic_store=int(generic)), runs=2)
    assert info["epi_warps"] == ew and info["tile_n"] == tile_n and info["tma_store"] == int(not generic)
    assert info["grid"] < ((M + 127) // 128) * ((N + tile_n - 1) // tile_n)
    check(got, Cref, Den, dout)


def test_tiled_epilogue_warps_choice_and_refusals(dev):
    # automatic: four for plain runs; with the fused epilogue eight for few
    # K blocks, four for long K (main loop bound)
    for K, want in [(128, 8), (1024, 8), (1088, 4)]:
        plan = H.hgemm_plan_create_ex(1024, 1024, K, K, 1024, 1024, 1, 0, 0, 0, DT["bf16"], DT["bf16"],
                                      H.Options(cta_pair=2, tile_n=256))
        try:
            info = H.hgemm_plan_get_info(plan)
            assert info["epi_warps"] == 4 and info["epi_warps_epilogue"] == want, K
        finally:
            H.hgemm_plan_destroy(plan)
    for opt, status in [(H.Options(cta_pair=2, tile_n=192, tiled_epi_warps=8), 2),
                        (H.Options(cta_pair=2, tiled_epi_warps=5), 1)]:
        with pytest.raises(H.HgemmError) as ei:
            H.hgemm_plan_create_ex(512, 512, 256, 256, 512, 512, 1, 0, 0, 0, DT["bf16"], DT["bf16"], opt)
        assert ei.value.status == status
    # 8-bit inputs keep four epilogue warps
    with pytest.raises(H.HgemmError) as ei:
        H.hgemm_plan_create_ex(512, 512, 256, 256, 256, 512, 1, 0, 0, 0, H.HGEMM_E4M3, DT["bf16"],
                               H.Options(cta_pair=2, tile_n=256, trans_b=1, tiled_epi_warps=8))
    assert ei.value.status == 2


def test_many_tiles_per_cta(dev):
    """More tiles than SMs: every CTA loops, both TMEM buffers and the stage
    ring wrap many times."""
    M, N, K = 2560, 2304, 256
    got, Cref, Den, info = run_case(dev, M, N, K, "f16", "f16", seed=6)
    assert info["grid"] < (M // 128) * (N // 256)  # 180 tiles
    check(got, Cref, Den, "f16")


# ---------------------------------------------------------------- strides, alignment, batches

@pytest.mark.parametrize("dout", ["f32", "f16"])
def test_padded_leading_dimensions(dev, dout):
    M, N, K = 200, 300, 150
    got, Cref, Den, info = run_case(dev, M, N, K, "f16", dout, lda=K + 50, ldb=N + 20,
                                    ldc=N + 12, seed=11)  # 200, 320, 312: 16-byte rows
    assert not info["repack_a"] and not info["repack_b"]
    check(got, Cref, Den, dout)


@pytest.mark.parametrize("N,ldc,dout", [(300, 312, "f16"), (300, 304, "bf16"), (258, 272, "f32"),
                                         (260, 272, "f16"), (296, 312, "f16"), (260, 272, "f32")])
def test_row_end_not_on_16_bytes(dev, N, ldc, dout):
    """A TMA store writes whole 16-byte chunks, so a row whose length is not a
    multiple of 16 bytes must not take the TMA-store epilogue: nothing after
    column N-1 (nor past the last row) may change."""
    M, K = 200, 96
    got, Cref, Den, info = run_case(dev, M, N, K, "f16", dout, ldc=ldc, seed=N + ldc)
    ob = 4 if dout == "f32" else 2
    assert info["tma_store"] == (1 if (N * ob) % 16 == 0 else 0)
    check(got, Cref, Den, dout)


@pytest.mark.parametrize("dout", ["f32", "f16", "bf16"])
def test_misaligned_leading_dimensions(dev, dout):
    """Odd leading dimensions: A and B are copied to aligned workspace and C
    is written with predicated stores."""
    M, N, K = 255, 257, 129
    din = "bf16" if dout == "bf16" else "f16"
    got, Cref, Den, info = run_case(dev, M, N, K, din, dout, lda=K, ldb=N, ldc=N, seed=12)
    assert info["repack_a"] and info["repack_b"] and not info["tma_store"]
    check(got, Cref, Den, dout)


def test_misaligned_base_pointers(dev):
    """Aligned leading dimensions but base pointers off by one element."""
    M, N, K = 256, 264, 136
    got, Cref, Den, _ = run_case(dev, M, N, K, "bf16", "f32", off_a=1, off_b=3, off_c=1, seed=13)
    check(got, Cref, Den, "f32")


@pytest.mark.parametrize("off", range(8))
def test_operand_copy_every_misalignment(dev, off):
    """The aligned copy reads whole 16-byte granules and shifts them: every
    start offset 0..7 elements, odd leading dimensions (so the offset changes
    from row to row), rows shorter than a granule, and rows of several
    1024-element segments (each copied by its own warp, which takes the
    granule after its segment from memory)."""
    for (M, N, K) in [(45, 29, 37), (130, 7, 3), (9, 300, 1), (9, 1100, 2501)]:
        got, Cref, Den, info = run_case(dev, M, N, K, "f16", "f32", lda=K, ldb=N, ldc=N,
                                        off_a=off, off_b=(off * 3) % 8, seed=100 + off + K,
                                        options=H.Options(force_path=H.HGEMM_PATH_TILED))
        assert info["repack_a"] or K % 8 != 0 or off != 0
        check(got, Cref, Den, "f32")


PAIR_COPY_CASES = [
    # M, N, K, kwargs: copies of A only, B only, both, B stored N x K, batches
    # with misaligned strides, K of one, several and a partial 1024-element
    # copy segment
    (300, 520, 600, dict(lda=600, ldb=521, ldc=520)),
    (513, 700, 2500, dict(lda=2500, ldb=700, ldc=701)),
    (1000, 1100, 4095, dict(lda=4095, ldb=1100, ldc=1100)),
    (600, 640, 1500, dict(off_a=1)),
    (600, 640, 1500, dict(off_b=5)),
    (260, 300, 2100, dict(lda=2101, ldb=2101, trans_b=True)),
    (270, 260, 1100, dict(batch=2, sA=270 * 1100 + 3, sB=1100 * 260 + 1, sC=270 * 260)),
]


@pytest.mark.parametrize("case", range(len(PAIR_COPY_CASES)))
@pytest.mark.parametrize("dout", ["f32", "f16"])
def test_cta_pair_on_copied_operands(dev, case, dout):
    """CTA pairs reading operands from their aligned copies (misaligned leading
    dimension, base pointer or batch stride): the result matches the oracle
    and three runs in a row agree bit for bit."""
    M, N, K, kw = PAIR_COPY_CASES[case]
    kw = dict(kw)
    tb = kw.pop("trans_b", False)
    opt = H.Options(cta_pair=1, trans_b=1 if tb else 0)
    if tb:
        got, Cref, Den, info = run_case_bt(dev, M, N, K, dout, opt, seed=300 + case, **kw)
    else:
        got, Cref, Den, info = run_case(dev, M, N, K, "f16", dout, seed=300 + case, options=opt,
                                        runs=3, **kw)
    assert info["tile_m"] == 256
    assert info["repack_a"] or info["repack_b"] or "off_a" in kw or "off_b" in kw
    check(got, Cref, Den, dout)


def run_case_bt(dev, M, N, K, dout, opt, *, lda, ldb, seed):
    """C = A . B_stored^T with B stored N x K (ldb >= K), through run_case's
    machinery: the oracle gets B transposed into K x N."""
    A = inputs.make_random((M * lda,), "f16", seed, "normal")
    Bs = inputs.make_random((N * ldb,), "f16", seed + 1, "normal")
    dA, dB = A.to(dev), Bs.to(dev)
    dC = torch.full((M * N + 64,), SENTINEL[dout], dtype=TORCH[dout], device=dev)
    plan = H.hgemm_plan_create_ex(M, N, K, lda, ldb, N, 1, 0, 0, 0, H.HGEMM_F16, DT[dout], opt)
    try:
        info = H.hgemm_plan_get_info(plan)
        res = []
        for _ in range(3):
            H.hgemm_run(plan, dA.data_ptr(), dB.data_ptr(), dC.data_ptr())
            assert H.hgemm_check(plan) == 0, H.hgemm_last_error_detail()
            res.append(dC.clone())
    finally:
        H.hgemm_plan_destroy(plan)
    for r in res[1:]:
        assert torch.equal(r, res[0]), "repeated runs differ"
    assert torch.all(dC[M * N:].cpu() == SENTINEL[dout])
    Bkn = torch.as_strided(Bs, (N, K), (ldb, 1)).t().contiguous().reshape(-1)
    Cref, Den = oracle.gemm(bits(torch.as_strided(A, (M, K), (lda, 1)).contiguous().reshape(-1)),
                            bits(Bkn), 0, M, N, K, K, N, 1, 0, 0)
    got = read_c(dC[:M * N], dout, M, N, N, 1, 0, 0)
    return got, Cref, Den, info


@pytest.mark.parametrize("opt", [H.Options(force_repack=1), H.Options(force_generic_store=1),
                                 H.Options(force_repack=1, force_generic_store=1)])
def test_forced_fallbacks_match(dev, opt):
    M, N, K = 333, 444, 222
    got, Cref, Den, _ = run_case(dev, M, N, K, "bf16", "bf16", seed=14, options=opt)
    check(got, Cref, Den, "bf16")


@pytest.mark.parametrize("dout", ["f32", "bf16"])
def test_batched_strided(dev, dout):
    M, N, K, batch = 130, 200, 96, 5
    lda, ldb, ldc = K + 8, N + 16, N + 8
    sA, sB, sC = M * lda + 64, K * ldb + 8, M * ldc + 24
    got, Cref, Den, _ = run_case(dev, M, N, K, "bf16", dout, lda=lda, ldb=ldb, ldc=ldc, batch=batch,
                                 sA=sA, sB=sB, sC=sC, seed=15)
    check(got, Cref, Den, dout)


def test_batched_misaligned_strides(dev):
    M, N, K, batch = 70, 90, 50, 3
    got, Cref, Den, info = run_case(dev, M, N, K, "f16", "f32", batch=batch,
                                    sA=M * K + 1, sB=K * N + 3, sC=M * N + 1, seed=16)
    assert info["repack_a"] and info["repack_b"]
    check(got, Cref, Den, "f32")


def test_batch_stride_zero_broadcasts_B(dev):
    """strideB = 0 reuses one B for every batch."""
    M, N, K, batch = 128, 256, 64, 4
    got, Cref, Den, _ = run_case(dev, M, N, K, "bf16", "f32", batch=batch, sB=0, seed=17)
    check(got, Cref, Den, "f32")


# ---------------------------------------------------------------- degenerate sizes

@pytest.mark.parametrize("dout", ["f32", "f16", "bf16"])
def test_k_zero_writes_zeros(dev, dout):
    got, Cref, Den, info = run_case(dev, 37, 53, 0, "f16", dout, lda=1, ldb=53)
    assert info["path"] == H.HGEMM_PATH_ZERO_FILL
    assert np.all(got == 0)
    check(got, Cref, Den, dout, exact=True)


@pytest.mark.parametrize("M,N", [(0, 10), (10, 0), (0, 0)])
def test_empty_output_is_a_no_op(dev, M, N):
    got, Cref, Den, info = run_case(dev, M, N, 16, "f16", "f32", lda=16, ldb=max(N, 1),
                                    ldc=max(N, 1))
    assert info["path"] == H.HGEMM_PATH_EMPTY and info["kernels_per_run"] == 0


def test_zero_rows_give_exact_zeros(dev):
    """A zero row and a zero column make Den == 0 entries: they must be 0."""
    M, N, K = 150, 270, 80
    A = inputs.make_random((M * K,), "bf16", 18).reshape(M, K)
    A[7] = 0
    B = inputs.make_random((K * N,), "bf16", 19).reshape(K, N)
    B[:, 100] = 0
    got, Cref, Den, _ = run_case(dev, M, N, K, "bf16", "bf16", A_flat=A.reshape(-1),
                                 B_flat=B.reshape(-1))
    assert np.all(got[0, 7] == 0) and np.all(got[0, :, 100] == 0)
    check(got, Cref, Den, "bf16")


def test_single_element(dev):
    got, Cref, Den, _ = run_case(dev, 1, 1, 1, "f16", "f32", seed=20)
    check(got, Cref, Den, "f32")


def test_k_not_multiple_of_16(dev):
    for K in (1, 7, 15, 17, 63, 65):
        got, Cref, Den, _ = run_case(dev, 140, 130, K, "f16", "f32", lda=K + (-K) % 8,
                                     seed=21 + K)
        check(got, Cref, Den, "f32")


# ---------------------------------------------------------------- skinny path

@pytest.mark.parametrize("M", [1, 8, 16, 17, 32])
@pytest.mark.parametrize("dout", ["bf16", "f32"])
def test_skinny_shapes(dev, M, dout):
    N, K = 1000, 640
    got, Cref, Den, info = run_case(dev, M, N, K, "bf16", dout, seed=30 + M, scale_b=0.02)
    assert info["path"] == H.HGEMM_PATH_SKINNY
    check(got, Cref, Den, dout)


@pytest.mark.parametrize("split", [1, 2, 3, 5, 10])
def test_skinny_split_k(dev, split):
    M, N, K = 8, 777, 640
    got, Cref, Den, info = run_case(dev, M, N, K, "bf16", "bf16", seed=40,
                                    options=H.Options(split_k=split), runs=3)
    assert info["split_k"] == split
    check(got, Cref, Den, "bf16")


@pytest.mark.parametrize("cols", [128, 192, 256, 384, 512])
@pytest.mark.parametrize("M,N,K,split", [(8, 1000, 640, 3), (1, 5000, 1024, 4), (32, 700, 256, 1),
                                         (17, 4096, 512, 2), (8, 28672, 256, 1)])
def test_skinny_unit_widths(dev, cols, M, N, K, split):
    """Work units of 128 to 512 columns (ragged last unit included).  192 and
    384 columns are an odd number of 64-column blocks: the last MMA of a unit
    is half used, its other 64 rows are never stored."""
    got, Cref, Den, info = run_case(dev, M, N, K, "bf16", "bf16", seed=M + N + cols, scale_b=0.02,
                                    options=H.Options(skinny_tile_n=cols, split_k=split), runs=2)
    assert info["path"] == H.HGEMM_PATH_SKINNY and info["tile_n"] == cols
    check(got, Cref, Den, "bf16")


@pytest.mark.parametrize("cols", [128, 192, 256, 512])
@pytest.mark.parametrize("M,N,K,batch", [(8, 1000, 640, 1), (1, 5000, 1024, 1), (32, 700, 256, 1),
                                         (17, 4096, 512, 1), (8, 3000, 4096, 1), (4, 900, 320, 3),
                                         (8, 200, 64, 1)])
@pytest.mark.parametrize("dout", ["bf16", "f32"])
def test_skinny_stream_k(dev, cols, M, N, K, batch, dout):
    """Deal mode: the (tile, K block) steps are dealt to the SMs in equal
    contiguous ranges, so column tiles are cut into pieces on consecutive
    CTAs (up to `split_k` of them) and the last piece to arrive sums them in
    K order.  Covers batches (a range crossing batch entries), a single K
    block (no tile is cut), ragged N and three runs that must agree bit for
    bit."""
    got, Cref, Den, info = run_case(dev, M, N, K, "bf16", dout, batch=batch, seed=M + N + K + cols,
                                    scale_b=0.02, runs=3,
                                    options=H.Options(skinny_tile_n=cols, skinny_stream_k=2))
    assert info["path"] == H.HGEMM_PATH_SKINNY and info["stream_k"] == 1 and info["tile_n"] == cols
    check(got, Cref, Den, dout)


def test_skinny_batched_and_misaligned(dev):
    M, N, K, batch = 5, 300, 200, 3
    got, Cref, Den, info = run_case(dev, M, N, K, "f16", "f16", batch=batch, ldb=N + 1,
                                    sB=K * (N + 1) + 5, seed=41)
    assert info["path"] == H.HGEMM_PATH_SKINNY and info["repack_b"]
    check(got, Cref, Den, "f16")


def test_skinny_matches_tiled(dev):
    """The two paths compute the same product: both within the bound, and
    equal to each other within twice the bound."""
    M, N, K = 16, 640, 512
    g1, Cref, Den, _ = run_case(dev, M, N, K, "bf16", "f32", seed=42,
                                options=H.Options(force_path=H.HGEMM_PATH_SKINNY))
    g2, _, _, _ = run_case(dev, M, N, K, "bf16", "f32", seed=42,
                           options=H.Options(force_path=H.HGEMM_PATH_TILED))
    check(g1, Cref, Den, "f32")
    check(g2, Cref, Den, "f32")


# ---------------------------------------------------------------- full-size workloads (sampled)

def sample_entries(batch, M, N, n, seed):
    rng = np.random.default_rng(seed)
    eb = list(rng.integers(0, batch, n))
    ei = list(rng.integers(0, M, n))
    ej = list(rng.integers(0, N, n))
    for b in {0, batch - 1}:  # corners and the ragged last row/column
        for i in (0, M - 1):
            for j in (0, N - 1):
                eb.append(b); ei.append(i); ej.append(j)
        for j in rng.integers(0, N, 32):
            eb.append(b); ei.append(M - 1); ej.append(int(j))
        for i in rng.integers(0, M, 32):
            eb.append(b); ei.append(int(i)); ej.append(N - 1)
    return np.array(eb), np.array(ei), np.array(ej)


@pytest.mark.parametrize("name", ["square4096", "square8192", "batched_qk", "ragged4095",
                                  "ragged4095_h", "skinny"])
def test_workload_full_size_sampled(dev, name):
    w = inputs.WORKLOADS[name]
    A, B = inputs.make_inputs(w)
    dA, dB = A.to(dev), B.to(dev)
    shape = (w.batch, w.M, w.N) if w.batch > 1 else (w.M, w.N)
    C = torch.empty(shape, dtype=TORCH[w.dtype_out], device=dev)
    plan = H.hgemm_plan_create(w.M, w.N, w.K, w.lda, w.ldb, w.ldc, w.batch, w.strideA, w.strideB,
                               w.strideC, DT[w.dtype_in], DT[w.dtype_out])
    try:
        H.hgemm_run(plan, dA, dB, C)
        st = H.hgemm_check(plan)
        assert st == 0, H.hgemm_last_error_detail()
    finally:
        H.hgemm_plan_destroy(plan)
    Cc = C.reshape(w.batch, w.M, w.N).cpu()
    eb, ei, ej = sample_entries(w.batch, w.M, w.N, 3000, 99)
    cref, den = oracle.gemm_entries(bits(A), bits(B), ORACLE_DT[w.dtype_in], w.K, w.lda, w.ldb,
                                    eb, ei, ej, w.strideA, w.strideB)
    vals = Cc[torch.as_tensor(eb), torch.as_tensor(ei), torch.as_tensor(ej)]
    if w.dtype_out == "f32":
        got = vals.double().numpy()
    else:
        got = oracle.decode(bits(vals), ORACLE_DT[w.dtype_out])
    err = oracle.normalized_error(got, cref, den)
    print(f"{name}: max normalised error on {eb.size} sampled entries {err:.3e}")
    assert err <= TOL[w.dtype_out], f"{name}: normalised error {err:.3e}"
    if w.dtype_out != "f32":
        assert err <= STATED_16BIT, f"{name}: normalised error {err:.3e} > {STATED_16BIT}"
    # properties that hold everywhere: finite output
    assert torch.isfinite(Cc.float()).all()


@pytest.mark.parametrize("name", ["square4096", "ragged4095", "ragged4095_h", "skinny"])
def test_workload_full_compare(dev, name):
    """Every element of the full-size product, run by the plan the bench times
    (same shape, leading dimensions and options), against the oracle's full
    product: the oracle needs a few seconds per 4096^3 product on the host
    cores.  (square8192 stays sampled: its oracle product takes minutes.)"""
    w = inputs.WORKLOADS[name]
    A, B = inputs.make_inputs(w)
    dA, dB = A.to(dev), B.to(dev)
    C = torch.full((w.M, w.N), SENTINEL[w.dtype_out], dtype=TORCH[w.dtype_out], device=dev)
    plan = H.hgemm_plan_create_ex(w.M, w.N, w.K, w.lda, w.ldb, w.ldc, w.batch, w.strideA,
                                  w.strideB, w.strideC, DT[w.dtype_in], DT[w.dtype_out],
                                  H.Options(trans_b=0))
    try:
        H.hgemm_run(plan, dA, dB, C)
        st = H.hgemm_check(plan)
        assert st == 0, H.hgemm_last_error_detail()
    finally:
        H.hgemm_plan_destroy(plan)
    Cref, Den = oracle.gemm(bits(A), bits(B), ORACLE_DT[w.dtype_in], w.M, w.N, w.K, w.lda, w.ldb)
    got = read_c(C.reshape(-1), w.dtype_out, w.M, w.N, w.ldc, 1, 0, 0)
    err = oracle.normalized_error(got, Cref, Den)
    print(f"{name}: max normalised error over all {w.M * w.N} entries {err:.3e}")
    assert err <= TOL[w.dtype_out], f"{name}: normalised error {err:.3e}"
    if w.dtype_out != "f32":
        assert err <= STATED_16BIT, f"{name}: normalised error {err:.3e} > {STATED_16BIT}"


def test_batched_qk_full_compare(dev):
    """The batched attention-shaped workload is small enough for the full
    oracle product: every element is checked."""
    w = inputs.WORKLOADS["batched_qk"]
    A, B = inputs.make_inputs(w)
    got, Cref, Den, info = run_case(dev, w.M, w.N, w.K, w.dtype_in, w.dtype_out, batch=w.batch,
                                    A_flat=A.reshape(-1), B_flat=B.reshape(-1))
    check(got, Cref, Den, w.dtype_out)


# ---------------------------------------------------------------- dependent launches

@pytest.mark.parametrize("opt2", [None, H.Options(cta_pair=2), H.Options(force_path=H.HGEMM_PATH_SKINNY)])
def test_back_to_back_dependent_products(dev, opt2):
    """The kernels may be scheduled while the previous kernel of the stream
    finishes; they must still wait for it before touching memory.  Chain on
    one stream, no synchronisation in between:
      1. C1 = A1 . B1            (pair kernel)
      2. C2 = C1[:M2] . B2       (reads C1: read-after-write)
      3. A1 <- C3 = A3 . B3      (overwrites product 1's input: write-after-read)
    and check 2 against the oracle on C1's actual bits."""
    M, N, K = 1024, 768, 2048
    M2 = 16 if opt2 is not None and opt2.force_path == H.HGEMM_PATH_SKINNY else 512
    N2 = 512
    A1 = inputs.make_random((M, K), "bf16", 90).to(dev)
    B1 = inputs.make_random((K, N), "bf16", 91).to(dev)
    B2 = inputs.make_random((N, N2), "bf16", 92).to(dev)
    C1 = torch.empty(M, N, dtype=torch.bfloat16, device=dev)
    C2 = torch.empty(M2, N2, dtype=torch.float32, device=dev)
    A3 = inputs.make_random((M, 256), "bf16", 93).to(dev)
    B3 = inputs.make_random((256, K), "bf16", 94).to(dev)
    A1_bits = bits(A1)
    p1 = H.hgemm_plan_create(M, N, K, K, N, N, 1, 0, 0, 0, H.HGEMM_BF16, H.HGEMM_BF16)
    p2 = H.hgemm_plan_create_ex(M2, N2, N, N, N2, N2, 1, 0, 0, 0, H.HGEMM_BF16, H.HGEMM_F32, opt2)
    p3 = H.hgemm_plan_create(M, K, 256, 256, K, K, 1, 0, 0, 0, H.HGEMM_BF16, H.HGEMM_BF16)
    try:
        for _ in range(3):
            A1.copy_(torch.from_numpy(A1_bits.view(np.int16).reshape(M, K)).view(torch.bfloat16))
            H.hgemm_run(p1, A1, B1, C1)
            H.hgemm_run(p2, C1, B2, C2)
            H.hgemm_run(p3, A3, B3, A1)
        assert H.hgemm_check(p1) == 0 and H.hgemm_check(p2) == 0 and H.hgemm_check(p3) == 0
    finally:
        for p in (p1, p2, p3):
            H.hgemm_plan_destroy(p)
    Cref1, Den1 = oracle.gemm(A1_bits, bits(B1), 1, M, N, K, K, N)
    check(oracle.decode(bits(C1), 1).reshape(1, M, N), Cref1, Den1, "bf16")
    Cref2, Den2 = oracle.gemm(bits(C1)[: M2 * N], bits(B2), 1, M2, N2, N, N, N2)
    check(C2.cpu().double().numpy()[None], Cref2, Den2, "f32")
    Cref3, Den3 = oracle.gemm(bits(A3), bits(B3), 1, M, K, 256, 256, K)
    check(oracle.decode(bits(A1), 1).reshape(1, M, K), Cref3, Den3, "bf16")


# ---------------------------------------------------------------- API surface

def test_one_shot_and_matmul(dev):
    from tensor_core_dense_swizzled_gb300 import matmul
    A = inputs.make_random((300, 200), "bf16", 50)
    B = inputs.make_random((200, 260), "bf16", 51)
    C1 = matmul(A.to(dev), B.to(dev), out_dtype=torch.float32)
    C2 = matmul(A.to(dev), B.to(dev), out_dtype=torch.float32)  # cached plan
    torch.cuda.synchronize()
    assert torch.equal(C1, C2)
    Cref, Den = oracle.gemm(bits(A), bits(B), 1, 300, 260, 200, 200, 260)
    check(C1.cpu().double().numpy()[None], Cref, Den, "f32")
    # batched front end
    Ab = inputs.make_random((3, 64, 80), "f16", 52)
    Bb = inputs.make_random((3, 80, 48), "f16", 53)
    Cb = matmul(Ab.to(dev), Bb.to(dev))
    Cref, Den = oracle.gemm(bits(Ab), bits(Bb), 0, 64, 48, 80, 80, 48, 3, 64 * 80, 80 * 48)
    check(oracle.decode(bits(Cb), 0).reshape(3, 64, 48), Cref, Den, "f16")
    H.hgemm_cache_clear()


def test_one_shot_on_two_streams_from_two_threads(dev):
    """hgemm() from two host threads, each on a stream of its own, many times
    over, on a split-K shape (partial sums in the plan's workspace): the
    cache gives each stream its own plan, so neither run disturbs the other."""
    import threading
    M, N, K = 16, 1024, 8192
    B = inputs.make_random((K, N), "bf16", 70)
    As = [inputs.make_random((M, K), "bf16", 71 + i) for i in range(2)]
    dB = B.to(dev)
    dA = [a.to(dev) for a in As]
    Cs = [torch.zeros(M, N, dtype=torch.float32, device=dev) for _ in range(2)]
    streams = [torch.cuda.Stream(device=dev) for _ in range(2)]
    H.hgemm_cache_clear()
    errors = []

    def work(i):
        try:
            with torch.cuda.stream(streams[i]):
                for _ in range(30):
                    H.hgemm(dA[i], dB, Cs[i], M, N, K, K, N, N, 1, 0, 0, 0, H.HGEMM_BF16, H.HGEMM_F32,
                            streams[i].cuda_stream)
        except Exception as e:  # reported below, on the main thread
            errors.append(e)

    threads = [threading.Thread(target=work, args=(i,)) for i in range(2)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    torch.cuda.synchronize()
    assert not errors, errors
    for i in range(2):
        Cref, Den = oracle.gemm(bits(As[i]), bits(B), 1, M, N, K, K, N)
        check(Cs[i].cpu().double().numpy()[None], Cref, Den, "f32")
    H.hgemm_cache_clear()


def test_matmul_planned_path_on_two_streams_from_two_threads(dev):
    """The torch front end's own plan cache (B given as W.t(): planned,
    transposed-B path) from two host threads on two streams, on a split-K
    shape: each stream gets its own plan."""
    import threading

    from tensor_core_dense_swizzled_gb300 import matmul, matmul_cache_clear
    M, N, K = 16, 1024, 8192
    W = inputs.make_random((N, K), "bf16", 80)  # stored N x K
    As = [inputs.make_random((M, K), "bf16", 81 + i) for i in range(2)]
    dW = W.to(dev)
    dA = [a.to(dev) for a in As]
    Cs = [torch.zeros(M, N, dtype=torch.float32, device=dev) for _ in range(2)]
    streams = [torch.cuda.Stream(device=dev) for _ in range(2)]
    matmul_cache_clear()
    errors = []

    def work(i):
        try:
            for _ in range(30):
                matmul(dA[i], dW.t(), out_dtype=torch.float32, out=Cs[i], stream=streams[i])
        except Exception as e:  # reported below, on the main thread
            errors.append(e)

    threads = [threading.Thread(target=work, args=(i,)) for i in range(2)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    torch.cuda.synchronize()
    assert not errors, errors
    for i in range(2):
        Cref, Den = oracle.gemm_bt(bits(As[i]), bits(W), 1, M, N, K, K, K)
        check(Cs[i].cpu().double().numpy()[None], Cref, Den, "f32")
    matmul_cache_clear()


def test_matmul_transposed_fp8_and_epilogue(dev):
    """The torch front end's planned paths: B given as W.t() (transposed-B
    kernels), 8-bit inputs, and the fused epilogue."""
    import types

    from tensor_core_dense_swizzled_gb300 import matmul, matmul_cache_clear
    M, N, K = 320, 384, 256
    A = inputs.make_random((M, K), "bf16", 60)
    W = inputs.make_random((N, K), "bf16", 61)  # stored N x K
    C = matmul(A.to(dev), W.to(dev).t(), out_dtype=torch.float32)
    Cref, Den = oracle.gemm_bt(bits(A), bits(W), 1, M, N, K, K, K)
    check(C.cpu().double().numpy()[None], Cref, Den, "f32")
    # 8-bit inputs
    A8 = inputs.make_random((M, K), "e4m3", 62)
    W8 = inputs.make_random((N, K), "e4m3", 63)
    C8 = matmul(A8.to(dev), W8.to(dev).t(), out_dtype=torch.float32)
    w8 = lambda t: oracle.widen8(t.contiguous().view(torch.uint8).numpy().reshape(-1))  # noqa: E731
    Cref8, Den8 = oracle.gemm_bt(w8(A8), w8(W8), oracle.E4M3, M, N, K, K, K)
    check(C8.cpu().double().numpy()[None], Cref8, Den8, "f32")
    with pytest.raises(ValueError):
        matmul(A8.to(dev), W8.t().contiguous().to(dev))  # 8-bit B must be W.t()
    # fused epilogue: bias + GELU, and beta reading out
    g = torch.Generator().manual_seed(64)
    bias = torch.randn(N, generator=g)
    Ce = matmul(A.to(dev), W.to(dev).t(), out_dtype=torch.float32, bias=bias.to(dev), activation="gelu")
    D, DenD = oracle.epilogue(Cref[0], Den[0], bias=bias.double().numpy(), act=oracle.ACT_GELU)
    assert oracle.normalized_error(Ce.cpu().double().numpy(), D, DenD) <= 1e-3
    prev = torch.randn(M, N, generator=g).to(dev)
    Cb = matmul(A.to(dev), W.to(dev).t(), out_dtype=torch.float32, out=prev.clone(), alpha=0.5, beta=2.0)
    D, DenD = oracle.epilogue(Cref[0], Den[0], alpha=0.5, beta=2.0, C_prev=prev.cpu().double().numpy())
    assert oracle.normalized_error(Cb.cpu().double().numpy(), D, DenD) <= 1e-3
    torch.cuda.synchronize()
    matmul_cache_clear()


def test_run_host_end_to_end(dev):
    M, N, K = 257, 320, 130
    A = inputs.make_random((M, K), "f16", 60).pin_memory()
    B = inputs.make_random((K, N), "f16", 61).pin_memory()
    C = torch.full((M, N + 8), -7.0, dtype=torch.float32).pin_memory()
    plan = H.hgemm_plan_create(M, N, K, K, N, N + 8, 1, 0, 0, 0, H.HGEMM_F16, H.HGEMM_F32)
    try:
        H.hgemm_run_host(plan, A, B, C)
    finally:
        H.hgemm_plan_destroy(plan)
    assert torch.all(C[:, N:] == -7.0)
    Cref, Den = oracle.gemm(bits(A), bits(B), 0, M, N, K, K, N)
    check(C[:, :N].double().numpy()[None], Cref, Den, "f32")


@pytest.mark.parametrize("M,N,K,lda,ldc,din,dout", [
    (2348, 1100, 4096, 4096, 1100, "bf16", "bf16"),  # chunks of 768 rows, the last of 44
    (1500, 1000, 4000, 4000, 1008, "f16", "f32"),    # chunks of 512, the last of 476; padded C rows
    (2000, 1300, 4095, 4095, 1301, "f16", "f16"),    # misaligned rows of A and C
    (1030, 4096, 4096, 4096, 4096, "bf16", "f32"),   # chunks of 512, 512 and 6 rows (skinny kernel)
])
def test_run_host_row_chunks(dev, M, N, K, lda, ldc, din, dout):
    """Large products through hgemm_run_host run in row chunks whose copies in,
    products and copies out overlap on three streams; every element of C is
    right, host elements outside the M x N block stay intact, and the plan
    gives the same C on a second call."""
    A = inputs.make_random((M * lda,), din, 62).pin_memory()
    B = inputs.make_random((K * N,), din, 63).pin_memory()
    C = torch.full((M * ldc,), -7.0, dtype=TORCH[dout]).pin_memory()
    plan = H.hgemm_plan_create(M, N, K, lda, N, ldc, 1, 0, 0, 0, DT[din], DT[dout])
    try:
        assert H.hgemm_plan_get_info(plan)["host_chunks"] > 1
        H.hgemm_run_host(plan, A, B, C)
        first = C.clone()
        H.hgemm_run_host(plan, A, B, C)
    finally:
        H.hgemm_plan_destroy(plan)
    assert torch.equal(C, first), "repeated calls differ"
    view = torch.as_strided(C, (M, N), (ldc, 1))
    mask = torch.ones(M * ldc, dtype=torch.bool)
    torch.as_strided(mask, (M, N), (ldc, 1)).fill_(False)
    assert torch.all(C[mask] == -7.0), "host elements outside C changed"
    Cref, Den = oracle.gemm(bits(A), bits(B), ORACLE_DT[din], M, N, K, lda, N)
    got = view.double().numpy()[None] if dout == "f32" else \
        oracle.decode(bits(view), ORACLE_DT[dout]).reshape(1, M, N)
    check(got, Cref, Den, dout)


@pytest.mark.parametrize("ldc,gap", [(96, 0), (104, 0), (96, 500)])
def test_run_host_batched_copies(dev, ldc, gap):
    """hgemm_run_host copies C back as one block (dense), one 2-D copy
    (batches stacked at the row pitch) or one 2-D copy per batch (gaps
    between batches); host elements outside the M x N blocks stay intact."""
    batch, M, N, K = 3, 70, 96, 64
    sC = M * ldc + gap
    A = inputs.make_random((batch, M, K), "bf16", 65).pin_memory()
    B = inputs.make_random((batch, K, N), "bf16", 66).pin_memory()
    C = torch.full((batch * sC,), -7.0, dtype=torch.float32).pin_memory()
    plan = H.hgemm_plan_create(M, N, K, K, N, ldc, batch, M * K, K * N, sC, H.HGEMM_BF16, H.HGEMM_F32)
    try:
        H.hgemm_run_host(plan, A, B, C)
    finally:
        H.hgemm_plan_destroy(plan)
    view = torch.as_strided(C, (batch, M, N), (sC, ldc, 1))
    mask = torch.ones(batch * sC, dtype=torch.bool)
    torch.as_strided(mask, (batch, M, N), (sC, ldc, 1)).fill_(False)
    assert torch.all(C[mask] == -7.0), "host elements outside C's blocks changed"
    Cref, Den = oracle.gemm(bits(A), bits(B), 1, M, N, K, K, N, batch, M * K, K * N)
    check(view.double().numpy(), Cref, Den, "f32")


def test_watchdog_selftest(dev):
    """A wait that can never complete gives up after its limit and reports
    HGEMM_ERR_TIMEOUT; the context stays usable afterwards."""
    st, code = H.hgemm_watchdog_selftest(2_000_000)  # 2 ms
    assert st == 6
    assert code & 0x80000000 and ((code >> 16) & 0xFF) == 5
    got, Cref, Den, _ = run_case(dev, 64, 64, 64, "f16", "f32", seed=70)
    check(got, Cref, Den, "f32")


@pytest.mark.parametrize("kb", [1, 2])
def test_tiled_kernel_abort_path(dev, kb):
    """A real GEMM pipeline whose wait cannot complete: the single-CTA tiled
    kernel's producer leaves the stage of K block `kb` unarmed
    (debug_withhold_kb), so the MMA issuer's wait on it runs out after 1 ms.
    Every role then takes its teardown (the producer waits, bounded, for its
    copies in flight; the MMA issuer for its MMAs; TMEM is freed), the run
    reports HGEMM_ERR_TIMEOUT, the error word is cleared on read, and a normal
    product on the same context right after is correct."""
    M = N = K = 128
    A = inputs.make_random((M * K,), "f16", 71, "normal")
    B = inputs.make_random((K * N,), "f16", 72, "normal")
    dA, dB = A.to(dev), B.to(dev)
    dC = torch.zeros(M * N, dtype=torch.float32, device=dev)
    opt = H.Options(cta_pair=2, timeout_ns=1_000_000, debug_withhold_kb=kb)
    plan = H.hgemm_plan_create_ex(M, N, K, K, N, N, 1, 0, 0, 0, H.HGEMM_F16, H.HGEMM_F32, opt)
    try:
        info = H.hgemm_plan_get_info(plan)
        assert info["path"] == H.HGEMM_PATH_TILED and info["tile_m"] == 128
        for _ in range(2):  # the same plan times out again after the word was cleared
            H.hgemm_run(plan, dA.data_ptr(), dB.data_ptr(), dC.data_ptr())
            st = H.hgemm_check(plan)
            assert st == 6, f"expected HGEMM_ERR_TIMEOUT, got {H.STATUS.get(st)}"
            detail = H.hgemm_last_error_detail()
            assert "timed out" in detail and ("MMA issuer" in detail or "epilogue" in detail), detail
            assert H.hgemm_check(plan) == 0, "error word not cleared on read"
    finally:
        H.hgemm_plan_destroy(plan)
    got, Cref, Den, _ = run_case(dev, M, N, K, "f16", "f32", seed=71,
                                 options=H.Options(cta_pair=2))
    check(got, Cref, Den, "f32")


def test_withhold_option_refused_off_the_single_cta_kernel(dev):
    for opt, shape in ((H.Options(cta_pair=1, debug_withhold_kb=1), (512, 512, 512)),
                       (H.Options(force_path=H.HGEMM_PATH_SKINNY, debug_withhold_kb=1), (8, 256, 256)),
                       (H.Options(cta_pair=2, debug_withhold_kb=3), (128, 128, 128))):
        M, N, K = shape
        with pytest.raises(H.HgemmError):
            H.hgemm_plan_create_ex(M, N, K, K, N, N, 1, 0, 0, 0, H.HGEMM_F16, H.HGEMM_F32, opt)


def test_plan_rejects_wrong_device_pointer_use(dev):
    plan = H.hgemm_plan_create(64, 64, 64, 64, 64, 64, 1, 0, 0, 0, H.HGEMM_F16, H.HGEMM_F32)
    try:
        with pytest.raises(H.HgemmError):
            H.hgemm_run(plan, None, None, None)
    finally:
        H.hgemm_plan_destroy(plan)
