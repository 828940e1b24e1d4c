"""GPU parity with 8-bit inputs (HGEMM_E4M3 / HGEMM_E5M2).

The input-type table of "tensor-cores-cutlass-and-cute" lists FP8 e4m3 with
fp32 accumulation, its instruction taking twice the K of a 16-bit type, and
the same page's FP8 kernel configurations take K blocks of 128 one-byte
elements where bf16 takes 64.  Each product of two 8-bit values is exact in
fp32, so the bound is the 16-bit inputs' one: max |C - Cref| / sum |a||b|
<= 1e-3 (fp32 out), 4e-3 (fp16 out) or 5e-3 (bf16 out), and bit-exact for
small integers.

8-bit operands are read in place in the layout the tensor cores take: A
M x K and B stored N x K (trans_b), 16-byte aligned rows.  Every case runs
through the C ABI and compares with the oracle's gemm_bt on the same bytes
(widened to the oracle's 16-bit pattern arrays).
"""
import types

import numpy as np
import pytest
import torch

import oracle
from tensor_core_dense_swizzled_gb300 import hgemm as H, inputs
from test_gpu_parity import DT, ORACLE_DT, TOL, TORCH, check, dev, read_c, span  # noqa: F401 (dev: fixture)

pytestmark = pytest.mark.gpu

SENT = 1234.0
F8 = {"e4m3": H.HGEMM_E4M3, "e5m2": H.HGEMM_E5M2}
ORACLE_F8 = {"e4m3": oracle.E4M3, "e5m2": oracle.E5M2}


def bits8(t):
    """Raw 8-bit patterns widened to the oracle's 16-bit arrays."""
    return oracle.widen8(t.contiguous().cpu().view(torch.uint8).numpy().reshape(-1))


def run_f8(dev, M, N, K, din, dout, *, lda=None, ldb=None, ldc=None, batch=1, options=None,
           seed=0, runs=1, dist="normal", epilogue=None, exact=False):
    lda = K if lda is None else lda
    ldb = K if ldb is None else ldb
    ldc = N if ldc is None else ldc
    sA = M * lda if batch > 1 else 0
    sB = N * ldb if batch > 1 else 0
    sC = M * ldc if batch > 1 else 0
    A = inputs.make_random((max(span(M, K, lda, batch, sA), 1),), din, seed, dist)
    Bs = inputs.make_random((max(span(N, K, ldb, batch, sB), 1),), din, seed + 1, dist)
    nC = max(span(M, N, ldc, batch, sC), 1)
    dA, dB = A.to(dev), Bs.to(dev)
    dC = torch.full((nC + 64,), SENT, dtype=TORCH[dout], device=dev)
    opt = options if options is not None else H.Options()
    opt.trans_b = 1
    plan = H.hgemm_plan_create_ex(M, N, K, lda, ldb, ldc, batch, sA, sB, sC, F8[din], DT[dout], opt)
    try:
        info = H.hgemm_plan_get_info(plan)
        outs = []
        for _ in range(runs):
            if epilogue is None:
                H.hgemm_run(plan, dA, dB, dC)
            else:
                H.hgemm_run_ex(plan, dA, dB, dC, epilogue)
            st = H.hgemm_check(plan)
            assert st == 0, f"hgemm_check: {H.STATUS.get(st)} {H.hgemm_last_error_detail()}"
            outs.append(dC.clone())
    finally:
        H.hgemm_plan_destroy(plan)
    for o in outs[1:]:
        assert torch.equal(o, outs[0]), "repeated runs differ"
    assert torch.all(dC[nC:].cpu() == SENT), "kernel wrote past the end of C"
    got = read_c(dC[:nC], dout, M, N, ldc, batch, sC, 0)
    Cref, Den = oracle.gemm_bt(bits8(A), bits8(Bs), ORACLE_F8[din], M, N, K, lda, ldb, batch, sA, sB)
    return info, got, Cref, Den


CASES = {
    # name: (M, N, K, batch, options, check on the plan)
    "pair_wide": (1024, 1024, 512, 1, H.Options(cta_pair=1),
                  lambda i: i["tile_m"] == 256 and i["wide_boxes"] == 1 and i["tile_k"] == 256),
    "pair_ragged_mn": (1000, 1000, 768, 1, H.Options(cta_pair=1), lambda i: i["wide_boxes"] == 1),
    "pair_k_not_128": (768, 512, 208, 1, H.Options(cta_pair=1), lambda i: i["wide_boxes"] == 0),
    "pair_k_odd_blocks": (512, 768, 384, 1, H.Options(cta_pair=1), lambda i: i["wide_boxes"] == 1),
    "pair_halves": (2816, 2048, 512, 1, H.Options(cta_pair=1, tail_mode=2), lambda i: i["tail_split"] == 2),
    "pair_stream_k": (2560, 2048, 512, 1, H.Options(cta_pair=1, tail_mode=3), lambda i: i["stream_k"] == 1),
    "pair_dealt": (1536, 2560, 1024, 1, H.Options(cta_pair=1, tail_mode=4), lambda i: i["stream_k"] == 2),
    "single_256": (640, 512, 320, 1, H.Options(cta_pair=2), lambda i: i["tile_m"] == 128 and i["tile_k"] == 128),
    "single_128": (500, 300, 256, 1, H.Options(cta_pair=2, tile_n=128), lambda i: i["tile_n"] == 128),
    "single_generic": (333, 444, 224, 1, H.Options(cta_pair=2, force_generic_store=1),
                       lambda i: not i["tma_store"]),
    "batched": (300, 256, 96, 3, H.Options(cta_pair=2), lambda i: i["tile_m"] == 128),
    "skinny": (8, 3000, 640, 1, H.Options(), lambda i: i["path"] == H.HGEMM_PATH_SKINNY),
    "skinny_256": (32, 5000, 1024, 1, H.Options(skinny_tile_n=256), lambda i: i["tile_n"] == 256),
    "skinny_split": (16, 1000, 2048, 1, H.Options(split_k=3), lambda i: i["split_k"] == 3),
    "skinny_dealt": (4, 900, 384, 3, H.Options(skinny_stream_k=2), lambda i: i["stream_k"] == 1),
}


@pytest.mark.parametrize("case", sorted(CASES))
@pytest.mark.parametrize("din,dout", [("e4m3", "bf16"), ("e5m2", "f32"), ("e4m3", "f16")])
def test_fp8_paths(dev, case, din, dout):
    M, N, K, batch, opt, expect = CASES[case]
    info, got, Cref, Den = run_f8(dev, M, N, K, din, dout, batch=batch, options=opt,
                                  seed=M + N + K, runs=2)
    check(got, Cref, Den, dout)
    assert expect(info), info


@pytest.mark.parametrize("din", ["e4m3", "e5m2"])
@pytest.mark.parametrize("path", ["pair", "single", "skinny"])
def test_fp8_small_integers_bit_exact(dev, din, path):
    """Integers in [-4, 4] are exact in both formats and every partial sum is
    an integer below 2^24: the fp32 result equals the exact product."""
    M = 8 if path == "skinny" else 512
    opt = H.Options(cta_pair=1 if path == "pair" else 2) if path != "skinny" else H.Options()
    info, got, Cref, Den = run_f8(dev, M, 512, 640, din, "f32", options=opt, seed=5, dist="int4")
    check(got, Cref, Den, "f32", exact=True)


def test_fp8_padded_leading_dimensions(dev):
    """Row pitches above K (multiples of 16 bytes) and a padded C."""
    info, got, Cref, Den = run_f8(dev, 640, 384, 200, "e4m3", "f32", lda=208, ldb=256, ldc=400, seed=9)
    check(got, Cref, Den, "f32")
    assert not info["repack_a"] and not info["repack_b"]


def test_fp8_dequant_epilogue(dev):
    """Per-row and per-column scales with a bias: the dequantising epilogue
    the same page describes for FP8 GEMMs (scales fused into the epilogue)."""
    M, N, K = 640, 512, 384
    g = torch.Generator().manual_seed(17)
    rs = torch.rand(M, generator=g) * 0.5 + 0.25
    cs = torch.rand(N, generator=g) * 0.5 + 0.25
    bias = torch.randn(N, generator=g)
    ep = types.SimpleNamespace(alpha=0.5, beta=0.0, bias=bias.to(dev), row_scale=rs.to(dev),
                               col_scale=cs.to(dev), activation=H.HGEMM_ACT_RELU)
    for opt in (H.Options(cta_pair=1), H.Options(cta_pair=2)):
        info, got, Cref, Den = run_f8(dev, M, N, K, "e4m3", "f32", options=opt, seed=21, epilogue=ep)
        D, DenD = oracle.epilogue(Cref[0], Den[0], alpha=0.5, bias=bias.double().numpy(),
                                  row_scale=rs.double().numpy(), col_scale=cs.double().numpy(),
                                  act=oracle.ACT_RELU)
        assert oracle.normalized_error(got[0], D, DenD) <= 1e-3
    # skinny path
    ep.row_scale = rs[:8].to(dev)
    info, got, Cref, Den = run_f8(dev, 8, N, K, "e5m2", "bf16", seed=23, epilogue=ep)
    D, DenD = oracle.epilogue(Cref[0], Den[0], alpha=0.5, bias=bias.double().numpy(),
                              row_scale=rs[:8].double().numpy(), col_scale=cs.double().numpy(),
                              act=oracle.ACT_RELU)
    assert oracle.normalized_error(got[0], D, DenD) <= TOL["bf16"]


def test_fp8_host_buffers(dev):
    """hgemm_run_host copies 1-byte elements (A and B spans in bytes)."""
    M, N, K = 256, 384, 256
    A = inputs.make_random((M * K,), "e4m3", 31)
    Bs = inputs.make_random((N * K,), "e4m3", 32)
    C = torch.empty(M * N, dtype=torch.float32).pin_memory()
    plan = H.hgemm_plan_create_ex(M, N, K, K, K, N, 1, 0, 0, 0, F8["e4m3"], DT["f32"], H.Options(trans_b=1))
    try:
        H.hgemm_run_host(plan, A.view(torch.uint8).pin_memory(), Bs.view(torch.uint8).pin_memory(), C)
    finally:
        H.hgemm_plan_destroy(plan)
    Cref, Den = oracle.gemm_bt(bits8(A), bits8(Bs), oracle.E4M3, M, N, K, K, K)
    check(C.double().numpy().reshape(1, M, N), Cref, Den, "f32")


def test_fp8_host_buffers_in_row_chunks(dev):
    """A large 8-bit product through hgemm_run_host runs in row chunks (plan
    info host_chunks > 1): chunk pointers stay 16-byte aligned, every element
    of C is right."""
    M, N, K = 2048, 1024, 8192
    A = inputs.make_random((M * K,), "e4m3", 33)
    Bs = inputs.make_random((N * K,), "e4m3", 34)
    C = torch.empty(M * N, dtype=torch.bfloat16).pin_memory()
    plan = H.hgemm_plan_create_ex(M, N, K, K, K, N, 1, 0, 0, 0, F8["e4m3"], DT["bf16"], H.Options(trans_b=1))
    try:
        assert H.hgemm_plan_get_info(plan)["host_chunks"] == 4
        H.hgemm_run_host(plan, A.view(torch.uint8).pin_memory(), Bs.view(torch.uint8).pin_memory(), C)
    finally:
        H.hgemm_plan_destroy(plan)
    Cref, Den = oracle.gemm_bt(bits8(A), bits8(Bs), oracle.E4M3, M, N, K, K, K)
    got = read_c(C, "bf16", M, N, N, 1, 0, 0)
    check(got, Cref, Den, "bf16")


def test_fp8_misaligned_pointer_is_unsupported(dev):
    """No aligned copy is made for 8-bit operands: a base pointer off the
    16-byte grid is refused at run time, before any launch."""
    M, N, K = 128, 128, 128
    buf = torch.zeros(M * K + 64, dtype=torch.uint8, device=dev)
    Bs = torch.zeros(N * K, dtype=torch.uint8, device=dev)
    C = torch.empty(M * N, dtype=torch.float32, device=dev)
    plan = H.hgemm_plan_create_ex(M, N, K, K, K, N, 1, 0, 0, 0, F8["e4m3"], DT["f32"], H.Options(trans_b=1))
    try:
        with pytest.raises(H.HgemmError) as ei:
            H.hgemm_run(plan, buf.data_ptr() + 8, Bs, C)
        assert ei.value.status == 2
        H.hgemm_run(plan, buf, Bs, C)
        assert H.hgemm_check(plan) == 0
    finally:
        H.hgemm_plan_destroy(plan)


@pytest.mark.parametrize("name", ["square4096_fp8", "skinny_fp8"])
def test_fp8_workload_full_size_sampled(dev, name):
    """The 8-bit workloads at full size, in the bench's launch configuration,
    on 3000 sampled entries (the oracle's entry-wise sums over K x N B, the
    stored N x K matrix transposed on the host)."""
    from test_gpu_parity import sample_entries
    w = inputs.WORKLOADS[name]
    A, Bs = inputs.make_inputs(w)
    C = torch.empty((w.M, w.N), dtype=TORCH[w.dtype_out], device=dev)
    plan = H.hgemm_plan_create_ex(w.M, w.N, w.K, w.lda, w.ldb, w.ldc, w.batch, w.strideA, w.strideB,
                                  w.strideC, F8[w.dtype_in], DT[w.dtype_out], H.Options(trans_b=1))
    try:
        H.hgemm_run(plan, A.to(dev), Bs.to(dev), C)
        st = H.hgemm_check(plan)
        assert st == 0, H.hgemm_last_error_detail()
    finally:
        H.hgemm_plan_destroy(plan)
    Bkn = Bs.view(torch.uint8).t().contiguous()
    eb, ei, ej = sample_entries(1, w.M, w.N, 3000, 99)
    cref, den = oracle.gemm_entries(bits8(A), oracle.widen8(Bkn.numpy().reshape(-1)),
                                    ORACLE_F8[w.dtype_in], w.K, w.K, w.N, eb, ei, ej)
    vals = C.cpu()[torch.as_tensor(ei), torch.as_tensor(ej)]
    got = vals.double().numpy() if w.dtype_out == "f32" else oracle.decode(
        vals.contiguous().view(torch.int16).numpy().view(np.uint16), ORACLE_DT[w.dtype_out])
    err = oracle.normalized_error(got, cref, den)
    assert err <= TOL[w.dtype_out], f"{name}: normalised error {err:.3e}"
