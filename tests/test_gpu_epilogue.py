"""GPU parity of the fused epilogue (hgemm_run_ex) against the oracle.

D = act(alpha * rs[i] * cs[j] * (A.B) + beta * C_prev + bias[j]) on every
path that writes C: CTA pairs (whole tiles, K halves, stream-K closing,
first-wave dealing), single-CTA tiles with TMA or predicated stores, the
skinny path unsplit and split-K, and K = 0.  The oracle's epilogue gives
the bound: |D - Dref| <= tol * DenD (tol 1e-3 for fp32 C, 4e-3 for fp16 and
5e-3 for bf16 C: the product's fp32 sums plus one rounding to the output
type, whose unit roundoff is 2^-11 for fp16 and 2^-8 for bf16), entries with
DenD = 0 exact.  C_prev is read in the output type, so the
oracle takes the same decoded values.
"""
import types

import numpy as np
import pytest
import torch

import oracle
from tensor_core_dense_swizzled_gb300 import hgemm as H, inputs
from test_gpu_parity import DT, ORACLE_DT, TORCH, bits, dev, read_c, span  # noqa: F401 (dev: fixture)

pytestmark = pytest.mark.gpu

TOL = {"f32": 1e-3, "f16": 4e-3, "bf16": 5e-3}

EPILOGUES = {
    "bias_relu": dict(alpha=1.5, beta=0.0, bias=True, rs=False, cs=False, act=H.HGEMM_ACT_RELU),
    "beta_gelu_scaled": dict(alpha=0.5, beta=-1.25, bias=False, rs=True, cs=True, act=H.HGEMM_ACT_GELU),
    "all": dict(alpha=2.0, beta=0.75, bias=True, rs=True, cs=True, act=H.HGEMM_ACT_NONE),
    "bias_gelu_tanh": dict(alpha=1.0, beta=0.0, bias=True, rs=False, cs=True, act=H.HGEMM_ACT_GELU_TANH),
}


def run_epi(dev, M, N, K, din, dout, epi, *, batch=1, ldc=None, options=None, seed=0, runs=1):
    lda, ldb = K, N
    ldc = N if ldc is None else ldc
    sA = M * lda if batch > 1 else 0
    sB = K * ldb if batch > 1 else 0
    sC = M * ldc if batch > 1 else 0
    g = torch.Generator().manual_seed(seed + 77)
    A = inputs.make_random((max(span(M, K, lda, batch, sA), 1),), din, seed)
    B = inputs.make_random((max(span(K, N, ldb, batch, sB), 1),), din, seed + 1)
    nC = max(span(M, N, ldc, batch, sC), 1)
    C0 = (torch.randn(nC, generator=g) * 3.0).to(TORCH[dout])
    bias = (torch.randn(N, generator=g) * 2.0) if epi["bias"] else None
    rs = (torch.rand(M, generator=g) * 1.5 + 0.25) if epi["rs"] else None
    cs = (torch.rand(N, generator=g) * 1.5 - 0.5) if epi["cs"] else None
    d = {k: (v.to(dev) if v is not None else None) for k, v in
         dict(bias=bias, row_scale=rs, col_scale=cs).items()}
    ep = types.SimpleNamespace(alpha=epi["alpha"], beta=epi["beta"], activation=epi["act"], **d)
    dA, dB = A.to(dev), B.to(dev)
    plan = H.hgemm_plan_create_ex(M, N, K, lda, ldb, ldc, batch, sA, sB, sC, DT[din], DT[dout], options)
    try:
        info = H.hgemm_plan_get_info(plan)
        outs = []
        for _ in range(runs):
            dC = C0.to(dev)
            H.hgemm_run_ex(plan, dA, dB, dC, ep)
            st = H.hgemm_check(plan)
            assert st == 0, f"hgemm_check: {H.STATUS.get(st)} {H.hgemm_last_error_detail()}"
            outs.append(dC.clone())
    finally:
        H.hgemm_plan_destroy(plan)
    for o in outs[1:]:
        assert torch.equal(o, outs[0]), "repeated runs differ"
    got = read_c(outs[0], dout, M, N, ldc, batch, sC, 0)
    prev = read_c(C0, dout, M, N, ldc, batch, sC, 0)
    Cref, Den = oracle.gemm(bits(A), bits(B), ORACLE_DT[din], M, N, K, lda, ldb, batch, sA, sB)
    D, DenD = oracle.epilogue(Cref, Den, alpha=epi["alpha"], beta=epi["beta"], C_prev=prev,
                              bias=None if bias is None else bias.double().numpy(),
                              row_scale=None if rs is None else rs.double().numpy(),
                              col_scale=None if cs is None else cs.double().numpy(),
                              act=epi["act"])
    err = oracle.normalized_error(got, D, DenD)
    assert err <= TOL[dout], f"normalised error {err}"
    return info


PATHS = {
    # name: (M, N, K, batch, options, expected)
    "pair_halves": (1024, 768, 512, 1, H.Options(cta_pair=1), lambda i: i["tail_split"] == 2),
    "pair_whole": (1024, 1024, 512, 1, H.Options(cta_pair=1, no_tail_split=1), lambda i: i["tile_m"] == 256),
    "pair_stream_k": (2560, 2048, 256, 1, H.Options(cta_pair=1, tail_mode=3), lambda i: i["stream_k"] == 1),
    "pair_dealt": (1536, 2560, 512, 1, H.Options(cta_pair=1, tail_mode=4), lambda i: i["stream_k"] == 2),
    "single_tma": (640, 512, 320, 1, H.Options(cta_pair=2), lambda i: i["tile_m"] == 128 and i["tma_store"]),
    "single_tma_4warps": (640, 512, 320, 1, H.Options(cta_pair=2, tiled_epi_warps=4),
                          lambda i: i["epi_warps"] == 4),
    "single_generic_8warps": (333, 444, 222, 1, H.Options(cta_pair=2, tile_n=256, force_generic_store=1,
                                                          tiled_epi_warps=8),
                              lambda i: not i["tma_store"] and i["epi_warps"] == 8),
    "single_generic": (333, 444, 222, 1, H.Options(cta_pair=2, force_generic_store=1),
                       lambda i: not i["tma_store"]),
    "batched": (300, 256, 96, 3, H.Options(cta_pair=2), lambda i: i["tile_m"] == 128),
    "skinny": (8, 3000, 640, 1, H.Options(), lambda i: i["path"] == H.HGEMM_PATH_SKINNY),
    "skinny_split": (5, 1000, 640, 1, H.Options(split_k=3),
                     lambda i: i["path"] == H.HGEMM_PATH_SKINNY and i["split_k"] == 3),
    "zero_k": (70, 90, 0, 2, H.Options(), lambda i: i["path"] == H.HGEMM_PATH_ZERO_FILL),
}


@pytest.mark.parametrize("path", sorted(PATHS))
@pytest.mark.parametrize("epi", sorted(EPILOGUES))
@pytest.mark.parametrize("din,dout", [("bf16", "bf16"), ("f16", "f32")])
def test_epilogue_paths(dev, path, epi, din, dout):
    M, N, K, batch, opt, expect = PATHS[path]
    info = run_epi(dev, M, N, K, din, dout, EPILOGUES[epi], batch=batch, options=opt,
                   seed=M + N + K, runs=2)
    assert expect(info), info


def test_epilogue_f16_out_and_ragged_ldc(dev):
    """fp16 output, a leading dimension that is not a multiple of 8 (the
    predicated-store path) and GELU with beta."""
    run_epi(dev, 257, 300, 130, "f16", "f16", EPILOGUES["beta_gelu_scaled"], ldc=301,
            options=H.Options(cta_pair=2))


def test_plain_epilogue_equals_hgemm_run(dev):
    """alpha = 1, beta = 0, no vectors, no activation: bit-identical to hgemm_run."""
    M, N, K = 512, 384, 256
    A = inputs.make_random((M * K,), "bf16", 5).to(dev)
    B = inputs.make_random((K * N,), "bf16", 6).to(dev)
    C1 = torch.empty(M * N, dtype=torch.float32, device=dev)
    C2 = torch.full((M * N,), float("nan"), dtype=torch.float32, device=dev)
    plan = H.hgemm_plan_create(M, N, K, K, N, N, 1, 0, 0, 0, DT["bf16"], DT["f32"])
    try:
        H.hgemm_run(plan, A, B, C1)
        H.hgemm_run_ex(plan, A, B, C2, types.SimpleNamespace(alpha=1.0, beta=0.0, activation=0,
                                                             bias=None, row_scale=None, col_scale=None))
        assert H.hgemm_check(plan) == 0
    finally:
        H.hgemm_plan_destroy(plan)
    assert torch.equal(C1, C2)


def test_epilogue_rejects_bad_arguments(dev):
    plan = H.hgemm_plan_create(64, 64, 64, 64, 64, 64, 1, 0, 0, 0, DT["bf16"], DT["f32"])
    A = torch.zeros(64 * 64, dtype=torch.bfloat16, device=dev)
    C = torch.zeros(64 * 64, dtype=torch.float32, device=dev)
    try:
        for bad in (dict(activation=7), dict(alpha=float("inf")), dict(beta=float("nan"))):
            e = types.SimpleNamespace(alpha=1.0, beta=0.0, activation=0, bias=None, row_scale=None,
                                      col_scale=None)
            for k, v in bad.items():
                setattr(e, k, v)
            with pytest.raises(H.HgemmError):
                H.hgemm_run_ex(plan, A, A, C, e)
    finally:
        H.hgemm_plan_destroy(plan)


@pytest.mark.parametrize("generic", [0, 1])
@pytest.mark.parametrize("act", [H.HGEMM_ACT_GELU, H.HGEMM_ACT_GELU_TANH])
@pytest.mark.parametrize("dout", ["bf16", "f32"])
def test_eight_epilogue_warps_ragged_last_tile(dev, generic, act, dout):
    """Eight epilogue warps split each 128 x 256 tile's eight 32-column chunks
    in two halves.  With N = 1904 (= 7 x 256 + 112) the last column tile holds
    3.5 chunks of C: the first half ends inside C and the second half lies
    wholly past column N-1, so its C-prefetch and stores must do nothing.
    beta != 0 (C read back), bias and GELU, TMA and predicated stores."""
    epi = dict(alpha=0.75, beta=0.5, bias=True, rs=False, cs=True, act=act)
    opt = H.Options(cta_pair=2, tile_n=256, tiled_epi_warps=8, force_generic_store=generic)
    info = run_epi(dev, 300, 1904, 256, "bf16", dout, epi, options=opt, seed=11, runs=2)
    assert info["epi_warps_epilogue"] == 8 and info["tile_n"] == 256
    assert bool(info["tma_store"]) == (not generic)
