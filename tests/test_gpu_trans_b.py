"""GPU parity with B stored N x K (hgemm_options_t.trans_b = 1: C = A . Bs^T).

B is staged K-major (like A) instead of MN-major: the TMA boxes, the
shared-memory descriptor and the instruction descriptor change, the rest of
every path is shared.  Each case compares with the oracle's gemm_bt, on the
same bound as the plain product.
"""
import numpy as np
import pytest
import torch

import oracle
from tensor_core_dense_swizzled_gb300 import hgemm as H, inputs
from test_gpu_parity import DT, ORACLE_DT, TORCH, bits, check, dev, read_c, span  # noqa: F401 (dev: fixture)

pytestmark = pytest.mark.gpu

SENT = 1234.0


def run_bt(dev, M, N, K, din, dout, *, ldb=None, lda=None, ldc=None, batch=1, options=None,
           seed=0, runs=1, off_b=0):
    lda = K if lda is None else lda
    ldb = K if ldb is None else ldb
    ldc = N if ldc is None else ldc
    sA = M * lda if batch > 1 else 0
    sB = N * ldb if batch > 1 else 0
    sC = M * ldc if batch > 1 else 0
    A = inputs.make_random((max(span(M, K, lda, batch, sA), 1),), din, seed)
    Bs = inputs.make_random((off_b + max(span(N, K, ldb, batch, sB), 1),), din, seed + 1)
    nC = max(span(M, N, ldc, batch, sC), 1)
    dA, dB = A.to(dev), Bs.to(dev)
    dC = torch.full((nC + 64,), SENT, dtype=TORCH[dout], device=dev)
    opt = options if options is not None else H.Options()
    opt.trans_b = 1
    plan = H.hgemm_plan_create_ex(M, N, K, lda, ldb, ldc, batch, sA, sB, sC, DT[din], DT[dout], opt)
    try:
        info = H.hgemm_plan_get_info(plan)
        outs = []
        for _ in range(runs):
            H.hgemm_run(plan, dA, dB.data_ptr() + 2 * off_b, dC)
            st = H.hgemm_check(plan)
            assert st == 0, f"hgemm_check: {H.STATUS.get(st)} {H.hgemm_last_error_detail()}"
            outs.append(dC.clone())
    finally:
        H.hgemm_plan_destroy(plan)
    for o in outs[1:]:
        assert torch.equal(o, outs[0]), "repeated runs differ"
    assert torch.all(dC[nC:].cpu() == SENT), "kernel wrote past the end of C"
    got = read_c(dC[:nC], dout, M, N, ldc, batch, sC, 0)
    Cref, Den = oracle.gemm_bt(bits(A), bits(Bs)[off_b:], ORACLE_DT[din], M, N, K, lda, ldb, batch, sA, sB)
    check(got, Cref, Den, dout)
    assert info["trans_b"] == 1
    return info


CASES = {
    # name: (M, N, K, batch, options, check on the plan)
    "pair_wide": (1024, 1024, 512, 1, H.Options(cta_pair=1), lambda i: i["tile_m"] == 256 and i["wide_boxes"] == 1),
    "pair_ragged_n": (1024, 1000, 512, 1, H.Options(cta_pair=1), lambda i: i["wide_boxes"] == 1),
    "pair_k_not_64": (768, 512, 200, 1, H.Options(cta_pair=1), lambda i: i["wide_boxes"] == 0),
    # lda = ldb = K = 333 (unaligned rows): both operands copied, rows padded
    # to 384 with zeros, so the one-copy-per-stage views apply
    "pair_k_odd_copied": (768, 640, 333, 1, H.Options(cta_pair=1),
                          lambda i: i["wide_boxes"] == 1 and i["repack_a"] == 1 and i["repack_b"] == 1),
    "pair_copied_batched": (512, 520, 201, 2, H.Options(cta_pair=1), lambda i: i["wide_boxes"] == 1),
    "pair_ks1": (1024, 768, 640, 1, H.Options(cta_pair=1, pair_k_blocks=1), lambda i: i["tile_k"] == 64),
    "pair_224": (768, 896, 320, 1, H.Options(cta_pair=1, tile_n=224), lambda i: i["tile_n"] == 224),
    "pair_stream_k": (2560, 2048, 256, 1, H.Options(cta_pair=1, tail_mode=3), lambda i: i["stream_k"] == 1),
    "pair_dealt": (1536, 2560, 512, 1, H.Options(cta_pair=1, tail_mode=4), lambda i: i["stream_k"] == 2),
    "single_tma": (640, 512, 320, 1, H.Options(cta_pair=2), lambda i: i["tile_m"] == 128),
    "single_192": (500, 576, 256, 1, H.Options(cta_pair=2, tile_n=192), lambda i: i["tile_n"] == 192),
    "single_generic": (333, 444, 222, 1, H.Options(cta_pair=2, force_generic_store=1), lambda i: not i["tma_store"]),
    "batched": (300, 256, 96, 3, H.Options(cta_pair=2), lambda i: i["tile_m"] == 128),
    "skinny": (8, 3000, 640, 1, H.Options(), lambda i: i["path"] == H.HGEMM_PATH_SKINNY),
    "skinny_192": (8, 3000, 640, 1, H.Options(skinny_tile_n=192), lambda i: i["tile_n"] == 192),
    "skinny_512_split": (16, 5000, 1024, 1, H.Options(skinny_tile_n=512, split_k=3),
                         lambda i: i["tile_n"] == 512 and i["split_k"] == 3),
    "skinny_dealt": (4, 900, 320, 3, H.Options(skinny_stream_k=2), lambda i: i["stream_k"] == 1),
}


@pytest.mark.parametrize("case", sorted(CASES))
@pytest.mark.parametrize("din,dout", [("bf16", "bf16"), ("f16", "f32")])
def test_trans_b_paths(dev, case, din, dout):
    M, N, K, batch, opt, expect = CASES[case]
    info = run_bt(dev, M, N, K, din, dout, batch=batch, options=opt, seed=M + N + K, runs=2)
    assert expect(info), info


@pytest.mark.parametrize("ldb,off_b", [(333, 0), (512, 3), (520, 0)])
def test_trans_b_leading_dimensions(dev, ldb, off_b):
    """A padded or odd leading dimension of the stored N x K matrix, and a
    base pointer off the 16-byte grid: the aligned-copy path for B."""
    info = run_bt(dev, 512, 384, 320, "bf16", "f32", ldb=ldb, off_b=off_b, seed=ldb + off_b)
    assert info["repack_b"] == int(ldb % 8 != 0) or off_b


def test_trans_b_worked_example(dev):
    """The page-1 worked example with B supplied as its transpose: bit-exact."""
    A = torch.tensor([[i for k in range(16)] for i in range(16)], dtype=torch.float16).reshape(-1)
    Bs = torch.tensor([[j for k in range(16)] for j in range(8)], dtype=torch.float16).reshape(-1)
    C = torch.empty(16 * 8, dtype=torch.float32, device=dev)
    opt = H.Options(trans_b=1)
    plan = H.hgemm_plan_create_ex(16, 8, 16, 16, 16, 8, 1, 0, 0, 0, DT["f16"], DT["f32"], opt)
    try:
        H.hgemm_run(plan, A.to(dev), Bs.to(dev), C)
        assert H.hgemm_check(plan) == 0
    finally:
        H.hgemm_plan_destroy(plan)
    i = np.arange(16)[:, None]
    j = np.arange(8)[None, :]
    assert np.array_equal(C.cpu().numpy().reshape(16, 8), 16.0 * i * j)


def test_trans_b_with_epilogue(dev):
    """trans_b composes with the fused epilogue (bias + GELU tanh form)."""
    import types
    M, N, K = 640, 512, 384
    A = inputs.make_random((M * K,), "bf16", 71)
    Bs = inputs.make_random((N * K,), "bf16", 72)
    bias = torch.randn(N, generator=torch.Generator().manual_seed(3))
    C = torch.empty(M * N, dtype=torch.float32, device=dev)
    opt = H.Options(trans_b=1)
    plan = H.hgemm_plan_create_ex(M, N, K, K, K, N, 1, 0, 0, 0, DT["bf16"], DT["f32"], opt)
    try:
        ep = types.SimpleNamespace(alpha=1.0, beta=0.0, bias=bias.to(dev), row_scale=None,
                                   col_scale=None, activation=H.HGEMM_ACT_GELU_TANH)
        H.hgemm_run_ex(plan, A.to(dev), Bs.to(dev), C, ep)
        assert H.hgemm_check(plan) == 0
    finally:
        H.hgemm_plan_destroy(plan)
    Cref, Den = oracle.gemm_bt(bits(A), bits(Bs), ORACLE_DT["bf16"], M, N, K, K, K)
    D, DenD = oracle.epilogue(Cref[0], Den[0], bias=bias.double().numpy(), act=oracle.ACT_GELU_TANH)
    assert oracle.normalized_error(C.cpu().double().numpy().reshape(M, N), D, DenD) <= 1e-3


def test_trans_b_validation():
    """ldb must cover a row of the stored N x K matrix (>= K), not N."""
    with pytest.raises(H.HgemmError):
        H.hgemm_plan_create_ex(64, 256, 128, 128, 100, 256, 1, 0, 0, 0, DT["bf16"], DT["f32"],
                               H.Options(trans_b=1))
    p = H.hgemm_plan_create_ex(64, 256, 128, 128, 128, 256, 1, 0, 0, 0, DT["bf16"], DT["f32"],
                               H.Options(trans_b=1))
    H.hgemm_plan_destroy(p)


@pytest.mark.parametrize("name", ["square4096_tn", "batched_qk_tn", "skinny_tn"])
def test_trans_b_workload_full_size_sampled(dev, name):
    """The transposed-B workloads at full size, in the bench's launch
    configuration, on 3000+ sampled entries: their B holds the same values as
    the plain workloads' (stored N x K), so the oracle takes the plain
    workload's K x N operand."""
    from test_gpu_parity import TOL, sample_entries
    w = inputs.WORKLOADS[name]
    plain = inputs.WORKLOADS[name[:-3]]
    A, Bs = inputs.make_inputs(w)
    _, B = inputs.make_inputs(plain)
    assert torch.equal(Bs, B.transpose(-1, -2))
    shape = (w.batch, w.M, w.N) if w.batch > 1 else (w.M, w.N)
    C = torch.empty(shape, dtype=TORCH[w.dtype_out], device=dev)
    plan = H.hgemm_plan_create_ex(w.M, w.N, w.K, w.lda, w.ldb, w.ldc, w.batch, w.strideA, w.strideB,
                                  w.strideC, DT[w.dtype_in], DT[w.dtype_out], H.Options(trans_b=1))
    try:
        H.hgemm_run(plan, A.to(dev), Bs.to(dev), C)
        st = H.hgemm_check(plan)
        assert st == 0, H.hgemm_last_error_detail()
    finally:
        H.hgemm_plan_destroy(plan)
    Cc = C.reshape(w.batch, w.M, w.N).cpu()
    eb, ei, ej = sample_entries(w.batch, w.M, w.N, 3000, 98)
    cref, den = oracle.gemm_entries(bits(A), bits(B), ORACLE_DT[w.dtype_in], plain.K, plain.lda,
                                    plain.ldb, eb, ei, ej, plain.strideA, plain.strideB)
    vals = Cc[torch.as_tensor(eb), torch.as_tensor(ei), torch.as_tensor(ej)]
    got = vals.double().numpy() if w.dtype_out == "f32" else oracle.decode(bits(vals), ORACLE_DT[w.dtype_out])
    err = oracle.normalized_error(got, cref, den)
    assert err <= TOL[w.dtype_out], f"{name}: normalised error {err:.3e}"
