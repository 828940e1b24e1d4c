"""Pointers that are not device memory of the plan's GPU are refused on the
host, before anything is launched.

Every run entry point checks its operands with cudaPointerGetAttributes (once
per pointer set, so a loop over the same buffers pays nothing): host memory
(pageable or pinned) where device memory is required gives
HGEMM_ERR_INVALID_ARG with the operand named, instead of a TMA load or a
store from a kernel at an address the GPU cannot use.  After a refusal the
plan runs normally.
"""
import ctypes

import pytest
import torch

from tensor_core_dense_swizzled_gb300 import hgemm as H
from tensor_core_dense_swizzled_gb300 import inputs
from test_gpu_parity import bits, check, dev  # noqa: F401 (dev: fixture)

import oracle

pytestmark = pytest.mark.gpu

INVALID_ARG = 1


def vp(x):
    return ctypes.c_void_p(x)


def test_gemm_refuses_host_operands(dev):
    M = N = K = 256
    A = inputs.make_random((M, K), "bf16", 90)
    B = inputs.make_random((K, N), "bf16", 91)
    dA, dB = A.to(dev), B.to(dev)
    dC = torch.zeros(M, N, dtype=torch.float32, device=dev)
    hC = torch.zeros(M, N, dtype=torch.float32)
    pA = A.pin_memory()
    lib = H.load()
    plan = H.hgemm_plan_create(M, N, K, K, N, N, 1, 0, 0, 0, H.HGEMM_BF16, H.HGEMM_F32)
    try:
        for ptrs, name in [((A.data_ptr(), dB.data_ptr(), dC.data_ptr()), "A"),
                           ((dA.data_ptr(), B.data_ptr(), dC.data_ptr()), "B"),
                           ((dA.data_ptr(), dB.data_ptr(), hC.data_ptr()), "C"),
                           ((pA.data_ptr(), dB.data_ptr(), dC.data_ptr()), "A")]:
            st = lib.hgemm_run(plan, *[vp(x) for x in ptrs], None)
            detail = H.hgemm_last_error_detail()
            assert st == INVALID_ARG, f"{name}: got {H.STATUS.get(st, st)}"
            assert detail.startswith(name) and "host memory" in detail, detail
        torch.cuda.synchronize()
        # the plan is unharmed: a normal run right after
        H.hgemm_run(plan, dA, dB, dC)
        assert H.hgemm_check(plan) == 0
    finally:
        H.hgemm_plan_destroy(plan)
    Cref, Den = oracle.gemm(bits(A), bits(B), 1, M, N, K, K, N)
    check(dC.cpu().double().numpy()[None], Cref, Den, "f32")


def test_zero_fill_refuses_a_host_output(dev):
    """K = 0 writes zeros to C without reading A or B: C is still checked."""
    M, N = 64, 96
    hC = torch.ones(M, N, dtype=torch.float32)
    lib = H.load()
    plan = H.hgemm_plan_create(M, N, 0, 1, N, N, 1, 0, 0, 0, H.HGEMM_F16, H.HGEMM_F32)
    try:
        st = lib.hgemm_run(plan, None, None, vp(hC.data_ptr()), None)
        assert st == INVALID_ARG and H.hgemm_last_error_detail().startswith("C")
        torch.cuda.synchronize()
        dC = torch.ones(M, N, dtype=torch.float32, device=dev)
        H.hgemm_run(plan, None, None, dC)
        assert H.hgemm_check(plan) == 0
        assert torch.count_nonzero(dC).item() == 0
    finally:
        H.hgemm_plan_destroy(plan)
    assert torch.all(hC == 1)


def test_attention_refuses_host_tensors(dev):
    bh, sq, skv = 2, 128, 128
    q, k, v = [inputs.make_random((bh, s, 128), "bf16", 95 + i) for i, s in enumerate((sq, skv, skv))]
    dq, dk, dv = q.to(dev), k.to(dev), v.to(dev)
    dO = torch.zeros_like(dq)
    hO = torch.zeros_like(q)
    lib = H.load()
    plan = H.hgemm_attention_plan_create(bh, sq, skv, 128, 128 ** -0.5, 0, H.HGEMM_BF16)
    try:
        for ptrs, name in [((q.data_ptr(), dk.data_ptr(), dv.data_ptr(), dO.data_ptr()), "Q"),
                           ((dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), hO.data_ptr()), "O")]:
            st = lib.hgemm_attention_run(plan, *[vp(x) for x in ptrs], None)
            detail = H.hgemm_last_error_detail()
            assert st == INVALID_ARG, f"{name}: got {H.STATUS.get(st, st)}"
            assert detail.startswith(name) and "host memory" in detail, detail
        torch.cuda.synchronize()
        H.hgemm_attention_run(plan, dq, dk, dv, dO)
        assert H.hgemm_attention_check(plan) == 0
    finally:
        H.hgemm_attention_plan_destroy(plan)
    assert torch.isfinite(dO.float()).all() and dO.abs().sum().item() > 0


def test_no_alloc_refuses_host_operands(dev):
    M, N, K = 8, 512, 256
    A = inputs.make_random((M, K), "bf16", 97)
    B = inputs.make_random((K, N), "bf16", 98)
    dA, dB = A.to(dev), B.to(dev)
    dC = torch.zeros(M, N, dtype=torch.float32, device=dev)
    hC = torch.zeros(M, N, dtype=torch.float32)
    lib = H.load()
    for ptrs, name in [((A.data_ptr(), dB.data_ptr(), dC.data_ptr()), "A"),
                       ((dA.data_ptr(), dB.data_ptr(), hC.data_ptr()), "C")]:
        st = lib.hgemm_skinny_noalloc(*[vp(x) for x in ptrs], M, N, K, K, N, N, H.HGEMM_BF16,
                                      H.HGEMM_F32, None)
        assert st == INVALID_ARG and H.hgemm_last_error_detail().startswith(name)
    torch.cuda.synchronize()
    H.hgemm_skinny_noalloc(dA, dB, dC, M, N, K, K, N, N, H.HGEMM_BF16, H.HGEMM_F32)
    assert H.hgemm_skinny_noalloc_check() == 0
    Cref, Den = oracle.gemm(bits(A), bits(B), 1, M, N, K, K, N)
    check(dC.cpu().double().numpy()[None], Cref, Den, "f32")


def test_fused_epilogue_refuses_host_vectors(dev):
    """The fused epilogue's bias, row_scale and col_scale are read by the
    kernels as well: a host vector is refused like a host operand."""
    import types
    M, N, K = 128, 256, 128
    A = inputs.make_random((M, K), "bf16", 99)
    B = inputs.make_random((K, N), "bf16", 100)
    dA, dB = A.to(dev), B.to(dev)
    dC = torch.zeros(M, N, dtype=torch.float32, device=dev)
    hvec = {"bias": torch.ones(N), "row_scale": torch.ones(M), "col_scale": torch.ones(N)}
    dvec = {k: v.to(dev) for k, v in hvec.items()}
    plan = H.hgemm_plan_create(M, N, K, K, N, N, 1, 0, 0, 0, H.HGEMM_BF16, H.HGEMM_F32)
    try:
        for name in hvec:
            ep = types.SimpleNamespace(**{k: (hvec[k] if k == name else dvec[k]) for k in hvec})
            with pytest.raises(H.HgemmError) as ei:
                H.hgemm_run_ex(plan, dA, dB, dC, ep)
            assert ei.value.status == INVALID_ARG and name in str(ei.value) and "host memory" in str(ei.value)
        torch.cuda.synchronize()
        H.hgemm_run_ex(plan, dA, dB, dC, types.SimpleNamespace(**dvec))
        assert H.hgemm_check(plan) == 0
    finally:
        H.hgemm_plan_destroy(plan)
    # all-ones scales and bias: C = A.B + 1
    Cref, Den = oracle.gemm(bits(A), bits(B), 1, M, N, K, K, N)
    check((dC.cpu().double().numpy() - 1.0)[None], Cref, Den, "f32")
