"""The allocation-free small-M entry point, hgemm_skinny_noalloc.

It serves callers that may not allocate device memory (a framework that owns
all allocations, a budget fixed at start-up, a loop that cannot afford
cudaMalloc's synchronisation).  Its scratch is a fixed array inside the
library that every call shares, so two calls in a row must both give the
same answer as the planned path (hgemm_plan_create / hgemm_run), within the
tolerance the other parity tests use: max |C - Cref| / sum_k |A_ik||B_kj|
<= 5e-3 for bf16 output (fp32 sums plus one rounding to bf16, unit roundoff
2^-8), 4e-3 for fp16 output.  This file is collected last on purpose and builds
everything it needs, so it also passes alone in a fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from tensor_core_dense_swizzled_gb300 import hgemm as H
from tensor_core_dense_swizzled_gb300 import inputs

pytestmark = pytest.mark.gpu


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


def noalloc(lib, A, B, C, M, N, K, lda, ldb, ldc, din, dout):
    return lib.hgemm_skinny_noalloc(ctypes.c_void_p(A.data_ptr()), ctypes.c_void_p(B.data_ptr()),
                                    ctypes.c_void_p(C.data_ptr()), M, N, K, lda, ldb, ldc, din, dout,
                                    ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def test_no_alloc_matches_planned_path_twice(dev):
    w = inputs.WORKLOADS["skinny"]  # M=8, N=28672, K=4096 bf16, bf16 out
    A, B = inputs.make_inputs(w)
    dA, dB = A.to(dev), B.to(dev)
    lib = H.load()
    # the planned path (allocating entry points)
    C_plan = torch.empty(w.M, w.N, dtype=torch.bfloat16, device=dev)
    plan = H.hgemm_plan_create(w.M, w.N, w.K, w.lda, w.ldb, w.ldc, 1, 0, 0, 0, H.HGEMM_BF16,
                               H.HGEMM_BF16)
    try:
        H.hgemm_run(plan, dA, dB, C_plan)
        assert H.hgemm_check(plan) == 0
    finally:
        H.hgemm_plan_destroy(plan)
    Cref, Den = oracle.gemm(bits(A), bits(B), 1, w.M, w.N, w.K, w.lda, w.ldb)
    planned = oracle.decode(bits(C_plan), 1).reshape(1, w.M, w.N)
    assert oracle.normalized_error(planned, Cref, Den) <= 5e-3
    # two calls in a row through the C ABI: the shared scratch keeps the first
    # call's contents and must not disturb the second
    outs = []
    for _ in range(2):
        C = torch.full((w.M, w.N), 7.0, dtype=torch.bfloat16, device=dev)
        st = noalloc(lib, dA, dB, C, w.M, w.N, w.K, w.lda, w.ldb, w.ldc, H.HGEMM_BF16, H.HGEMM_BF16)
        assert st == 0, H.hgemm_last_error_detail()
        # the allocation-free status check: no watchdog timeout, word cleared
        assert H.hgemm_skinny_noalloc_check(torch.cuda.current_stream().cuda_stream) == 0
        torch.cuda.synchronize()
        got = oracle.decode(bits(C), 1).reshape(1, w.M, w.N)
        diff = np.abs(got - planned)
        nz = Den > 0
        assert np.max(diff[nz] / Den[nz]) <= 5e-3
        assert oracle.normalized_error(got, Cref, Den) <= 5e-3
        outs.append(C.cpu())
    assert torch.equal(outs[0], outs[1])


def test_no_alloc_small_shapes_and_outputs(dev):
    lib = H.load()
    for (M, N, K, dout) in [(1, 304, 200, H.HGEMM_F32), (17, 1000, 640, H.HGEMM_F16),
                            (32, 256, 64, H.HGEMM_BF16)]:
        A = inputs.make_random((M, K), "f16", M + N)
        B = inputs.make_random((K, N), "f16", M + N + 1)
        td = {H.HGEMM_F32: torch.float32, H.HGEMM_F16: torch.float16, H.HGEMM_BF16: torch.bfloat16}[dout]
        for _ in range(2):
            C = torch.empty(M, N, dtype=td, device=dev)
            st = noalloc(lib, A.to(dev), B.to(dev), C, M, N, K, K, N, N, H.HGEMM_F16, dout)
            assert st == 0, H.hgemm_last_error_detail()
            assert H.hgemm_skinny_noalloc_check() == 0, H.hgemm_last_error_detail()
            torch.cuda.synchronize()
            Cref, Den = oracle.gemm(bits(A), bits(B), 0, M, N, K, K, N)
            got = C.cpu().double().numpy()[None] if dout == H.HGEMM_F32 else \
                oracle.decode(bits(C), 0 if dout == H.HGEMM_F16 else 1).reshape(1, M, N)
            tol = {H.HGEMM_F32: 1e-3, H.HGEMM_F16: 4e-3, H.HGEMM_BF16: 5e-3}[dout]
            assert oracle.normalized_error(got, Cref, Den) <= tol


def test_no_alloc_lowers_the_split_to_fit(dev):
    """M = 32, N = 16384, K = 8192: the planned path splits K seven ways
    (64 column tiles of 256 fill too few of the SMs), and its fp32 partials,
    7 x 128 sub-tiles x 32 x 128 x 4 bytes = 14 MiB, would not fit the 8 MiB
    array.  The allocation-free call runs with the split lowered to three
    (6 MiB) and must still match the oracle and the planned path, twice."""
    M, N, K = 32, 16384, 8192
    A = inputs.make_random((M, K), "bf16", 31)
    B = inputs.make_random((K, N), "bf16", 32, "normal", 0.02)
    dA, dB = A.to(dev), B.to(dev)
    lib = H.load()
    C_plan = torch.empty(M, N, dtype=torch.float32, device=dev)
    plan = H.hgemm_plan_create(M, N, K, K, N, N, 1, 0, 0, 0, H.HGEMM_BF16, H.HGEMM_F32)
    try:
        info = H.hgemm_plan_get_info(plan)
        # the premise: the planned split would overflow the fixed array
        num_n = (N + info["tile_n"] - 1) // info["tile_n"] * (info["tile_n"] // 128)
        assert info["split_k"] * num_n * 32 * 128 * 4 > (8 << 20)
        H.hgemm_run(plan, dA, dB, C_plan)
        assert H.hgemm_check(plan) == 0
    finally:
        H.hgemm_plan_destroy(plan)
    Cref, Den = oracle.gemm(bits(A), bits(B), 1, M, N, K, K, N)
    planned = C_plan.cpu().double().numpy()[None]
    assert oracle.normalized_error(planned, Cref, Den) <= 1e-3
    outs = []
    for _ in range(2):
        C = torch.full((M, N), 7.0, dtype=torch.float32, device=dev)
        st = noalloc(lib, dA, dB, C, M, N, K, K, N, N, H.HGEMM_BF16, H.HGEMM_F32)
        assert st == 0, H.hgemm_last_error_detail()
        torch.cuda.synchronize()
        got = C.cpu().double().numpy()[None]
        assert oracle.normalized_error(got, Cref, Den) <= 1e-3
        nz = Den > 0
        assert np.max(np.abs(got - planned)[nz] / Den[nz]) <= 1e-3
        outs.append(C.cpu())
    assert torch.equal(outs[0], outs[1])


def test_no_alloc_refuses_what_it_cannot_do(dev):
    lib = H.load()
    A = torch.zeros(64 * 72, dtype=torch.float16, device=dev)
    B = torch.zeros(72 * 80, dtype=torch.float16, device=dev)
    C = torch.zeros(64 * 80, dtype=torch.float32, device=dev)
    # M > 32
    assert noalloc(lib, A, B, C, 64, 80, 64, 64, 80, 80, H.HGEMM_F16, H.HGEMM_F32) == 2
    # misaligned leading dimension: no aligned copy can be made without scratch
    assert noalloc(lib, A, B, C, 8, 80, 63, 63, 80, 80, H.HGEMM_F16, H.HGEMM_F32) == 2
    assert "aligned" in H.hgemm_last_error_detail()
    # N beyond what the fixed array holds, even unsplit (checked before any launch)
    huge = (8 << 20) // 16 * 128 + 128
    assert noalloc(lib, A, B, C, 8, huge, 64, 64, huge, huge, H.HGEMM_F16, H.HGEMM_F32) == 2
    assert "scratch" in H.hgemm_last_error_detail()
    # bad dtype
    assert noalloc(lib, A, B, C, 8, 80, 64, 64, 80, 80, H.HGEMM_F32, H.HGEMM_F32) == 1
