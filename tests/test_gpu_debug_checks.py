"""Debug invariant checks of the kernels and the debugging environment
overrides (HGEMM_DEBUG, HGEMM_TIMEOUT_NS, HGEMM_FORCE_CONFIG).

With debug_checks every CTA walks its whole sequence of work items before
its roles start (tile and its coordinates inside the output, K range inside
K, piece inside its tile) and reports a violation through the device error
word, never by trapping; a CTA with a bad item does no work.  Checks that
never fire must not change any result; a planted out-of-range tile
(debug_checks = 2, testing only) must be caught, reported by hgemm_check as
HGEMM_ERR_INTERNAL, and leave the context usable.
"""
import os

import pytest
import torch

from tensor_core_dense_swizzled_gb300 import hgemm as H, inputs
from test_gpu_parity import check, dev, run_case  # noqa: F401 (dev: fixture)

pytestmark = pytest.mark.gpu

INTERNAL = 7

# (M, N, K, din, dout, options): every kernel and tail schedule
CASES = [
    (1024, 768, 640, "bf16", "bf16", dict(cta_pair=1)),                    # pair, K halves
    (2560, 2048, 256, "f16", "f32", dict(cta_pair=1, tail_mode=3)),        # pair, stream-K
    (1536, 2048, 320, "bf16", "f16", dict(cta_pair=1, tail_mode=4)),       # pair, dealt pieces
    (300, 4095, 130, "f16", "f32", dict(cta_pair=1)),                      # pair on copied operands
    (640, 1000, 333, "bf16", "bf16", dict(cta_pair=2)),                    # single-CTA
    (640, 1024, 256, "bf16", "bf16", dict(cta_pair=2, tiled_epi_warps=8)),  # eight epilogue warps
    (8, 3000, 1024, "bf16", "bf16", dict(force_path=H.HGEMM_PATH_SKINNY)),             # skinny
    (17, 1000, 640, "f16", "f32", dict(force_path=H.HGEMM_PATH_SKINNY, split_k=3)),     # split
    (8, 2048, 1024, "bf16", "f32", dict(force_path=H.HGEMM_PATH_SKINNY, skinny_stream_k=2)),
]


@pytest.mark.parametrize("case", range(len(CASES)))
def test_checks_on_change_nothing(dev, case):
    M, N, K, din, dout, kw = CASES[case]
    got, Cref, Den, _ = run_case(dev, M, N, K, din, dout, seed=400 + case,
                                 options=H.Options(debug_checks=1, **kw), runs=2)
    check(got, Cref, Den, dout)


@pytest.mark.parametrize("kw", [dict(cta_pair=1, tail_mode=1), dict(cta_pair=2),
                                dict(force_path=H.HGEMM_PATH_SKINNY),
                                dict(force_path=H.HGEMM_PATH_SKINNY, split_k=2)])
def test_planted_tile_is_caught(dev, kw):
    """CTA 0 (pair 0) is handed a tile past the last one; the check stops the
    CTA before any load or store, the run reports
    HGEMM_ERR_INTERNAL, the error word is cleared on read, and a normal run
    right after is correct."""
    skinny = kw.get("force_path") == H.HGEMM_PATH_SKINNY
    M, N, K = (8, 2048, 512) if skinny else (1024, 1024, 256)
    A = inputs.make_random((M * K,), "bf16", 81).to(dev)
    B = inputs.make_random((K * N,), "bf16", 82).to(dev)
    C = torch.zeros(M * N, dtype=torch.float32, device=dev)
    plan = H.hgemm_plan_create_ex(M, N, K, K, N, N, 1, 0, 0, 0, H.HGEMM_BF16, H.HGEMM_F32,
                                  H.Options(debug_checks=2, timeout_ns=10_000_000, **kw))
    try:
        H.hgemm_run(plan, A.data_ptr(), B.data_ptr(), C.data_ptr())
        st = H.hgemm_check(plan)
        assert st == INTERNAL, f"expected HGEMM_ERR_INTERNAL, got {H.STATUS.get(st)}"
        assert "invariant check failed" in H.hgemm_last_error_detail()
        assert H.hgemm_check(plan) == 0, "error word not cleared on read"
    finally:
        H.hgemm_plan_destroy(plan)
    got, Cref, Den, _ = run_case(dev, M, N, K, "bf16", "f32", seed=81, options=H.Options(**kw))
    check(got, Cref, Den, "f32")


@pytest.fixture
def env():
    saved = {k: os.environ.get(k) for k in ("HGEMM_DEBUG", "HGEMM_TIMEOUT_NS", "HGEMM_FORCE_CONFIG")}
    yield os.environ
    for k, v in saved.items():
        if v is None:
            os.environ.pop(k, None)
        else:
            os.environ[k] = v


def test_env_force_config(dev, env):
    """HGEMM_FORCE_CONFIG picks the kernel when the options leave it open;
    explicit options win."""
    args = (2048, 2048, 1024, 1024, 2048, 2048, 1, 0, 0, 0, H.HGEMM_BF16, H.HGEMM_BF16)

    def tile_m(opt=None):
        plan = H.hgemm_plan_create_ex(*args, opt)
        try:
            return H.hgemm_plan_get_info(plan)["tile_m"], H.hgemm_plan_get_info(plan)["tile_n"]
        finally:
            H.hgemm_plan_destroy(plan)

    env.pop("HGEMM_FORCE_CONFIG", None)
    assert tile_m()[0] == 256
    env["HGEMM_FORCE_CONFIG"] = "single:128"
    assert tile_m() == (128, 128)
    assert tile_m(H.Options(cta_pair=1))[0] == 256
    env["HGEMM_FORCE_CONFIG"] = "pair"
    assert tile_m(H.Options(tile_n=256))[0] == 256
    env["HGEMM_FORCE_CONFIG"] = "nonsense"
    assert tile_m()[0] == 256


def test_env_debug_and_timeout(dev, env):
    """HGEMM_DEBUG=1 turns the checks on (results unchanged); HGEMM_TIMEOUT_NS
    sets the watchdog limit of plans that do not set one: a withheld stage
    times out within it."""
    env["HGEMM_DEBUG"] = "1"
    got, Cref, Den, _ = run_case(dev, 640, 1000, 333, "bf16", "bf16", seed=91,
                                 options=H.Options(cta_pair=1))
    check(got, Cref, Den, "bf16")
    env.pop("HGEMM_DEBUG")
    env["HGEMM_TIMEOUT_NS"] = "1000000"
    M = N = K = 128
    A = inputs.make_random((M * K,), "f16", 92).to(dev)
    B = inputs.make_random((K * N,), "f16", 93).to(dev)
    C = torch.zeros(M * N, dtype=torch.float32, device=dev)
    plan = H.hgemm_plan_create_ex(M, N, K, K, N, N, 1, 0, 0, 0, H.HGEMM_F16, H.HGEMM_F32,
                                  H.Options(cta_pair=2, debug_withhold_kb=1))
    try:
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        start.record()
        H.hgemm_run(plan, A.data_ptr(), B.data_ptr(), C.data_ptr())
        end.record()
        assert H.hgemm_check(plan) == 6
        assert start.elapsed_time(end) < 500.0, "the 1 ms limit from the environment was not used"
    finally:
        H.hgemm_plan_destroy(plan)
