"""Host-side checks of the C ABI that need no GPU.

* the library builds, loads and exports every function ``include/hgemm.h``
  declares;
* status strings and the version;
* argument validation: every malformed request is refused with
  HGEMM_ERR_INVALID_ARG before any device is touched (the Ampere wrapper in
  "tensor-cores-cutlass-and-cute" section 四.4 refuses a wrong dtype rather
  than reinterpreting it; the same holds here);
* well-formed requests on a machine without an sm_103 GPU fail with
  HGEMM_ERR_NO_DEVICE, never with a crash.
"""
import ctypes
import os
import re

import pytest

from tensor_core_dense_swizzled_gb300 import build as B
from tensor_core_dense_swizzled_gb300 import hgemm as H

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    B.build()
    return H.load()


def declared_functions():
    text = open(os.path.join(ROOT, "include", "hgemm.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*(hgemm[A-Za-z0-9_]*)\s*\(",
                       text, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_abi():
    names = declared_functions()
    for must in ("hgemm_plan_create", "hgemm_run", "hgemm_check", "hgemm_plan_destroy", "hgemm",
                 "hgemm_status_string", "hgemm_last_error_detail", "hgemm_run_host"):
        assert must in names


def test_every_declared_symbol_is_exported(lib):
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, f"not exported: {missing}"


def test_status_strings_and_version(lib):
    for code, name in H.STATUS.items():
        assert H.hgemm_status_string(code) == name
    assert H.hgemm_status_string(99) == "HGEMM_ERR_UNKNOWN"
    assert H.hgemm_version() >= 100


def _create(*args):
    lib = H.load()
    h = ctypes.c_void_p()
    st = lib.hgemm_plan_create(ctypes.byref(h), *args)
    return st, h.value


GOOD = (64, 64, 64, 64, 64, 64, 1, 0, 0, 0, H.HGEMM_BF16, H.HGEMM_BF16)


@pytest.mark.parametrize("args,why", [
    ((64, 64, 64, 64, 64, 64, 1, 0, 0, 0, H.HGEMM_F32, H.HGEMM_BF16), "fp32 input"),
    ((64, 64, 64, 64, 64, 64, 1, 0, 0, 0, 7, H.HGEMM_BF16), "unknown input dtype"),
    ((64, 64, 64, 64, 64, 64, 1, 0, 0, 0, H.HGEMM_F16, 9), "unknown output dtype"),
    ((-1, 64, 64, 64, 64, 64, 1, 0, 0, 0, H.HGEMM_F16, H.HGEMM_F32), "negative M"),
    ((64, -1, 64, 64, 64, 64, 1, 0, 0, 0, H.HGEMM_F16, H.HGEMM_F32), "negative N"),
    ((64, 64, -1, 64, 64, 64, 1, 0, 0, 0, H.HGEMM_F16, H.HGEMM_F32), "negative K"),
    ((64, 64, 64, 63, 64, 64, 1, 0, 0, 0, H.HGEMM_F16, H.HGEMM_F32), "lda < K"),
    ((64, 64, 64, 64, 63, 64, 1, 0, 0, 0, H.HGEMM_F16, H.HGEMM_F32), "ldb < N"),
    ((64, 64, 64, 64, 64, 63, 1, 0, 0, 0, H.HGEMM_F16, H.HGEMM_F32), "ldc < N"),
    ((64, 64, 64, 64, 64, 64, 0, 0, 0, 0, H.HGEMM_F16, H.HGEMM_F32), "batch 0"),
    ((64, 64, 64, 64, 64, 64, 2, -1, 0, 4096, H.HGEMM_F16, H.HGEMM_F32), "negative strideA"),
    ((64, 64, 64, 64, 64, 64, 2, 4096, 4096, 100, H.HGEMM_F16, H.HGEMM_F32), "overlapping C batches"),
])
def test_invalid_arguments_are_refused(lib, args, why):
    st, h = _create(*args)
    assert st == 1, f"{why}: got {H.STATUS.get(st, st)}"
    assert h is None
    assert H.hgemm_last_error_detail()


def test_null_plan_pointer(lib):
    st = lib.hgemm_plan_create(None, *GOOD)
    assert st == 1


def test_oversized_request_is_unsupported(lib):
    st, _ = _create(1 << 31, 64, 64, 64, 64, 64, 1, 0, 0, 0, H.HGEMM_F16, H.HGEMM_F32)
    assert st == 2


@pytest.mark.parametrize("args,why", [
    ((1 << 20, 64, 64, 1 << 45, 64, 64, 1, 0, 0, 0, H.HGEMM_F16, H.HGEMM_F32), "huge lda"),
    ((64, 64, 1 << 20, 1 << 20, 1 << 45, 64, 1, 0, 0, 0, H.HGEMM_F16, H.HGEMM_F32), "huge ldb"),
    ((1 << 20, 64, 64, 64, 64, 1 << 45, 1, 0, 0, 0, H.HGEMM_F16, H.HGEMM_F32), "huge ldc"),
    ((64, 64, 64, 64, 64, 64, 1 << 20, 1 << 45, 4096, 4096, H.HGEMM_F16, H.HGEMM_F32), "huge strideA"),
    ((64, 64, 64, 64, (1 << 62) + 1, 64, 1 << 10, 4096, 1, 4096, H.HGEMM_F16, H.HGEMM_F32),
     "span past 64 bits"),
])
def test_spans_beyond_2_60_bytes_are_unsupported(lib, args, why):
    """A leading dimension or batch stride whose operand span passes 2^60
    bytes is refused before any byte count could overflow."""
    st, h = _create(*args)
    assert st == 2, f"{why}: got {H.STATUS.get(st, st)}"
    assert h is None
    assert "2^60" in H.hgemm_last_error_detail()


def test_null_handles(lib):
    assert lib.hgemm_run(None, None, None, None, None) == 1
    assert lib.hgemm_check(None, None) == 1
    assert lib.hgemm_plan_destroy(None) == 0
    assert lib.hgemm_plan_get_info(None, None) == 1
    assert lib.hgemm_run_host(None, None, None, None, None) == 1


def test_bad_options_are_refused(lib):
    h = ctypes.c_void_p()
    for opt in (H.Options(force_path=7), H.Options(tile_n=160), H.Options(split_k=-2),
                H.Options(debug_withhold_kb=-1), H.Options(debug_checks=3)):
        st = lib.hgemm_plan_create_ex(ctypes.byref(h), *GOOD, ctypes.byref(opt))
        assert st == 1
    # the skinny path is for M <= 32
    opt = H.Options(force_path=H.HGEMM_PATH_SKINNY)
    st = lib.hgemm_plan_create_ex(ctypes.byref(h), *GOOD, ctypes.byref(opt))
    assert st == 2


def test_fp8_layout_rules(lib):
    """8-bit inputs are read in place: B must be stored N x K (trans_b),
    rows and batch strides on 16-byte boundaries, and only the 8-bit tile
    set; each breach is HGEMM_ERR_UNSUPPORTED, found before any device is
    touched.  8-bit outputs do not exist (HGEMM_ERR_INVALID_ARG)."""
    h = ctypes.c_void_p()
    E4 = H.HGEMM_E4M3

    def create(M, N, K, lda, ldb, batch=1, sA=0, sB=0, din=E4, dout=H.HGEMM_BF16, **kw):
        opt = H.Options(**{"trans_b": 1, **kw})
        return lib.hgemm_plan_create_ex(ctypes.byref(h), M, N, K, lda, ldb, N, batch, sA, sB,
                                        M * N * batch, din, dout, ctypes.byref(opt))

    assert create(64, 64, 64, 64, 64, trans_b=0) == 2
    assert create(64, 64, 64, 72, 64) == 2          # lda not a multiple of 16
    assert create(64, 64, 40, 48, 40) == 2          # ldb not a multiple of 16
    assert create(64, 64, 64, 64, 64, batch=2, sA=64 * 64 + 8, sB=64 * 64) == 2
    assert create(64, 64, 64, 64, 64, tile_n=192) == 2
    assert create(64, 64, 64, 64, 64, pair_k_blocks=1) == 2
    assert create(8, 64, 64, 64, 64, skinny_tile_n=192) == 2
    assert create(64, 64, 64, 64, 64, force_repack=1) == 2
    assert create(64, 64, 64, 64, 64, din=H.HGEMM_E5M2, trans_b=0) == 2
    assert create(64, 64, 64, 64, 64, dout=H.HGEMM_E4M3) == 1
    assert create(64, 64, 64, 64, 64, dout=H.HGEMM_E5M2) == 1
    # K == 0 writes zeros whatever the layout; a well-formed request reaches
    # the device check
    import torch
    if not torch.cuda.is_available():
        assert create(64, 64, 0, 64, 64, trans_b=0) == 3
        assert create(64, 64, 200, 208, 224) == 3
        assert create(64, 64, 64, 64, 64, din=H.HGEMM_E5M2, batch=2, sA=64 * 64, sB=64 * 64) == 3


def test_attention_argument_checks_need_no_gpu(lib):
    """The attention plan's checks run before any device is touched."""
    h = ctypes.c_void_p()
    bad = [((0, 16, 16, 128, 1.0, 0, H.HGEMM_BF16), 1),     # no heads
           ((2, -1, 16, 128, 1.0, 0, H.HGEMM_BF16), 1),     # negative seq_q
           ((2, 16, 16, 128, 0.0, 0, H.HGEMM_BF16), 1),     # scale 0
           ((2, 16, 16, 128, -1.0, 0, H.HGEMM_BF16), 1),    # negative scale
           ((2, 32, 16, 128, 1.0, 1, H.HGEMM_BF16), 1),     # causal, seq_q > seq_kv
           ((2, 16, 16, 128, 1.0, 2, H.HGEMM_BF16), 1),     # causal not 0 / 1
           ((2, 16, 16, 128, 1.0, 0, H.HGEMM_E4M3), 1),     # 8-bit inputs
           ((2, 16, 16, 64, 1.0, 0, H.HGEMM_BF16), 2),      # head_dim 64
           (((1 << 31) - 1, 16, (1 << 31) - 1, 128, 1.0, 0, H.HGEMM_BF16), 2)]  # K / V past 2^60 bytes
    for args, want in bad:
        assert lib.hgemm_attention_plan_create(ctypes.byref(h), *args) == want, args
    assert lib.hgemm_attention_plan_create(None, 2, 16, 16, 128, 1.0, 0, H.HGEMM_BF16) == 1
    assert lib.hgemm_attention_run(None, None, None, None, None, None) == 1
    assert lib.hgemm_attention_check(None, None) == 1
    assert lib.hgemm_attention_plan_destroy(None) == 0
    import torch
    if not torch.cuda.is_available():
        assert lib.hgemm_attention_plan_create(ctypes.byref(h), 2, 16, 16, 128, 1.0, 0, H.HGEMM_BF16) == 3


def test_valid_request_without_gpu_reports_no_device(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    st, h = _create(*GOOD)
    assert st == 3 and h is None
    assert "device" in H.hgemm_last_error_detail().lower()


def test_python_binding_raises_with_status(lib):
    with pytest.raises(H.HgemmError) as ei:
        H.hgemm_plan_create(-1, 1, 1, 1, 1, 1, 1, 0, 0, 0, H.HGEMM_F16, H.HGEMM_F32)
    assert ei.value.status == 1 and "negative" in str(ei.value)


def test_matmul_front_end_refuses_cpu_tensors():
    import torch

    from tensor_core_dense_swizzled_gb300 import matmul
    a = torch.zeros(4, 4, dtype=torch.float16)
    with pytest.raises((ValueError, TypeError)):
        matmul(a, a)
    with pytest.raises(TypeError):
        matmul(a.float(), a.float())
