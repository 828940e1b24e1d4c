"""ctypes binding of libhgemm's C ABI (include/hgemm.h).

Argument marshalling only: every function below forwards to the entry point
of the same name in ``libhgemm.so``; all arithmetic runs in the library's CUDA
kernels.  Torch tensors are accepted where the C ABI takes a pointer (their
``data_ptr()`` is passed) and torch streams where it takes a ``cudaStream_t``.
If the shared library is missing, every call raises -- there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
import threading

__all__ = [
    "HGEMM_F16", "HGEMM_BF16", "HGEMM_F32", "HGEMM_E4M3", "HGEMM_E5M2", "HGEMM_PATH_EMPTY", "HGEMM_PATH_ZERO_FILL",
    "HGEMM_PATH_TILED", "HGEMM_PATH_SKINNY", "HgemmError", "Options", "PlanInfo", "lib_path",
    "load", "hgemm_plan_create", "hgemm_plan_create_ex", "hgemm_run", "hgemm_run_host",
    "hgemm_check", "hgemm_plan_destroy", "hgemm_plan_get_info", "hgemm", "hgemm_cache_clear",
    "hgemm_watchdog_selftest", "hgemm_skinny_noalloc", "hgemm_skinny_noalloc_check",
    "hgemm_status_string", "Epilogue",
    "hgemm_run_ex", "HGEMM_ACT_NONE", "HGEMM_ACT_RELU", "HGEMM_ACT_GELU", "HGEMM_ACT_GELU_TANH",
    "hgemm_last_error_detail", "hgemm_version", "hgemm_attention_plan_create",
    "hgemm_attention_run", "hgemm_attention_run_host", "hgemm_attention_check",
    "hgemm_attention_plan_destroy",
    "STATUS",
]

HGEMM_F16, HGEMM_BF16, HGEMM_F32, HGEMM_E4M3, HGEMM_E5M2 = 0, 1, 2, 3, 4
HGEMM_PATH_EMPTY, HGEMM_PATH_ZERO_FILL, HGEMM_PATH_TILED, HGEMM_PATH_SKINNY = 0, 1, 2, 3
STATUS = {
    0: "HGEMM_OK", 1: "HGEMM_ERR_INVALID_ARG", 2: "HGEMM_ERR_UNSUPPORTED",
    3: "HGEMM_ERR_NO_DEVICE", 4: "HGEMM_ERR_CUDA", 5: "HGEMM_ERR_OOM", 6: "HGEMM_ERR_TIMEOUT",
    7: "HGEMM_ERR_INTERNAL",
}

_HERE = os.path.dirname(os.path.abspath(__file__))
_lock = threading.Lock()
_lib = None


def lib_path() -> str:
    return os.path.join(_HERE, "libhgemm.so")


class HgemmError(RuntimeError):
    def __init__(self, status: int, where: str, detail: str):
        self.status = status
        self.name = STATUS.get(status, f"status {status}")
        super().__init__(f"{where}: {self.name}: {detail}")


class Options(ctypes.Structure):
    _fields_ = [
        ("force_path", ctypes.c_int),
        ("force_generic_store", ctypes.c_int),
        ("force_repack", ctypes.c_int),
        ("tile_n", ctypes.c_int),
        ("split_k", ctypes.c_int),
        ("timeout_ns", ctypes.c_uint64),
        ("cta_pair", ctypes.c_int),
        ("skinny_tile_n", ctypes.c_int),
        ("no_tail_split", ctypes.c_int),
        ("pair_k_blocks", ctypes.c_int),
        ("tail_mode", ctypes.c_int),
        ("skinny_stream_k", ctypes.c_int),
        ("skinny_prefetch", ctypes.c_int),
        ("group_m", ctypes.c_int),
        ("trans_b", ctypes.c_int),
        ("tiled_epi_warps", ctypes.c_int),
        ("debug_withhold_kb", ctypes.c_int),
        ("debug_checks", ctypes.c_int),
    ]


HGEMM_ACT_NONE, HGEMM_ACT_RELU, HGEMM_ACT_GELU, HGEMM_ACT_GELU_TANH = 0, 1, 2, 3


class Epilogue(ctypes.Structure):
    """hgemm_epilogue_t: D = act(alpha * rs[i] * cs[j] * (A.B) + beta * C + bias[j]).
    Pointers are device addresses (ints) or None."""
    _fields_ = [
        ("alpha", ctypes.c_float),
        ("beta", ctypes.c_float),
        ("bias", ctypes.c_void_p),
        ("row_scale", ctypes.c_void_p),
        ("col_scale", ctypes.c_void_p),
        ("activation", ctypes.c_int),
    ]


class PlanInfo(ctypes.Structure):
    _fields_ = [
        ("path", ctypes.c_int),
        ("tile_m", ctypes.c_int),
        ("tile_n", ctypes.c_int),
        ("tile_k", ctypes.c_int),
        ("stages", ctypes.c_int),
        ("split_k", ctypes.c_int),
        ("grid", ctypes.c_int),
        ("repack_a", ctypes.c_int),
        ("repack_b", ctypes.c_int),
        ("tma_store", ctypes.c_int),
        ("kernels_per_run", ctypes.c_int),
        ("workspace_bytes", ctypes.c_int64),
        ("tail_split", ctypes.c_int),
        ("wide_boxes", ctypes.c_int),
        ("trans_b", ctypes.c_int),
        ("stream_k", ctypes.c_int),
        ("epi_warps", ctypes.c_int),
        ("epi_warps_epilogue", ctypes.c_int),
        ("host_chunks", ctypes.c_int),
    ]

    def as_dict(self) -> dict:
        return {name: getattr(self, name) for name, _ in self._fields_}


def load():
    """Loads libhgemm.so (built by ``__graft_entry__.build()``); raises if absent."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = lib_path()
        if not os.path.exists(path):
            raise ImportError(f"{path} is missing: build the CUDA library first "
                              "(python -c 'import __graft_entry__ as g; g.build()')")
        lib = ctypes.CDLL(path)
        i64, p, st = ctypes.c_int64, ctypes.c_void_p, ctypes.c_int
        plan_p = ctypes.POINTER(ctypes.c_void_p)
        lib.hgemm_plan_create.argtypes = [plan_p, i64, i64, i64, i64, i64, i64, i64, i64, i64, i64,
                                          ctypes.c_int, ctypes.c_int]
        lib.hgemm_plan_create_ex.argtypes = lib.hgemm_plan_create.argtypes + [ctypes.POINTER(Options)]
        lib.hgemm_run.argtypes = [p, p, p, p, p]
        lib.hgemm_run_host.argtypes = [p, p, p, p, p]
        lib.hgemm_run_ex.argtypes = [p, p, p, p, p, ctypes.POINTER(Epilogue)]
        lib.hgemm_check.argtypes = [p, p]
        lib.hgemm_plan_destroy.argtypes = [p]
        lib.hgemm_plan_get_info.argtypes = [p, ctypes.POINTER(PlanInfo)]
        lib.hgemm.argtypes = [p, p, p, i64, i64, i64, i64, i64, i64, i64, i64, i64, i64,
                              ctypes.c_int, ctypes.c_int, p]
        lib.hgemm_cache_clear.argtypes = []
        lib.hgemm_watchdog_selftest.argtypes = [ctypes.c_uint64, p, ctypes.POINTER(ctypes.c_int32)]
        lib.hgemm_skinny_noalloc.argtypes = [p, p, p, i64, i64, i64, i64, i64, i64, ctypes.c_int,
                                             ctypes.c_int, p]
        lib.hgemm_skinny_noalloc_check.argtypes = [p]
        lib.hgemm_attention_plan_create.argtypes = [plan_p, i64, i64, i64, i64, ctypes.c_float,
                                                    ctypes.c_int, ctypes.c_int]
        lib.hgemm_attention_run.argtypes = [p, p, p, p, p, p]
        lib.hgemm_attention_run_host.argtypes = [p, p, p, p, p, p]
        lib.hgemm_attention_check.argtypes = [p, p]
        lib.hgemm_attention_plan_destroy.argtypes = [p]
        for name in ("hgemm_plan_create", "hgemm_plan_create_ex", "hgemm_run", "hgemm_run_host",
                     "hgemm_run_ex", "hgemm_attention_plan_create", "hgemm_attention_run",
                     "hgemm_attention_run_host", "hgemm_attention_check",
                     "hgemm_attention_plan_destroy",
                     "hgemm_check", "hgemm_plan_destroy", "hgemm_plan_get_info", "hgemm",
                     "hgemm_cache_clear", "hgemm_watchdog_selftest", "hgemm_skinny_noalloc",
                     "hgemm_skinny_noalloc_check"):
            getattr(lib, name).restype = st
        lib.hgemm_status_string.argtypes = [ctypes.c_int]
        lib.hgemm_status_string.restype = ctypes.c_char_p
        lib.hgemm_last_error_detail.argtypes = []
        lib.hgemm_last_error_detail.restype = ctypes.c_char_p
        lib.hgemm_version.argtypes = []
        lib.hgemm_version.restype = ctypes.c_int32
        _lib = lib
        return lib


def _ptr(x) -> int | None:
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(s) -> int | None:
    if s is None:
        try:
            import torch
            if torch.cuda.is_available():
                return torch.cuda.current_stream().cuda_stream
        except Exception:  # pragma: no cover - torch without CUDA
            pass
        return None
    if isinstance(s, int):
        return s
    return s.cuda_stream


def _check(status: int, where: str):
    if status != 0:
        detail = load().hgemm_last_error_detail()
        raise HgemmError(status, where, detail.decode() if detail else "")


def hgemm_plan_create(M, N, K, lda, ldb, ldc, batch, strideA, strideB, strideC, dtype_in, dtype_out) -> int:
    lib = load()
    h = ctypes.c_void_p()
    _check(lib.hgemm_plan_create(ctypes.byref(h), M, N, K, lda, ldb, ldc, batch, strideA, strideB,
                                 strideC, dtype_in, dtype_out), "hgemm_plan_create")
    return h.value


def hgemm_plan_create_ex(M, N, K, lda, ldb, ldc, batch, strideA, strideB, strideC, dtype_in,
                         dtype_out, options: Options | None = None) -> int:
    lib = load()
    h = ctypes.c_void_p()
    opt = ctypes.byref(options) if options is not None else None
    _check(lib.hgemm_plan_create_ex(ctypes.byref(h), M, N, K, lda, ldb, ldc, batch, strideA,
                                    strideB, strideC, dtype_in, dtype_out, opt),
           "hgemm_plan_create_ex")
    return h.value


def hgemm_run(plan: int, A, B, C, stream=None):
    _check(load().hgemm_run(plan, _ptr(A), _ptr(B), _ptr(C), _stream(stream)), "hgemm_run")


def hgemm_run_ex(plan: int, A, B, C, epilogue=None, stream=None):
    """hgemm_run with a fused epilogue (an Epilogue, or None).  Vector
    arguments of the Epilogue may be given as tensors: they are converted to
    device addresses here (the caller keeps the tensors alive)."""
    ep = None
    if epilogue is not None:
        ep = Epilogue(float(getattr(epilogue, "alpha", 1.0)), float(getattr(epilogue, "beta", 0.0)),
                      _ptr(epilogue.bias) if getattr(epilogue, "bias", None) is not None else None,
                      _ptr(epilogue.row_scale) if getattr(epilogue, "row_scale", None) is not None else None,
                      _ptr(epilogue.col_scale) if getattr(epilogue, "col_scale", None) is not None else None,
                      int(getattr(epilogue, "activation", 0)))
    _check(load().hgemm_run_ex(plan, _ptr(A), _ptr(B), _ptr(C), _stream(stream),
                               ctypes.byref(ep) if ep is not None else None), "hgemm_run_ex")


def hgemm_run_host(plan: int, A_host, B_host, C_host, stream=None):
    _check(load().hgemm_run_host(plan, _ptr(A_host), _ptr(B_host), _ptr(C_host), _stream(stream)),
           "hgemm_run_host")


def hgemm_check(plan: int, stream=None) -> int:
    """Returns the status (0 or HGEMM_ERR_TIMEOUT=6 ...) instead of raising,
    so callers can test for a watchdog timeout."""
    return load().hgemm_check(plan, _stream(stream))


def hgemm_plan_destroy(plan: int):
    _check(load().hgemm_plan_destroy(plan), "hgemm_plan_destroy")


def hgemm_plan_get_info(plan: int) -> dict:
    info = PlanInfo()
    _check(load().hgemm_plan_get_info(plan, ctypes.byref(info)), "hgemm_plan_get_info")
    return info.as_dict()


def hgemm(A, B, C, M, N, K, lda, ldb, ldc, batch, strideA, strideB, strideC, dtype_in, dtype_out,
          stream=None):
    _check(load().hgemm(_ptr(A), _ptr(B), _ptr(C), M, N, K, lda, ldb, ldc, batch, strideA, strideB,
                        strideC, dtype_in, dtype_out, _stream(stream)), "hgemm")


def hgemm_cache_clear():
    _check(load().hgemm_cache_clear(), "hgemm_cache_clear")


def hgemm_watchdog_selftest(timeout_ns: int, stream=None) -> tuple[int, int]:
    """Returns ``(status, device_code)``."""
    code = ctypes.c_int32(0)
    st = load().hgemm_watchdog_selftest(timeout_ns, _stream(stream), ctypes.byref(code))
    return st, code.value


def hgemm_skinny_noalloc(A, B, C, M, N, K, lda, ldb, ldc, dtype_in, dtype_out, stream=None):
    """Small-M product that allocates no device memory (its scratch is a fixed
    array inside the library); see include/hgemm.h for its limits."""
    _check(load().hgemm_skinny_noalloc(_ptr(A), _ptr(B), _ptr(C), M, N, K, lda, ldb, ldc,
                                       dtype_in, dtype_out, _stream(stream)),
           "hgemm_skinny_noalloc")


def hgemm_skinny_noalloc_check(stream=None) -> int:
    """Status of the last hgemm_skinny_noalloc product on the current device
    (0, or HGEMM_ERR_TIMEOUT=6); returned instead of raised, like hgemm_check."""
    return load().hgemm_skinny_noalloc_check(_stream(stream))


def hgemm_status_string(status: int) -> str:
    return load().hgemm_status_string(status).decode()


def hgemm_last_error_detail() -> str:
    d = load().hgemm_last_error_detail()
    return d.decode() if d else ""


def hgemm_version() -> int:
    return load().hgemm_version()


# ---------------------------------------------------------------- attention

def hgemm_attention_plan_create(batch_heads, seq_q, seq_kv, head_dim, scale, causal, dtype) -> int:
    lib = load()
    h = ctypes.c_void_p()
    _check(lib.hgemm_attention_plan_create(ctypes.byref(h), batch_heads, seq_q, seq_kv, head_dim,
                                           float(scale), int(causal), dtype),
           "hgemm_attention_plan_create")
    return h.value


def hgemm_attention_run(plan: int, Q, K, V, O, stream=None):
    _check(load().hgemm_attention_run(plan, _ptr(Q), _ptr(K), _ptr(V), _ptr(O), _stream(stream)),
           "hgemm_attention_run")


def hgemm_attention_run_host(plan: int, Q_host, K_host, V_host, O_host, stream=None):
    _check(load().hgemm_attention_run_host(plan, _ptr(Q_host), _ptr(K_host), _ptr(V_host),
                                           _ptr(O_host), _stream(stream)),
           "hgemm_attention_run_host")


def hgemm_attention_check(plan: int, stream=None) -> int:
    """Status instead of an exception (HGEMM_ERR_TIMEOUT = 6 after a watchdog timeout)."""
    return load().hgemm_attention_check(plan, _stream(stream))


def hgemm_attention_plan_destroy(plan: int):
    _check(load().hgemm_attention_plan_destroy(plan), "hgemm_attention_plan_destroy")
