"""libhgemm: half-precision tensor-core GEMM for GB300 (sm_103a).

* :mod:`.hgemm` -- ctypes binding of the C ABI in ``include/hgemm.h``;
* :func:`matmul` -- a torch-tensor front end (plain, transposed-B, 8-bit and
  fused-epilogue products), :func:`matmul_cache_clear`;
* :mod:`.inputs` -- seeded synthetic workloads;
* :mod:`.build` -- builds ``libhgemm.so`` with nvcc.
"""
from .torch_gemm import matmul, matmul_cache_clear  # noqa: F401
