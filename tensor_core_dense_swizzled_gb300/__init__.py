"""libhgemm: half-precision tensor-core GEMM for GB300 (sm_103a).

* :mod:`.hgemm` -- ctypes binding of the C ABI in ``include/hgemm.h``;
* :func:`matmul` -- a torch-tensor convenience over the one-shot ``hgemm`` call;
* :mod:`.inputs` -- seeded synthetic workloads;
* :mod:`.build` -- builds ``libhgemm.so`` with nvcc.
"""
from .torch_gemm import matmul  # noqa: F401
