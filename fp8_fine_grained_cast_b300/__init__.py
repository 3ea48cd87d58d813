"""Fine-grained FP8 (E4M3) quantization and block-scaled FP8 GEMM for B300 (sm_103a).

The compute lives in libfp8fg.so (CUDA kernels behind the C ABI of include/fp8fg.h).
``_lib`` is the ctypes binding with the C names; ``ops`` wraps it for torch tensors;
``inputs`` generates the seeded synthetic workloads.
"""
from ._lib import Fp8fgError, LIB_PATH  # noqa: F401

__version__ = "0.1.0"
