"""GB300-native single-precision GEMM: C = alpha*A*B + beta*C (row-major FP32).

The compute path is the C-ABI CUDA library built from ``csrc/`` for sm_103a;
``sgemm`` below only marshals arguments to it.  Importing the package does not
load the library; the first call does, and raises if it is missing.
"""
from .binding import sgemm, sgemm_ex, SgemmError, PATH_AUTO, PATH_FFMA, PATH_TF32X3  # noqa: F401

__all__ = ["sgemm", "sgemm_ex", "SgemmError", "PATH_AUTO", "PATH_FFMA", "PATH_TF32X3"]
