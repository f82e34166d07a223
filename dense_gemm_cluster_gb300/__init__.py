"""GB300-native (sm_103a) cluster GEMM: C = alpha*A*B + beta*C with bf16 operands.

Submodules:
  gemm     ctypes binding of the C ABI (include/densegemm.h); needs the built library
  build    nvcc build of libdensegemm.so
  inputs   seeded synthetic inputs (no GEMM arithmetic)
  traffic  analytic L2->SM operand-byte accounting

Importing the package does not load the CUDA library; ``from
dense_gemm_cluster_gb300 import gemm`` does, and fails if it is not built.
"""
