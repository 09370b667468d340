"""GB300 (sm_103a) library for the UFP4 hot path: fused Random Hadamard
Transform + block-scaled 4-bit quantizer and the quantized GEMM consumer.

Submodules:
  ufp4    -- ctypes binding of libufp4.so (include/ufp4.h), same names as the C ABI
  build   -- in-tree nvcc build of libufp4.so
  inputs  -- seeded synthetic inputs (numpy only)
"""
__all__ = ["ufp4", "build", "inputs"]
