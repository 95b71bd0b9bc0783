"""GB300 (sm_103a) dense half-precision GEMM behind a small C ABI.

Submodules:
  hgemm      ctypes binding of include/hgemm.h (loads libhgemm.so; fails loudly if missing)
  build      nvcc build of libhgemm.so
  workloads  seeded synthetic inputs and the workload table
"""
__version__ = "0.1.0"
