"""fgemm: dense half-precision GEMM on GB300 (sm_103a) -- classical and
Strassen-like low-complexity forms behind a C ABI, with an analytical picker.

    from complexity_matmul_tcgen05_gb300 import fgemm
    C = fgemm.matmul(A, B, epilogue="scale_bias", bias=b)        # algo="auto"

Submodules: ``fgemm`` (the binding), ``inputs`` (seeded synthetic inputs),
``build`` (compiles the C library with nvcc).  The binding raises if the
library has not been built.
"""
