"""GB300-native CSR SpMM: C[M x N] = A[M x K, CSR] . B[K x N, row-major].

Importing the package loads nothing compiled.  The CUDA library and its thin
ctypes binding live in :mod:`csr_spmm_02_gb300.spmm`; seeded synthetic inputs
in :mod:`csr_spmm_02_gb300.gen`.
"""
