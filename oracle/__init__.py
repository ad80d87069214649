"""CPU oracle for CSR SpMM -- TEST INFRASTRUCTURE, not part of the product.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
(and ``--impl reference``) leg may import this package.  It shares no code
with the CUDA library (``csr_spmm_02_gb300``) and imports nothing from it.

The arithmetic lives in ``spmm_oracle.c``: a single-threaded double-precision
CSR row loop that follows the SpMM definition (page "Performance
Optimization of Deep Learning Sparse Matrix Kernels on Intel Max Series
GPU", SPMM section, Fig. 5 and Algorithm 2).  This module compiles it with
gcc on first use and calls it through ctypes.

Functions
---------
``build()``            compile the C oracle (idempotent).
``spmm_reference``     C and the magnitude sum S for all rows or a row list.
``sddmm_reference``    the sampled dot products out[p] = C_i . B_j and their bound.
``fusedmm_reference``  E = (SDDMM values) . D and its bound.
``semiring_reference`` C with a general (+) / (x) pair (sum/min/max over
                       multiply/add), and S for the sum.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "spmm_oracle.c")
_LIBDIR = os.path.join(_HERE, "_lib")
_LIB = os.path.join(_LIBDIR, "libspmm_oracle.so")
_lock = threading.Lock()
_handle = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (no fast-math, no FMA contraction)."""
    os.makedirs(_LIBDIR, exist_ok=True)
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c99", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
           "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def load_library(path: str) -> ctypes.CDLL:
    """Open an oracle library (the default one, or a test's modified copy)."""
    lib = ctypes.CDLL(path)
    f = lib.spmm_oracle_rows_f64
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_void_p,
                  ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32,
                  ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p]
    vp, i32 = ctypes.c_void_p, ctypes.c_int32
    g = lib.sddmm_oracle_f64
    g.restype = ctypes.c_int
    g.argtypes = [i32, i32, i32, vp, vp, vp, vp, vp, vp]
    h = lib.fusedmm_oracle_f64
    h.restype = ctypes.c_int
    h.argtypes = [i32, i32, i32, vp, vp, vp, vp, vp, vp, vp, vp]
    k = lib.spmm_semiring_oracle_f64
    k.restype = ctypes.c_int
    k.argtypes = [i32, i32, i32, vp, vp, vp, vp, i32, i32, vp, vp]
    return lib


def _lib():
    global _handle
    with _lock:
        if _handle is None:
            _handle = load_library(build())
    return _handle


def _ptr(a):
    return ctypes.c_void_p(a.ctypes.data) if a is not None else None


def spmm_reference(rowptr, colind, vals, B, *, b_dtype="f32", rows=None, with_bound=True,
                   library=None):
    """Return (C, S) in float64 for the listed rows (all rows when rows is None).

    rowptr int32[M+1], colind int32[nnz], vals float32[nnz]; B float32[K, N],
    or uint16[K, N] bf16 bit patterns when b_dtype == "bf16".
    C[t, n] = sum_p vals[p] * B[colind[p], n] over row rows[t];
    S[t, n] = sum_p |vals[p] * B[colind[p], n]| (None when with_bound is False).
    `library` selects another oracle build (see ``load_library``).
    """
    rowptr = np.ascontiguousarray(rowptr, dtype=np.int32)
    colind = np.ascontiguousarray(colind, dtype=np.int32)
    vals = np.ascontiguousarray(vals, dtype=np.float32)
    if b_dtype == "f32":
        B = np.ascontiguousarray(B, dtype=np.float32)
    elif b_dtype == "bf16":
        B = np.ascontiguousarray(B, dtype=np.uint16)
    else:
        raise ValueError(b_dtype)
    if B.ndim != 2:
        raise ValueError("B must be 2-D")
    M = len(rowptr) - 1
    K, N = B.shape
    if rows is not None:
        rows = np.ascontiguousarray(rows, dtype=np.int32)
        nrows = len(rows)
    else:
        nrows = M
    C = np.empty((nrows, N), dtype=np.float64)
    S = np.empty((nrows, N), dtype=np.float64) if with_bound else None
    lib = library if library is not None else _lib()
    rc = lib.spmm_oracle_rows_f64(M, K, N, _ptr(rowptr), _ptr(colind), _ptr(vals), _ptr(B),
                                  1 if b_dtype == "bf16" else 0, _ptr(rows), nrows,
                                  _ptr(C), _ptr(S))
    if rc == -2:
        raise ValueError("oracle: invalid CSR (decreasing rowptr or column index outside [0, K))")
    if rc != 0:
        raise ValueError("oracle rejected its arguments")
    return C, S


def _check_rc(rc):
    if rc == -2:
        raise ValueError("oracle: invalid CSR (decreasing rowptr or column index outside [0, K))")
    if rc != 0:
        raise ValueError("oracle rejected its arguments")


def sddmm_reference(rowptr, colind, C, B, *, library=None):
    """(out, S): out[p] = C[i] . B[colind[p]] for each stored p of row i, float64."""
    rowptr = np.ascontiguousarray(rowptr, dtype=np.int32)
    colind = np.ascontiguousarray(colind, dtype=np.int32)
    C = np.ascontiguousarray(C, dtype=np.float32)
    B = np.ascontiguousarray(B, dtype=np.float32)
    M = len(rowptr) - 1
    K, N = B.shape
    if C.shape != (M, N):
        raise ValueError("C must be M x N with B's width")
    out = np.empty(len(colind), dtype=np.float64)
    S = np.empty(len(colind), dtype=np.float64)
    lib = library if library is not None else _lib()
    _check_rc(lib.sddmm_oracle_f64(M, K, N, _ptr(rowptr), _ptr(colind), _ptr(C), _ptr(B), _ptr(out), _ptr(S)))
    return out, S


def fusedmm_reference(rowptr, colind, C, B, D, *, library=None, with_values=False):
    """(E, S[, a]): E = SDDMM(C, B on A's pattern) . D in float64, its bound S, and the values a."""
    rowptr = np.ascontiguousarray(rowptr, dtype=np.int32)
    colind = np.ascontiguousarray(colind, dtype=np.int32)
    C = np.ascontiguousarray(C, dtype=np.float32)
    B = np.ascontiguousarray(B, dtype=np.float32)
    D = np.ascontiguousarray(D, dtype=np.float32)
    M = len(rowptr) - 1
    K, N = B.shape
    if C.shape != (M, N) or D.shape != (K, N):
        raise ValueError("C must be M x N and D K x N, with B's width")
    E = np.empty((M, N), dtype=np.float64)
    S = np.empty((M, N), dtype=np.float64)
    a = np.empty(len(colind), dtype=np.float64)
    lib = library if library is not None else _lib()
    _check_rc(lib.fusedmm_oracle_f64(M, K, N, _ptr(rowptr), _ptr(colind), _ptr(C), _ptr(B), _ptr(D),
                                     _ptr(E), _ptr(S), _ptr(a)))
    return (E, S, a) if with_values else (E, S)


SEMIRING_ADD = {"sum": 0, "min": 1, "max": 2}
SEMIRING_MUL = {"mul": 0, "add": 1}


def semiring_reference(rowptr, colind, vals, B, add="sum", mul="mul", *, library=None):
    """(C, S): C[i, n] = add-reduction over row i of vals[p] mul B[colind[p], n], float64.

    add in {"sum", "min", "max"}, mul in {"mul", "add"}; an empty row gives the
    identity of add (0, +inf, -inf).  S (the magnitude sum) is filled for "sum"
    and zero otherwise.  B is float32."""
    rowptr = np.ascontiguousarray(rowptr, dtype=np.int32)
    colind = np.ascontiguousarray(colind, dtype=np.int32)
    vals = np.ascontiguousarray(vals, dtype=np.float32)
    B = np.ascontiguousarray(B, dtype=np.float32)
    M = len(rowptr) - 1
    K, N = B.shape
    C = np.empty((M, N), dtype=np.float64)
    S = np.empty((M, N), dtype=np.float64)
    lib = library if library is not None else _lib()
    _check_rc(lib.spmm_semiring_oracle_f64(M, K, N, _ptr(rowptr), _ptr(colind), _ptr(vals), _ptr(B),
                                           SEMIRING_ADD[add], SEMIRING_MUL[mul], _ptr(C), _ptr(S)))
    return C, S
