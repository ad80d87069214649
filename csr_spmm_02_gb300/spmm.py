"""Thin ctypes binding over the C ABI in ``include/spmm.h``.

Argument marshalling only: every step of the multiplication runs in the CUDA
library ``_lib/libcsr_spmm_gb300.so``.  There is no CPU fallback; if the
library is missing, importing the functions below raises.

Functions carry the C names:

* ``spmm_csr_plan(rowptr, M, nnz, N, kernel=..., items_per_cta=0)`` -> Plan
* ``spmm_csr_f32_exec(plan, K, colind, vals, B, C)``
* ``spmm_csr_bf16f32_exec(plan, K, colind, vals, B_bits, C)``
* ``spmm_csr_f32(M, K, N, rowptr, colind, vals, B, C)``
* ``spmm_csr_bf16f32(M, K, N, rowptr, colind, vals, B_bits, C)``
* ``spmm_csr_validate(rowptr, colind, M, K, nnz)``
* ``spmm_plan_check_device(plan)``

Tensors are CUDA tensors: rowptr/colind int32, vals float32, B float32 (or a
uint16/int16/bfloat16 tensor holding bf16 bits), C float32, all contiguous.
Calls run on the current torch CUDA stream unless ``stream`` is given.
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import build as _build

SPMM_OK = 0
STATUS_NAMES = {0: "SPMM_OK", 1: "SPMM_ERR_INVALID_ARG", 2: "SPMM_ERR_INVALID_CSR",
                3: "SPMM_ERR_UNSUPPORTED", 4: "SPMM_ERR_PLAN_MISMATCH", 5: "SPMM_ERR_CUDA",
                6: "SPMM_ERR_DEVICE_TIMEOUT", 7: "SPMM_ERR_OUT_OF_BOUNDS"}
KERNELS = {"auto": 0, "row": 1, "balanced": 2, "window": 3, "smalln": 4, "window_tc": 5}
KERNEL_NAMES = {1: "row", 2: "balanced", 3: "window", 4: "smalln", 5: "window_tc"}

EXPORTS = ["spmm_csr_plan", "spmm_csr_plan_ex", "spmm_plan_get_info", "spmm_plan_destroy",
           "spmm_csr_f32_exec", "spmm_csr_bf16f32_exec", "spmm_csr_f32", "spmm_csr_bf16f32",
           "spmm_csr_validate", "spmm_plan_check_device", "spmm_plan_set_split_event",
           "spmm_csr_f32_noalloc", "spmm_csr_sddmm_f32", "spmm_csr_fusedmm_f32", "spmm_csr_semiring_f32_exec",
           "spmm_plan_set_group_lanes", "spmm_plan_set_column_tile", "spmm_pool_release",
           "spmm_check_device", "spmm_csr_row_blocks", "spmm_status_string"]


class SpmmError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {STATUS_NAMES.get(status, status)}")


class PlanInfo(ctypes.Structure):
    _fields_ = [("kernel", ctypes.c_int32), ("M", ctypes.c_int32), ("nnz", ctypes.c_int64),
                ("N", ctypes.c_int32), ("max_row_nnz", ctypes.c_int32), ("empty_rows", ctypes.c_int32),
                ("items_per_cta", ctypes.c_int32), ("num_ctas", ctypes.c_int32),
                ("workspace_bytes", ctypes.c_int64), ("group_lanes", ctypes.c_int32),
                ("column_tile", ctypes.c_int32)]


_lib = None


def library_path() -> str:
    return _build.lib_path()


def load(path: str | None = None) -> ctypes.CDLL:
    """Open the CUDA library (raises if it has not been built)."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or library_path()
    if not os.path.exists(p):
        raise RuntimeError(f"CUDA SpMM library not built ({p}); run __graft_entry__.build()")
    lib = ctypes.CDLL(p)
    vp, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
    sig = {
        "spmm_csr_plan": [vp, i32, i64, i32, vp, ctypes.POINTER(vp)],
        "spmm_csr_plan_ex": [vp, i32, i64, i32, i32, i32, vp, ctypes.POINTER(vp)],
        "spmm_plan_get_info": [vp, ctypes.POINTER(PlanInfo)],
        "spmm_plan_destroy": [vp],
        "spmm_csr_f32_exec": [vp, i32, vp, vp, vp, vp, vp],
        "spmm_csr_bf16f32_exec": [vp, i32, vp, vp, vp, vp, vp],
        "spmm_csr_f32": [i32, i32, i32, vp, vp, vp, vp, vp, vp],
        "spmm_csr_bf16f32": [i32, i32, i32, vp, vp, vp, vp, vp, vp],
        "spmm_csr_validate": [vp, vp, i32, i32, i64, vp],
        "spmm_plan_check_device": [vp, vp],
        "spmm_plan_set_split_event": [vp, vp],
        "spmm_csr_f32_noalloc": [i32, i32, i32, i64, vp, vp, vp, vp, vp, vp],
        "spmm_csr_sddmm_f32": [vp, i32, vp, vp, vp, vp, vp],
        "spmm_csr_fusedmm_f32": [vp, i32, vp, vp, vp, vp, vp, vp],
        "spmm_csr_semiring_f32_exec": [vp, i32, vp, vp, vp, vp, i32, i32, vp],
        "spmm_plan_set_group_lanes": [vp, i32],
        "spmm_plan_set_column_tile": [vp, i32],
        "spmm_pool_release": [],
        "spmm_check_device": [vp],
        "spmm_csr_row_blocks": [vp, i32, i32, vp],
        "spmm_status_string": [ctypes.c_int],
    }
    for name, args in sig.items():
        f = getattr(lib, name)
        f.argtypes = args
        f.restype = ctypes.c_char_p if name == "spmm_status_string" else ctypes.c_int
    if path is None:
        _lib = lib
    return lib


def _check(status: int, where: str):
    if status != SPMM_OK:
        raise SpmmError(status, where)


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _ptr(t, dtype, name, allow_none=False):
    if t is None:
        if allow_none:
            return None
        raise ValueError(f"{name} is required")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if dtype is not None and t.dtype not in dtype:
        raise TypeError(f"{name} has dtype {t.dtype}, expected one of {dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return ctypes.c_void_p(t.data_ptr()) if t.numel() else None


def _need(t, n, name):
    """Refuse a buffer smaller than the call will read or write (checked before
    any pointer reaches the library).  Every size the call knows on the host
    is checked this way; the one exception is colind and vals of the one-call
    forms spmm_csr_f32 / spmm_csr_bf16f32, whose length rowptr[M] exists only
    on the device (the caller must size them)."""
    if t is not None and t.numel() < n:
        raise ValueError(f"{name} holds {t.numel()} elements; the call needs at least {n}")


_I32 = (torch.int32,)
_F32 = (torch.float32,)
_BF16_BITS = (torch.uint16, torch.int16, torch.bfloat16) if hasattr(torch, "uint16") else (torch.int16, torch.bfloat16)


class Plan:
    """Owns a ``spmm_plan_t``; keeps the rowptr tensor alive while the plan lives."""

    def __init__(self, handle: int, rowptr: torch.Tensor, M: int = 0, nnz: int = 0, N: int = 0):
        self.handle = ctypes.c_void_p(handle)
        self.rowptr = rowptr
        self.M, self.nnz, self.N = M, nnz, N  # the sizes the plan is bound to

    def info(self) -> dict:
        pi = PlanInfo()
        _check(load().spmm_plan_get_info(self.handle, ctypes.byref(pi)), "spmm_plan_get_info")
        d = {name: getattr(pi, name) for name, _ in PlanInfo._fields_}
        d["kernel"] = KERNEL_NAMES.get(d["kernel"], d["kernel"])
        return d

    def destroy(self):
        if self.handle:
            load().spmm_plan_destroy(self.handle)
            self.handle = ctypes.c_void_p(0)

    def __del__(self):
        try:
            self.destroy()
        except Exception:
            pass


def spmm_csr_plan(rowptr, M, nnz, N, kernel="auto", items_per_cta=0, stream=None) -> Plan:
    _need(rowptr, M + 1, "rowptr")
    out = ctypes.c_void_p()
    st = load().spmm_csr_plan_ex(_ptr(rowptr, _I32, "rowptr"), M, nnz, N, KERNELS[kernel], items_per_cta,
                                 _stream(stream), ctypes.byref(out))
    _check(st, "spmm_csr_plan")
    return Plan(out.value, rowptr, M, nnz, N)


def _need_exec(plan, K, colind, vals, B, C):
    _need(colind, plan.nnz, "colind")
    _need(vals, plan.nnz, "vals")
    _need(B, K * plan.N, "B")
    _need(C, plan.M * plan.N, "C")


def spmm_csr_f32_exec(plan: Plan, K, colind, vals, B, C, stream=None):
    _need_exec(plan, K, colind, vals, B, C)
    _check(load().spmm_csr_f32_exec(plan.handle, K, _ptr(colind, _I32, "colind", True),
                                    _ptr(vals, _F32, "vals", True), _ptr(B, _F32, "B", True),
                                    _ptr(C, _F32, "C"), _stream(stream)), "spmm_csr_f32_exec")
    return C


def spmm_csr_bf16f32_exec(plan: Plan, K, colind, vals, B, C, stream=None):
    _need_exec(plan, K, colind, vals, B, C)
    _check(load().spmm_csr_bf16f32_exec(plan.handle, K, _ptr(colind, _I32, "colind", True),
                                        _ptr(vals, _F32, "vals", True), _ptr(B, _BF16_BITS, "B", True),
                                        _ptr(C, _F32, "C"), _stream(stream)), "spmm_csr_bf16f32_exec")
    return C


def _need_one_call(M, K, N, rowptr, B, C):
    # nnz = rowptr[M] is only known on the device: colind and vals are not checked here
    _need(rowptr, M + 1, "rowptr")
    _need(B, K * N, "B")
    _need(C, M * N, "C")


def spmm_csr_f32(M, K, N, rowptr, colind, vals, B, C, stream=None):
    _need_one_call(M, K, N, rowptr, B, C)
    _check(load().spmm_csr_f32(M, K, N, _ptr(rowptr, _I32, "rowptr"), _ptr(colind, _I32, "colind", True),
                               _ptr(vals, _F32, "vals", True), _ptr(B, _F32, "B", True), _ptr(C, _F32, "C"),
                               _stream(stream)), "spmm_csr_f32")
    return C


def spmm_csr_bf16f32(M, K, N, rowptr, colind, vals, B, C, stream=None):
    _need_one_call(M, K, N, rowptr, B, C)
    _check(load().spmm_csr_bf16f32(M, K, N, _ptr(rowptr, _I32, "rowptr"), _ptr(colind, _I32, "colind", True),
                                   _ptr(vals, _F32, "vals", True), _ptr(B, _BF16_BITS, "B", True),
                                   _ptr(C, _F32, "C"), _stream(stream)), "spmm_csr_bf16f32")
    return C


def spmm_csr_sddmm_f32(plan: Plan, K, colind, C, B, out, stream=None):
    """out[p] = C[i] . B[colind[p]] on A's pattern (fp32)."""
    _need(colind, plan.nnz, "colind")
    _need(C, plan.M * plan.N, "C")
    _need(B, K * plan.N, "B")
    _need(out, plan.nnz, "out")
    _check(load().spmm_csr_sddmm_f32(plan.handle, K, _ptr(colind, _I32, "colind", True), _ptr(C, _F32, "C", True),
                                     _ptr(B, _F32, "B", True), _ptr(out, _F32, "out", True), _stream(stream)),
           "spmm_csr_sddmm_f32")
    return out


def spmm_plan_set_group_lanes(plan: Plan, lanes: int):
    """Lanes (2, 4, 8, 16, 32) that share a row in a SMALLN plan."""
    _check(load().spmm_plan_set_group_lanes(plan.handle, lanes), "spmm_plan_set_group_lanes")


def spmm_plan_set_column_tile(plan: Plan, columns: int):
    """Cap the row/balanced kernels' column tile at `columns` (N-slicing; 0: no cap)."""
    _check(load().spmm_plan_set_column_tile(plan.handle, columns), "spmm_plan_set_column_tile")


ADD_OPS = {"sum": 0, "min": 1, "max": 2}
MUL_OPS = {"mul": 0, "add": 1}


def spmm_csr_semiring_f32_exec(plan: Plan, K, colind, vals, B, C, add="sum", mul="mul", stream=None):
    """C[i, n] = add-reduction over row i of vals[p] mul B[colind[p], n] (fp32).

    add in {"sum", "min", "max"}, mul in {"mul", "add"}; an empty row gives the
    identity of add (0, +inf, -inf)."""
    _need_exec(plan, K, colind, vals, B, C)
    _check(load().spmm_csr_semiring_f32_exec(plan.handle, K, _ptr(colind, _I32, "colind", True),
                                             _ptr(vals, _F32, "vals", True), _ptr(B, _F32, "B", True),
                                             _ptr(C, _F32, "C"), ADD_OPS[add], MUL_OPS[mul], _stream(stream)),
           "spmm_csr_semiring_f32_exec")
    return C


def spmm_csr_fusedmm_f32(plan: Plan, K, colind, C, B, D, E, stream=None):
    """E = SDDMM(C, B on A's pattern) . D without storing the SDDMM values (fp32)."""
    _need(colind, plan.nnz, "colind")
    _need(C, plan.M * plan.N, "C")
    _need(B, K * plan.N, "B")
    _need(D, K * plan.N, "D")
    _need(E, plan.M * plan.N, "E")
    _check(load().spmm_csr_fusedmm_f32(plan.handle, K, _ptr(colind, _I32, "colind", True), _ptr(C, _F32, "C", True),
                                       _ptr(B, _F32, "B", True), _ptr(D, _F32, "D", True), _ptr(E, _F32, "E"),
                                       _stream(stream)), "spmm_csr_fusedmm_f32")
    return E


def spmm_csr_f32_noalloc(M, K, N, nnz, rowptr, colind, vals, B, C, stream=None):
    """C = A . B (fp32) with the library's fixed scratch array: no allocation anywhere.

    nnz must equal rowptr[M]; the library checks that on the device and
    reports a mismatch (and any bounded wait that gave up) through
    ``spmm_check_device``, not through this call's status."""
    _need_one_call(M, K, N, rowptr, B, C)
    _need(colind, nnz, "colind")
    _need(vals, nnz, "vals")
    _check(load().spmm_csr_f32_noalloc(M, K, N, nnz, _ptr(rowptr, _I32, "rowptr"), _ptr(colind, _I32, "colind", True),
                                       _ptr(vals, _F32, "vals", True), _ptr(B, _F32, "B", True), _ptr(C, _F32, "C"),
                                       _stream(stream)), "spmm_csr_f32_noalloc")
    return C


def spmm_check_device(stream=None) -> int:
    """Synchronise, read and clear the one-call forms' device error word (a status code)."""
    return load().spmm_check_device(_stream(stream))


def spmm_csr_row_blocks(rowptr, parts: int):
    """First row of each of `parts` row blocks (numpy int32[parts + 1]) for
    splitting one A over `parts` GPUs; rowptr is a host (numpy) int32 array."""
    import numpy as np
    rp = np.ascontiguousarray(rowptr, dtype=np.int32)
    if rp.ndim != 1 or rp.size < 1:
        raise ValueError("rowptr must be a 1-D array of M + 1 entries")
    out = np.empty(max(parts, 0) + 1, dtype=np.int32)
    _check(load().spmm_csr_row_blocks(ctypes.c_void_p(rp.ctypes.data), rp.size - 1, parts,
                                      ctypes.c_void_p(out.ctypes.data)), "spmm_csr_row_blocks")
    return out


def spmm_pool_release() -> None:
    """Hand back the device memory the one-call forms' pools keep between calls."""
    _check(load().spmm_pool_release(), "spmm_pool_release")


def spmm_csr_validate(rowptr, colind, M, K, nnz, stream=None) -> int:
    """Return the status code (SPMM_OK or SPMM_ERR_INVALID_CSR); raise on other errors."""
    st = load().spmm_csr_validate(_ptr(rowptr, _I32, "rowptr"), _ptr(colind, _I32, "colind", True), M, K, nnz,
                                  _stream(stream))
    if st not in (0, 2):
        raise SpmmError(st, "spmm_csr_validate")
    return st


def spmm_plan_check_device(plan: Plan, stream=None) -> int:
    return load().spmm_plan_check_device(plan.handle, _stream(stream))


def spmm_plan_set_split_event(plan: Plan, event) -> None:
    """Record `event` (a torch.cuda.Event, or None) after the main kernel of every exec."""
    handle = None
    if event is not None:
        if not event.cuda_event:
            event.record()  # torch creates the CUDA event on its first record
        handle = ctypes.c_void_p(event.cuda_event)
    plan._split_event = event  # keep it alive while it is set
    _check(load().spmm_plan_set_split_event(plan.handle, handle), "spmm_plan_set_split_event")


def spmm_status_string(status: int) -> str:
    return load().spmm_status_string(status).decode()
