"""The C-ABI library on a machine without a GPU: it loads, exports every
symbol include/spmm.h declares, and rejects bad arguments before any CUDA call."""
import ctypes
import os
import re

import pytest

import __graft_entry__
from csr_spmm_02_gb300 import spmm

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "spmm.h")


@pytest.fixture(scope="module")
def lib():
    __graft_entry__.build()
    return spmm.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[\w\s\*]+?\b(spmm_\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_binding_exports():
    assert declared_functions() == sorted(spmm.EXPORTS)


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_status_strings(lib):
    for code, name in spmm.STATUS_NAMES.items():
        assert spmm.spmm_status_string(code) == name
    assert spmm.spmm_status_string(99) == "SPMM_ERR_UNKNOWN"


def test_argument_errors_without_cuda(lib):
    out = ctypes.c_void_p()
    null = ctypes.c_void_p()
    # negative sizes, NULL output, bad option values: INVALID_ARG
    assert lib.spmm_csr_plan(null, -1, 0, 4, null, ctypes.byref(out)) == 1
    assert lib.spmm_csr_plan(null, 4, 0, -1, null, ctypes.byref(out)) == 1
    assert lib.spmm_csr_plan(null, 4, 0, 4, null, None) == 1
    assert lib.spmm_csr_plan(null, 4, 0, 4, null, ctypes.byref(out)) == 1  # NULL rowptr with M > 0
    assert lib.spmm_csr_plan_ex(ctypes.c_void_p(16), 4, 0, 4, 7, 0, null, ctypes.byref(out)) == 1
    assert lib.spmm_csr_plan_ex(ctypes.c_void_p(16), 4, 0, 4, 0, 300, null, ctypes.byref(out)) == 1
    # M or nnz beyond SPMM_MAX_EXTENT (2^31 - 65536): UNSUPPORTED, at every entry point
    big = (1 << 31) - 65536 + 1
    assert lib.spmm_csr_plan(ctypes.c_void_p(16), 4, 1 << 31, 4, null, ctypes.byref(out)) == 3
    assert lib.spmm_csr_plan(ctypes.c_void_p(16), 4, big, 4, null, ctypes.byref(out)) == 3
    assert lib.spmm_csr_plan(ctypes.c_void_p(16), big, 4, 4, null, ctypes.byref(out)) == 3
    assert lib.spmm_csr_f32_noalloc(4, 4, 4, big, ctypes.c_void_p(16), ctypes.c_void_p(16), ctypes.c_void_p(16),
                                    ctypes.c_void_p(16), ctypes.c_void_p(16), null) == 3
    assert lib.spmm_csr_f32_noalloc(big, 4, 4, 4, ctypes.c_void_p(16), ctypes.c_void_p(16), ctypes.c_void_p(16),
                                    ctypes.c_void_p(16), ctypes.c_void_p(16), null) == 3
    assert lib.spmm_csr_validate(ctypes.c_void_p(16), ctypes.c_void_p(16), big, 4, 4, null) == 3
    assert lib.spmm_csr_validate(ctypes.c_void_p(16), ctypes.c_void_p(16), 4, 4, big, null) == 3
    # exec without a plan: PLAN_MISMATCH
    assert lib.spmm_csr_f32_exec(null, 4, null, null, null, null, null) == 4
    assert lib.spmm_csr_bf16f32_exec(null, 4, null, null, null, null, null) == 4
    # one-call forms: negative sizes rejected, M = 0 or N = 0 is a no-op success
    assert lib.spmm_csr_f32(-1, 4, 4, null, null, null, null, null, null) == 1
    assert lib.spmm_csr_f32(0, 4, 4, null, null, null, null, null, null) == 0
    assert lib.spmm_csr_bf16f32(4, 4, 0, null, null, null, null, null, null) == 0
    assert lib.spmm_csr_validate(null, null, 4, 4, 0, null) == 1
    assert lib.spmm_csr_validate(ctypes.c_void_p(16), null, -1, 4, 0, null) == 1
    assert lib.spmm_plan_destroy(null) == 0
    assert lib.spmm_plan_check_device(null, null) == 1


def test_binding_refuses_cpu_tensors(lib):
    import torch
    with pytest.raises(ValueError):
        spmm.spmm_csr_plan(torch.zeros(5, dtype=torch.int32), 4, 0, 8)


def test_binding_refuses_short_buffers(lib):
    """Buffer sizes are checked against the plan (or the call's sizes) before
    any pointer reaches the library."""
    import torch
    f32 = lambda n: torch.zeros(n, dtype=torch.float32)  # noqa: E731
    i32 = lambda n: torch.zeros(n, dtype=torch.int32)  # noqa: E731
    plan = spmm.Plan(0, i32(5), M=4, nnz=6, N=8)  # M=4, nnz=6, N=8; K=3 below
    cases = [
        (lambda: spmm.spmm_csr_f32_exec(plan, 3, i32(5), f32(6), f32(24), f32(32)), "colind"),
        (lambda: spmm.spmm_csr_f32_exec(plan, 3, i32(6), f32(5), f32(24), f32(32)), "vals"),
        (lambda: spmm.spmm_csr_f32_exec(plan, 3, i32(6), f32(6), f32(23), f32(32)), "B"),
        (lambda: spmm.spmm_csr_bf16f32_exec(plan, 3, i32(6), f32(6), torch.zeros(24, dtype=torch.int16), f32(31)),
         "C"),
        (lambda: spmm.spmm_csr_semiring_f32_exec(plan, 3, i32(6), f32(6), f32(24), f32(31), "min", "add"), "C"),
        (lambda: spmm.spmm_csr_sddmm_f32(plan, 3, i32(6), f32(32), f32(24), f32(5)), "out"),
        (lambda: spmm.spmm_csr_fusedmm_f32(plan, 3, i32(6), f32(32), f32(24), f32(23), f32(32)), "D"),
        (lambda: spmm.spmm_csr_fusedmm_f32(plan, 3, i32(6), f32(32), f32(24), f32(24), f32(31)), "E"),
        (lambda: spmm.spmm_csr_plan(i32(4), 4, 0, 8), "rowptr"),
        (lambda: spmm.spmm_csr_f32(4, 3, 8, i32(5), i32(6), f32(6), f32(24), f32(31)), "C"),
        (lambda: spmm.spmm_csr_f32_noalloc(4, 3, 8, 6, i32(5), i32(6), f32(5), f32(24), f32(32)), "vals"),
    ]
    for call, name in cases:
        with pytest.raises(ValueError, match=f"^{name} holds"):
            call()
    # sizes that fit: refused only because the tensors are not on a GPU
    with pytest.raises(ValueError, match="CUDA"):
        spmm.spmm_csr_f32_exec(plan, 3, i32(6), f32(6), f32(24), f32(32))


C_USER = r"""
#include <stdio.h>
#include <stddef.h>
#include "spmm.h"

/* A C99 user of the library: argument errors come back as status codes
   before any CUDA call, so this runs on a machine without a GPU. */
int main(void) {
  spmm_plan_t plan = (spmm_plan_t)0;
  int bad = 0;
  if (spmm_csr_plan(NULL, 10, 5, 4, NULL, &plan) != SPMM_ERR_INVALID_ARG) bad |= 1;
  if (plan != NULL) bad |= 2;
  if (spmm_csr_plan_ex(NULL, 0, 0, 4, 99, 0, NULL, &plan) != SPMM_ERR_INVALID_ARG) bad |= 4;
  if (spmm_csr_f32(-1, 1, 1, NULL, NULL, NULL, NULL, NULL, NULL) != SPMM_ERR_INVALID_ARG) bad |= 8;
  if (spmm_csr_f32_exec(NULL, 1, NULL, NULL, NULL, NULL, NULL) != SPMM_ERR_PLAN_MISMATCH) bad |= 16;
  if (spmm_plan_set_column_tile(NULL, 8) != SPMM_ERR_PLAN_MISMATCH) bad |= 32;
  printf("%s %d\n", spmm_status_string(SPMM_ERR_INVALID_CSR), bad);
  return bad;
}
"""


def test_header_states_the_size_limit():
    m = re.search(r"#define SPMM_MAX_EXTENT (\d+)", open(HEADER).read())
    assert m and int(m.group(1)) == (1 << 31) - 65536


def test_header_is_c99_and_a_c_program_links(lib, tmp_path):
    """include/spmm.h compiles as strict C99 and a C program links the library."""
    import subprocess
    src = tmp_path / "user.c"
    src.write_text(C_USER)
    exe = tmp_path / "user"
    libpath = spmm.library_path()
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic", "-I", os.path.dirname(HEADER),
                    str(src), "-o", str(exe), libpath, f"-Wl,-rpath,{os.path.dirname(libpath)}"], check=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True)
    assert out.returncode == 0 and out.stdout.split() == ["SPMM_ERR_INVALID_CSR", "0"], (out.returncode, out.stdout)
