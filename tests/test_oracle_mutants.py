"""Plant plausible mistakes in copies of the C oracle and check the pins catch each.

Every mutant is a textual edit of oracle/spmm_oracle.c compiled on the CPU into
a temporary directory; the real oracle is untouched.  A mutant that no pin
catches would mean the pins leave that part of the oracle unchecked.
"""
import os
import subprocess

import pytest

import oracle
from tests import oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "spmm_oracle.c")

MUTANTS = {
    "drop_last_term": ("p < rowptr[i + 1]; ++p", "p + 1 < rowptr[i + 1]; ++p"),
    "drop_first_term": ("int64_t p = rowptr[i];", "int64_t p = rowptr[i] + 1;"),
    "wrong_sign": ("c[n] += prod;", "c[n] -= prod;"),
    "transposed_B": ("row_of_b * N + n", "n * (int64_t)K + row_of_b"),
    "vals_local_index": ("double a = (double)vals[p];", "double a = (double)vals[p - rowptr[i]];"),
    "colind_local_index": ("int64_t row_of_b = colind[p];", "int64_t row_of_b = colind[p - rowptr[i]];"),
    "no_row_reset": ("      c[n] = 0.0;\n", "      c[n] = t > 0 ? C_out[(t - 1) * (int64_t)N + n] : 0.0;\n"),
    "float_accumulator": ("c[n] += prod;", "c[n] = (float)(c[n] + prod);"),
    "bf16_wrong_shift": ("((uint32_t)bits) << 16", "((uint32_t)bits) << 8"),
    "bound_without_abs": ("s[n] += fabs(prod);", "s[n] += prod;"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) >= 1, f"mutation anchor for {name} not found"
    mutated = tmp_path / "mutant.c"
    mutated.write_text(src.replace(old, new))
    lib = tmp_path / "libmutant.so"
    subprocess.run(["gcc", "-O2", "-std=c99", "-ffp-contract=off", "-fPIC", "-shared", "-o", str(lib),
                    str(mutated), "-lm"], check=True)
    failed = pins.failing_pins(pins.oracle_callable(oracle.load_library(str(lib))))
    assert failed, f"no pin catches the planted mistake {name!r}"
