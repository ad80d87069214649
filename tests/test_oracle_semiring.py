"""The semiring SpMM oracle against its pins (no GPU), and planted mistakes."""
import os
import subprocess

import pytest

import oracle
from tests import oracle_pins_semiring as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "spmm_oracle.c")


@pytest.mark.parametrize("pin", pins.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    pin(pins.callables())


MUTANTS = {
    "min_identity_zero": ("add_op == 1 ? INFINITY : -INFINITY", "add_op == 1 ? 0.0 : -INFINITY"),
    "min_max_swapped": ("if (t < c[n]) c[n] = t;", "if (t > c[n]) c[n] = t;"),
    "mul_ops_swapped": ("const double t = mul_op == 0 ? a * b : a + b;", "const double t = mul_op == 0 ? a + b : a * b;"),
    "skips_last_entry": ("    for (int64_t p = rowptr[i]; p < rowptr[i + 1]; ++p) {\n      const double a = (double)vals[p];\n      const int64_t j = colind[p];\n      if (j < 0 || j >= K) return -2;\n      for (int32_t n = 0; n < N; ++n) {\n        const double b",
                         "    for (int64_t p = rowptr[i]; p + 1 < rowptr[i + 1]; ++p) {\n      const double a = (double)vals[p];\n      const int64_t j = colind[p];\n      if (j < 0 || j >= K) return -2;\n      for (int32_t n = 0; n < N; ++n) {\n        const double b"),
    "bound_without_abs": ("          if (s) s[n] += fabs(t);", "          if (s) s[n] += t;"),
    "b_row_from_row_index": ("        const double b = (double)B[j * N + n];", "        const double b = (double)B[(i % K) * N + n];"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor for {name} must be unique"
    mutated = tmp_path / "mutant.c"
    mutated.write_text(src.replace(old, new))
    lib = tmp_path / "libmutant.so"
    subprocess.run(["gcc", "-O2", "-std=c99", "-ffp-contract=off", "-fPIC", "-shared", "-o", str(lib),
                    str(mutated), "-lm"], check=True)
    assert pins.failing_pins(oracle.load_library(str(lib))), f"no pin catches {name!r}"
