"""The SDDMM and FusedMM oracles against their pins (no GPU)."""
import os
import subprocess

import pytest

import oracle
from tests import oracle_pins_sddmm as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "spmm_oracle.c")


@pytest.mark.parametrize("pin", pins.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    pin(*pins.callables())


MUTANTS = {
    "sddmm_drops_last_term": ("for (int32_t n = 0; n < N; ++n) {\n        const double prod = (double)C[(int64_t)i * N + n] * (double)B[j * N + n];",
                              "for (int32_t n = 0; n + 1 < N; ++n) {\n        const double prod = (double)C[(int64_t)i * N + n] * (double)B[j * N + n];"),
    "sddmm_row_of_C_from_colind": ("const double prod = (double)C[(int64_t)i * N + n] * (double)B[j * N + n];\n        dot += prod;",
                                   "const double prod = (double)C[(j % M) * N + n] * (double)B[j * N + n];\n        dot += prod;"),
    "fusedmm_uses_B_for_D": ("const double prod = a * (double)D[j * N + n];", "const double prod = a * (double)B[j * N + n];"),
    "fusedmm_unsigned_values": ("      if (A_out) A_out[p] = a;", "      a = fabs(a);\n      if (A_out) A_out[p] = a;"),
    "fusedmm_no_row_reset": ("      e[n] = 0.0;\n      if (s) s[n] = 0.0;\n    }\n    if (rowptr[i + 1] < rowptr[i]) return -2;\n    for (int64_t p = rowptr[i]; p < rowptr[i + 1]; ++p) {\n      const int64_t j = colind[p];\n      if (j < 0 || j >= K) return -2;\n      double a",
                             "      e[n] = i > 0 ? e[n - N] : 0.0;\n      if (s) s[n] = 0.0;\n    }\n    if (rowptr[i + 1] < rowptr[i]) return -2;\n    for (int64_t p = rowptr[i]; p < rowptr[i + 1]; ++p) {\n      const int64_t j = colind[p];\n      if (j < 0 || j >= K) return -2;\n      double a"),
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
