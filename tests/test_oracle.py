"""The CPU oracle against its pins (no GPU)."""
import numpy as np
import pytest

import oracle
from tests import oracle_pins as pins


@pytest.mark.parametrize("pin", pins.ALL_PINS, ids=lambda f: f.__name__)
def test_oracle_pin(pin):
    pin(pins.oracle_callable())


def test_oracle_rejects_bad_csr():
    rowptr = np.array([0, 2, 1], dtype=np.int32)  # decreasing
    with pytest.raises(ValueError):
        oracle.spmm_reference(rowptr, np.array([0, 1], np.int32), np.ones(2, np.float32),
                              np.ones((2, 3), np.float32))
    rowptr = np.array([0, 1], dtype=np.int32)
    with pytest.raises(ValueError):  # column index outside [0, K)
        oracle.spmm_reference(rowptr, np.array([5], np.int32), np.ones(1, np.float32),
                              np.ones((2, 3), np.float32))


def test_oracle_empty_and_degenerate():
    # M = 0
    C, S = oracle.spmm_reference(np.zeros(1, np.int32), np.zeros(0, np.int32),
                                 np.zeros(0, np.float32), np.ones((4, 3), np.float32))
    assert C.shape == (0, 3)
    # nnz = 0: all-zero output
    C, S = oracle.spmm_reference(np.zeros(6, np.int32), np.zeros(0, np.int32),
                                 np.zeros(0, np.float32), np.ones((4, 3), np.float32))
    assert C.shape == (5, 3) and not C.any() and not S.any()
    # N = 0
    C, S = oracle.spmm_reference(np.array([0, 1], np.int32), np.array([0], np.int32),
                                 np.ones(1, np.float32), np.ones((1, 0), np.float32))
    assert C.shape == (1, 0)
