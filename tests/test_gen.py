"""Seeded input generators: structure, reproducibility, recipes (no GPU)."""
import numpy as np
import pytest
import torch

from csr_spmm_02_gb300 import gen


def _check_csr(p, distinct_sorted=True):
    assert p.rowptr.dtype == np.int32 and p.colind.dtype == np.int32 and p.vals.dtype == np.float32
    assert p.rowptr[0] == 0 and np.all(np.diff(p.rowptr) >= 0) and p.rowptr[-1] == len(p.colind)
    assert p.colind.min(initial=0) >= 0 and p.colind.max(initial=0) < p.K
    if distinct_sorted:
        d = np.diff(p.colind.astype(np.int64))
        starts = p.rowptr[1:-1]
        inside = np.ones(len(d), dtype=bool)
        inside[starts[(starts > 0) & (starts <= len(d))] - 1] = False
        assert np.all(d[inside] > 0), "columns inside a row must be strictly increasing"
    assert p.B.shape == (p.K, p.N)


@pytest.mark.parametrize("name,nnz,cbytes", [("uniform1k", 16384, 397316), ("uniform64k", 2097152, 50593796)])
def test_uniform_workloads(name, nnz, cbytes):
    p = gen.make_workload(name)
    _check_csr(p)
    assert p.nnz == nnz and p.compulsory_bytes() == cbytes
    assert np.all(np.diff(p.rowptr) == gen.WORKLOADS[name]["per_row"])
    assert p.vals.min() >= -1 and p.vals.max() <= 1 and p.B.dtype == np.float32
    assert p.digest() == gen.make_workload(name).digest(), "same seed, same arrays"


def test_banded_workload():
    """The banded structure (row i: columns i-32 .. i+31, clipped) on a smaller matrix with the
    same band, and the full-size nnz / compulsory bytes in closed form: every row holds 64
    columns except the 32 first and 31 last rows, clipped by 32-i and i-(K-32) columns."""
    spec = gen.WORKLOADS["banded"]
    M, below, above, N = spec["M"], spec["below"], spec["above"], spec["N"]
    clipped = sum(below - i for i in range(below)) + sum(above - i for i in range(above))
    nnz_full = M * (below + above + 1) - clipped
    assert nnz_full == 16776192
    assert 4 * (M + 1) + 8 * nnz_full + M * N * 2 + 4 * M * N == 537911300  # compulsory bytes, bf16 B
    m = 5000
    rowptr, colind = gen.banded_structure(m, m, below, above)
    assert int(rowptr[-1]) == m * (below + above + 1) - clipped and len(colind) == int(rowptr[-1])
    for i in (0, 1, 31, 32, 2500, m - 32, m - 1):
        cols = colind[rowptr[i]:rowptr[i + 1]]
        assert np.array_equal(cols, np.arange(max(0, i - below), min(m - 1, i + above) + 1))
    small = gen.random_csr(np.random.default_rng(0), 40, 30, 16, b_dtype="bf16")
    assert small.B.dtype == np.uint16 and small.B.shape == (30, 16)


def test_bf16_rounding_matches_torch():
    x = np.random.default_rng(0).standard_normal(100000).astype(np.float32)
    x[:4] = [1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -(1.0 + 2 ** -8), 0.0]  # ties to even
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(gen.f32_to_bf16_bits(x), ref)


def _rmat_sequential(rng, scale, edge_factor):
    """One plain pass over the stream, level by level (the recipe as stated)."""
    a, b, c, _ = gen.RMAT_ABCD
    E = edge_factor << scale
    src = np.zeros(E, np.int64)
    dst = np.zeros(E, np.int64)
    for level in range(scale):
        u = rng.random(E)
        bit = 1 << (scale - 1 - level)
        src[u >= a + b] |= bit
        dst[((u >= a) & (u < a + b)) | (u >= a + b + c)] |= bit
    return src, dst


@pytest.mark.parametrize("scale", [6, 13])
def test_rmat_jump_ahead_equals_sequential(scale):
    s1, d1 = gen.rmat_edges(np.random.default_rng(3), scale, 16)
    r = np.random.default_rng(3)
    s2, d2 = _rmat_sequential(r, scale, 16)
    assert np.array_equal(s1, s2) and np.array_equal(d1, d2)
    r1 = np.random.default_rng(3)
    gen.rmat_edges(r1, scale, 16)
    assert np.array_equal(r1.random(4), r.random(4)), "stream position after the edges"


def test_rmat_structure_recipe():
    scale = 14
    src, dst = gen.rmat_edges(np.random.default_rng(1), scale, 16)
    n = 1 << scale
    # quadrant probabilities: a row bit is set with c + d = 0.24, a column bit with b + d = 0.24
    bits = np.array([(src >> k) & 1 for k in range(scale)]).mean()
    cbits = np.array([(dst >> k) & 1 for k in range(scale)]).mean()
    assert abs(bits - 0.24) < 0.003 and abs(cbits - 0.24) < 0.003
    rowptr, colind = gen.rmat_structure(np.random.default_rng(1), scale, 16)
    rows = np.repeat(np.arange(n), np.diff(rowptr))
    assert not np.any(rows == colind), "self-loops removed"
    keys = rows.astype(np.int64) * n + colind
    assert np.all(np.diff(keys) > 0), "sorted and duplicate-free"
    assert len(keys) < 16 * n


def test_random_csr_options():
    rng = np.random.default_rng(0)
    p = gen.random_csr(rng, 50, 20, 7, mean_row=4, long_rows=[(3, 20)], duplicates=False)
    _check_csr(p)
    assert p.rowptr[4] - p.rowptr[3] == 20
    p = gen.random_csr(rng, 50, 20, 7, duplicates=True, sort_cols=False, integer=True, b_dtype="bf16")
    _check_csr(p, distinct_sorted=False)
    assert p.B.dtype == np.uint16


@pytest.mark.parametrize("name,prefixes", [
    ("uniform1k", ("4f124b61969c4f0f", "a59d395f092f2e5a", "2ca73052517df28f", "e9bad8adf6e3237f")),
    ("uniform64k", ("f8675858ad786334", "c9b7206181dbc2ac", "67d8484d3eee11a5", "9436afcbe8c5a585")),
])
def test_workload_digests_are_stable(name, prefixes):
    """The generator reproduces the arrays recorded with the measurements (rowptr, colind, vals, B)."""
    d = gen.make_workload(name).digest()
    assert tuple(d[k][:16] for k in ("rowptr", "colind", "vals", "B")) == prefixes
