"""Seeded synthetic CSR inputs for SpMM, C[M x N] = A[M x K, CSR] . B[K x N].

This module only *makes inputs*: sparsity structures, values and dense B
matrices, drawn from numpy's PCG64 generator (``numpy.random.default_rng``).
It performs none of the multiplication's arithmetic, so both the CUDA path
and the CPU oracle can take their inputs from here without sharing any
computation.

Workloads (the five benchmark matrices of this library):

* ``uniform1k``  -- M=K=1024, exactly 16 distinct random columns per row
  (sorted), vals U[-1,1], B 1024x32 fp32 U[-1,1], seed 0.
* ``uniform64k`` -- M=K=65536, 32 distinct random columns per row, vals
  U[-1,1], B 65536x64 fp32 U[-1,1], seed 1.
* ``rmat20``     -- R-MAT scale 20 (M=K=2^20), edge factor 16,
  (a,b,c,d)=(.57,.19,.19,.05), self-loops removed, duplicates removed, one
  random vertex permutation applied to rows and columns; vals U[0,1];
  B 2^20 x 128 fp32 U[-1,1]; seed 2.
* ``banded``     -- M=K=262144, row i holds columns max(0,i-32)..min(K-1,i+31);
  vals N(0,1); B 262144x256 drawn N(0,1) then rounded to bf16; seed 3.
* ``rmat22``     -- R-MAT scale 22, same recipe as ``rmat20``; vals U[-1,1];
  B 2^22 x 32 fp32 U[-1,1]; seed 4.

Draw order for every workload: structure first, then vals in CSR order,
then B in row-major order.  Values are drawn in float64 and rounded to fp32
with round-to-nearest-even; bf16 B is rounded (nearest-even) from those fp32
values.  bf16 arrays are carried as their raw uint16 bit patterns.

The matrices stand in for the matrix collections the source papers measure
on (uniform and banded for regular short-row matrices, R-MAT for graph-like
power-law ones); no item of those collections is reproduced.
"""
from __future__ import annotations

import dataclasses
import hashlib

import numpy as np

# R-MAT quadrant probabilities (a, b, c, d); d = 1 - a - b - c.
RMAT_ABCD = (0.57, 0.19, 0.19, 0.05)

WORKLOADS = {
    "uniform1k": dict(kind="uniform", M=1024, per_row=16, N=32, b="f32", seed=0, vals="pm1"),
    "uniform64k": dict(kind="uniform", M=65536, per_row=32, N=64, b="f32", seed=1, vals="pm1"),
    "rmat20": dict(kind="rmat", scale=20, edge_factor=16, N=128, b="f32", seed=2, vals="01"),
    "banded": dict(kind="banded", M=262144, below=32, above=31, N=256, b="bf16", seed=3, vals="normal"),
    "rmat22": dict(kind="rmat", scale=22, edge_factor=16, N=32, b="f32", seed=4, vals="pm1"),
}

# The order in which the workloads are listed by the benchmark definition.
WORKLOAD_ORDER = ["uniform1k", "uniform64k", "rmat20", "banded", "rmat22"]

_CHUNK = 1 << 22  # elements per value-draw chunk (keeps float64 temporaries small)


@dataclasses.dataclass
class CsrProblem:
    """One SpMM input: A in CSR (int32 rowptr/colind, fp32 vals) and dense B."""

    name: str
    M: int
    K: int
    N: int
    rowptr: np.ndarray  # int32 [M+1]
    colind: np.ndarray  # int32 [nnz]
    vals: np.ndarray  # float32 [nnz]
    B: np.ndarray  # float32 [K, N] or uint16 (bf16 bit patterns) [K, N]
    b_dtype: str  # "f32" or "bf16"
    seed: int | None = None

    @property
    def nnz(self) -> int:
        return int(self.rowptr[-1])

    def compulsory_bytes(self) -> int:
        """rowptr + colind + vals + B read once + C written once."""
        bsz = 4 if self.b_dtype == "f32" else 2
        return 4 * (self.M + 1) + 8 * self.nnz + self.K * self.N * bsz + 4 * self.M * self.N

    def flops(self) -> int:
        return 2 * self.nnz * self.N

    def digest(self) -> dict:
        """SHA-256 of every array (reproducibility record)."""
        out = {}
        for key in ("rowptr", "colind", "vals", "B"):
            arr = np.ascontiguousarray(getattr(self, key))
            out[key] = hashlib.sha256(arr.tobytes()).hexdigest()
        return out


# ----------------------------------------------------------------------------
# value draws
# ----------------------------------------------------------------------------
def _draw_f32(rng: np.random.Generator, n: int, dist: str) -> np.ndarray:
    """Draw n values in float64 (chunked, same stream as one call) -> fp32."""
    out = np.empty(n, dtype=np.float32)
    for s in range(0, n, _CHUNK):
        e = min(n, s + _CHUNK)
        if dist == "pm1":
            out[s:e] = rng.uniform(-1.0, 1.0, e - s)
        elif dist == "01":
            out[s:e] = rng.uniform(0.0, 1.0, e - s)
        elif dist == "normal":
            out[s:e] = rng.standard_normal(e - s)
        else:
            raise ValueError(f"unknown value distribution {dist!r}")
    return out


def dense_f32(rng: np.random.Generator, rows: int, cols: int, dist: str = "pm1") -> np.ndarray:
    """A seeded row-major fp32 matrix (the dense operands of SDDMM / FusedMM)."""
    return _draw_f32(rng, rows * cols, dist).reshape(rows, cols)


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 values to bf16 (nearest, ties to even); return uint16 bits.

    Input preparation only (the benchmark's bf16 B is defined as the
    nearest-even bf16 of an fp32 draw).  Finite inputs only: for them the
    32-bit sum below cannot wrap (largest pattern 0xFF7FFFFF + 0x8000).
    """
    flat = np.ascontiguousarray(x, dtype=np.float32).reshape(-1)
    out = np.empty(flat.shape, dtype=np.uint16)
    for s in range(0, flat.size, _CHUNK):
        bits = flat[s:s + _CHUNK].view(np.uint32).copy()
        lsb = (bits >> 16) & 1
        bits += 0x7FFF
        bits += lsb
        bits >>= 16
        out[s:s + _CHUNK] = bits
    return out.reshape(np.shape(x))


def _dense_b(rng, K, N, dist, b_dtype):
    vals = _draw_f32(rng, K * N, dist).reshape(K, N)
    if b_dtype == "f32":
        return vals
    if b_dtype == "bf16":
        return f32_to_bf16_bits(vals)
    raise ValueError(b_dtype)


# ----------------------------------------------------------------------------
# structures
# ----------------------------------------------------------------------------
def rowptr_from_counts(counts: np.ndarray) -> np.ndarray:
    rowptr = np.zeros(len(counts) + 1, dtype=np.int64)
    np.cumsum(counts, out=rowptr[1:])
    if rowptr[-1] > np.iinfo(np.int32).max:
        raise ValueError("nnz exceeds int32")
    return rowptr.astype(np.int32)


def uniform_structure(rng, M, K, per_row):
    """Each row: `per_row` distinct columns sampled without replacement, sorted."""
    colind = np.empty(M * per_row, dtype=np.int32)
    for i in range(M):
        cols = rng.choice(K, size=per_row, replace=False)
        cols.sort()
        colind[i * per_row:(i + 1) * per_row] = cols
    rowptr = (np.arange(M + 1, dtype=np.int64) * per_row).astype(np.int32)
    return rowptr, colind


def banded_structure(M, K, below, above):
    """Row i holds columns max(0, i-below) .. min(K-1, i+above), in order."""
    width = below + above + 1
    cols = np.arange(M, dtype=np.int64)[:, None] - below + np.arange(width, dtype=np.int64)[None, :]
    inside = (cols >= 0) & (cols < K)
    rowptr = rowptr_from_counts(inside.sum(axis=1))
    colind = cols[inside].astype(np.int32)  # row-major order keeps rows in order
    return rowptr, colind


def _rmat_chunk(state, scale, E, e0, e1, thresholds):
    """Edges [e0, e1): level L of edge e uses double number L*E + e of the stream."""
    t1, t2, t3 = thresholds
    n = e1 - e0
    src = np.zeros(n, dtype=np.int32)
    dst = np.zeros(n, dtype=np.int32)
    u = np.empty(n, dtype=np.float64)
    for level in range(scale):
        bg = np.random.PCG64()
        bg.state = state
        bg.advance(level * E + e0)
        np.random.Generator(bg).random(out=u)
        row_bit = u >= t2  # quadrants c, d
        col_bit = u >= t3  # quadrant d
        col_bit |= (u >= t1) & (u < t2)  # quadrant b
        src <<= 1
        src |= row_bit
        dst <<= 1
        dst |= col_bit
    return src, dst


def rmat_edges(rng, scale, edge_factor, abcd=RMAT_ABCD, threads=8):
    """Raw R-MAT edge list (src, dst) as int64, before any clean-up.

    Each edge descends `scale` levels, most significant bit first; at each
    level u ~ U[0,1) picks quadrant a (u < a), b (sets the column bit),
    c (sets the row bit) or d (sets both).  The draws are consumed level by
    level (all E edges of level 0, then level 1, ...); chunks of edges are
    generated independently by jumping the PCG64 stream, which gives the same
    numbers as one sequential pass.
    """
    import concurrent.futures as cf

    if not isinstance(rng.bit_generator, np.random.PCG64):
        raise TypeError("R-MAT generation expects a PCG64 generator")
    a, b, c, _ = abcd
    E = edge_factor * (1 << scale)
    state = rng.bit_generator.state
    chunk = 1 << 20
    bounds = [(e0, min(E, e0 + chunk)) for e0 in range(0, E, chunk)]
    src = np.empty(E, dtype=np.int64)
    dst = np.empty(E, dtype=np.int64)
    with cf.ThreadPoolExecutor(max_workers=threads) as ex:
        futs = {ex.submit(_rmat_chunk, state, scale, E, e0, e1, (a, a + b, a + b + c)): (e0, e1)
                for e0, e1 in bounds}
        for f in cf.as_completed(futs):
            e0, e1 = futs[f]
            s, d = f.result()
            src[e0:e1] = s
            dst[e0:e1] = d
    rng.bit_generator.advance(scale * E)
    return src, dst


def _sorted_unique(keys: np.ndarray) -> np.ndarray:
    keys = np.sort(keys)
    if keys.size == 0:
        return keys
    first = np.empty(keys.size, dtype=bool)
    first[0] = True
    np.not_equal(keys[1:], keys[:-1], out=first[1:])
    return keys[first]


def rmat_structure(rng, scale, edge_factor, remove_self_loops=True, permute=True):
    n = 1 << scale
    src, dst = rmat_edges(rng, scale, edge_factor)
    if remove_self_loops:
        keep = src != dst
        src, dst = src[keep], dst[keep]
    keys = _sorted_unique((src << np.int64(scale)) | dst)  # dedup
    src = keys >> np.int64(scale)
    dst = keys & np.int64(n - 1)
    if permute:
        perm = rng.permutation(n).astype(np.int64)
        src, dst = perm[src], perm[dst]
        keys = np.sort((src << np.int64(scale)) | dst)
        src = keys >> np.int64(scale)
        dst = keys & np.int64(n - 1)
    counts = np.bincount(src, minlength=n)
    rowptr = rowptr_from_counts(counts)
    return rowptr, dst.astype(np.int32)


# ----------------------------------------------------------------------------
# workloads
# ----------------------------------------------------------------------------
def make_workload(name: str) -> CsrProblem:
    """Build one of the five benchmark workloads (deterministic in its seed)."""
    spec = WORKLOADS[name]
    rng = np.random.default_rng(spec["seed"])
    kind = spec["kind"]
    if kind == "uniform":
        M = K = spec["M"]
        rowptr, colind = uniform_structure(rng, M, K, spec["per_row"])
    elif kind == "banded":
        M = K = spec["M"]
        rowptr, colind = banded_structure(M, K, spec["below"], spec["above"])
    elif kind == "rmat":
        M = K = 1 << spec["scale"]
        rowptr, colind = rmat_structure(rng, spec["scale"], spec["edge_factor"])
    else:
        raise ValueError(kind)
    vals = _draw_f32(rng, int(rowptr[-1]), spec["vals"])
    B = _dense_b(rng, K, spec["N"], "normal" if spec["vals"] == "normal" else "pm1", spec["b"])
    return CsrProblem(name, M, K, spec["N"], rowptr, colind, vals, B, spec["b"], spec["seed"])


# ----------------------------------------------------------------------------
# small and special inputs for parity tests
# ----------------------------------------------------------------------------
def random_csr(rng, M, K, N, *, mean_row=8.0, max_row=None, empty_frac=0.2,
               long_rows=(), duplicates=False, sort_cols=True, b_dtype="f32",
               vals="pm1", integer=False):
    """Random CSR with a mix of row lengths.

    Row lengths are geometric around `mean_row` (capped by `max_row` or K),
    a fraction `empty_frac` of rows is empty, and each (row, length) pair in
    `long_rows` forces that row's length.  With `duplicates` columns are drawn
    with replacement (repeated (i, j) entries), otherwise distinct.  With
    `integer` the values are small integers (vals in -2..2, B in -3..3) so
    that every partial sum is exactly representable in fp32.
    """
    cap = K if max_row is None else min(K, max_row)
    p = 1.0 / max(1.0, mean_row)
    lens = np.minimum(rng.geometric(p, size=M), cap)
    lens[rng.random(M) < empty_frac] = 0
    for r, L in long_rows:
        lens[r] = L if duplicates else min(L, K)
    rowptr = rowptr_from_counts(lens)
    colind = np.empty(int(rowptr[-1]), dtype=np.int32)
    for i in range(M):
        L = int(lens[i])
        if L == 0:
            continue
        if duplicates:
            cols = rng.integers(0, K, size=L)
        else:
            cols = rng.choice(K, size=L, replace=False)
        if sort_cols:
            cols = np.sort(cols)
        colind[rowptr[i]:rowptr[i + 1]] = cols
    nnz = int(rowptr[-1])
    if integer:
        v = rng.integers(-2, 3, size=nnz).astype(np.float32)
        Bf = rng.integers(-3, 4, size=(K, N)).astype(np.float32)
    else:
        v = _draw_f32(rng, nnz, vals)
        Bf = _draw_f32(rng, K * N, "pm1").reshape(K, N)
    B = Bf if b_dtype == "f32" else f32_to_bf16_bits(Bf)
    return CsrProblem("random", M, K, N, rowptr, colind, v, B, b_dtype)


def identity_csr(n, scale=1.0):
    rowptr = np.arange(n + 1, dtype=np.int32)
    colind = np.arange(n, dtype=np.int32)
    vals = np.full(n, scale, dtype=np.float32)
    return rowptr, colind, vals


def permutation_csr(perm):
    """Row i holds a single 1 at column perm[i]."""
    n = len(perm)
    rowptr = np.arange(n + 1, dtype=np.int32)
    return rowptr, np.asarray(perm, dtype=np.int32), np.ones(n, dtype=np.float32)


def uniform_b(rng, K, N, b_dtype="f32"):
    Bf = _draw_f32(rng, K * N, "pm1").reshape(K, N)
    return Bf if b_dtype == "f32" else f32_to_bf16_bits(Bf)


def row_stats(rowptr: np.ndarray) -> dict:
    lens = np.diff(rowptr.astype(np.int64))
    return dict(M=len(lens), nnz=int(rowptr[-1]), max=int(lens.max(initial=0)),
                mean=float(lens.mean()) if len(lens) else 0.0,
                empty=int((lens == 0).sum()))
