/*
 * CPU oracle for CSR SpMM -- TEST INFRASTRUCTURE, not part of the product.
 *
 * Only the tests, the smoke check and the benchmark's CPU-baseline leg may
 * load this file's library.  It shares no code, header or table with the
 * CUDA library: it is a plain single-threaded C restatement of the
 * operation's definition, accumulating in double precision.
 *
 * Definition followed (SpMM, page "Performance Optimization of Deep Learning
 * Sparse Matrix Kernels on Intel Max Series GPU", SPMM section, Fig. 5 and
 * Algorithm 2): row C_i of the dense output is produced by walking the
 * nonzeros of sparse row A_i; for the nonzero with value s at column k the
 * scaled dense row s * B_k is added to C_i (a SAXPY).  C_i starts at zero
 * and is written once.  In index form
 *
 *     C[i][n] = sum_{p = rowptr[i]}^{rowptr[i+1]-1} vals[p] * B[colind[p]][n].
 *
 * The Sgap page ("Sgap: Towards Efficient Sparse Tensor Algebra Compilation
 * for GPU", sparse-dense hybrid algebra section) states the same reduction:
 * SpMM reduces over the sparse dimension j.  The kkmem page ("Sparse
 * Matrix-Matrix Multiplication on Multilevel Memory Architectures", access
 * pattern observations) describes the same row-by-row order: A streamed,
 * each C row written once, B row j read once per nonzero in column j.
 *
 * Beside C the oracle returns S[i][n] = sum_p |vals[p] * B[colind[p]][n]|,
 * the magnitude sum that scales the acceptance bound of a floating-point
 * result (|C_gpu - C| <= rel * S + abs).
 *
 * Readings where the pages are silent: duplicate (i, j) entries are summed;
 * column order inside a row is free; an empty row gives an exact zero row;
 * C is overwritten, never accumulated into.  bf16 B values are decoded from
 * their bit patterns as the upper half of an IEEE-754 binary32 (exact).
 *
 * Every floating-point step is a double-precision multiply and add, with
 * contraction disabled at build time (-ffp-contract=off), so results are the
 * same on every host.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* bfloat16 is the top 16 bits of a binary32; decoding is a bit move. */
static double oracle_bf16_to_double(uint16_t bits) {
  uint32_t w = ((uint32_t)bits) << 16;
  float f;
  memcpy(&f, &w, sizeof f);
  return (double)f;
}

static double oracle_b_value(const void* B, int32_t b_is_bf16, int64_t idx) {
  if (b_is_bf16) return oracle_bf16_to_double(((const uint16_t*)B)[idx]);
  return (double)((const float*)B)[idx];
}

/*
 * C_out[t][n], S_out[t][n] for the rows listed in rows[0..nrows) (all rows
 * 0..M-1 in order when rows == NULL, nrows then ignored).  B has K rows of N
 * values.  S_out may be NULL.  Returns 0; -1 on an argument error (bad
 * sizes, a listed row outside [0, M)); -2 when a visited row's rowptr range
 * is decreasing or a visited column index lies outside [0, K).
 */
int spmm_oracle_rows_f64(int32_t M, int32_t K, int32_t N, const int32_t* rowptr,
                         const int32_t* colind, const float* vals, const void* B,
                         int32_t b_is_bf16, const int32_t* rows, int64_t nrows, double* C_out,
                         double* S_out) {
  if (M < 0 || K < 0 || N < 0 || !rowptr || !C_out) return -1;
  if (rows == NULL) nrows = M;
  for (int64_t t = 0; t < nrows; ++t) {
    int32_t i = rows ? rows[t] : (int32_t)t;
    if (i < 0 || i >= M) return -1;
    double* c = C_out + t * (int64_t)N;
    double* s = S_out ? S_out + t * (int64_t)N : NULL;
    for (int32_t n = 0; n < N; ++n) {
      c[n] = 0.0;
      if (s) s[n] = 0.0;
    }
    if (rowptr[i + 1] < rowptr[i]) return -2;
    for (int64_t p = rowptr[i]; p < rowptr[i + 1]; ++p) {
      double a = (double)vals[p];
      int64_t row_of_b = colind[p];
      if (row_of_b < 0 || row_of_b >= K) return -2;
      for (int32_t n = 0; n < N; ++n) {
        double prod = a * oracle_b_value(B, b_is_bf16, row_of_b * N + n);
        c[n] += prod;
        if (s) s[n] += fabs(prod);
      }
    }
  }
  return 0;
}

/*
 * SDDMM (page "Performance Optimization of Deep Learning Sparse Matrix
 * Kernels on Intel Max Series GPU", SDDMM section, Algorithm 1, Figs. 3-4):
 * the dense product C . B^T is computed only where A has a stored entry; the
 * entry (i, j) receives the dot product of row i of C (M x N) and row j of B
 * (K x N).  A's stored values are not used (the page stores the products into
 * A).  out[p] for every stored position p; S_out[p] = sum_n |C[i][n] B[j][n]|.
 * Returns 0, -1 on a size error, -2 on malformed CSR (as above).
 */
int sddmm_oracle_f64(int32_t M, int32_t K, int32_t N, const int32_t* rowptr, const int32_t* colind,
                     const float* C, const float* B, double* out, double* S_out) {
  if (M < 0 || K < 0 || N < 0 || !rowptr || !out) return -1;
  for (int32_t i = 0; i < M; ++i) {
    if (rowptr[i + 1] < rowptr[i]) return -2;
    for (int64_t p = rowptr[i]; p < rowptr[i + 1]; ++p) {
      const int64_t j = colind[p];
      if (j < 0 || j >= K) return -2;
      double dot = 0.0, mag = 0.0;
      for (int32_t n = 0; n < N; ++n) {
        const double prod = (double)C[(int64_t)i * N + n] * (double)B[j * N + n];
        dot += prod;
        mag += fabs(prod);
      }
      out[p] = dot;
      if (S_out) S_out[p] = mag;
    }
  }
  return 0;
}

/*
 * FusedMM (same page, FusedMM section, Fig. 6, Algorithm 3, Fig. 11): row by
 * row, the SDDMM values a_ij = C_i . B_j of the row's stored positions are
 * computed and, without being stored, used at once as the sparse values of an
 * SpMM with a third dense matrix D (K x N): E_i = sum_j a_ij D_j.  Inputs are
 * the pattern (rowptr, colind), C, B and D; the output is E (M x N).
 * S_out[i][n] = sum_j |a_ij| |D_j[n]|, with a_ij exact, bounds the SpMM half;
 * A_out (nullable) receives the a_ij values in CSR order.
 */
int fusedmm_oracle_f64(int32_t M, int32_t K, int32_t N, const int32_t* rowptr, const int32_t* colind,
                       const float* C, const float* B, const float* D, double* E_out, double* S_out,
                       double* A_out) {
  if (M < 0 || K < 0 || N < 0 || !rowptr || !E_out) return -1;
  for (int32_t i = 0; i < M; ++i) {
    double* e = E_out + (int64_t)i * N;
    double* s = S_out ? S_out + (int64_t)i * N : NULL;
    for (int32_t n = 0; n < N; ++n) {
      e[n] = 0.0;
      if (s) s[n] = 0.0;
    }
    if (rowptr[i + 1] < rowptr[i]) return -2;
    for (int64_t p = rowptr[i]; p < rowptr[i + 1]; ++p) {
      const int64_t j = colind[p];
      if (j < 0 || j >= K) return -2;
      double a = 0.0;
      for (int32_t n = 0; n < N; ++n) a += (double)C[(int64_t)i * N + n] * (double)B[j * N + n];
      if (A_out) A_out[p] = a;
      for (int32_t n = 0; n < N; ++n) {
        const double prod = a * (double)D[j * N + n];
        e[n] += prod;
        if (s) s[n] += fabs(prod);
      }
    }
  }
  return 0;
}

/*
 * Semiring SpMM (page "Sgap: Towards Efficient Sparse Tensor Algebra
 * Compilation for GPU", sparse-dense hybrid algebra section, Eq. 3): the
 * reduction of SpMM generalised to a commutative operation (+) over the
 * row's stored entries of a binary operation (x) of the entry's value and
 * the dense element,
 *
 *     C[i][n] = (+)_{p = rowptr[i]}^{rowptr[i+1]-1} ( vals[p] (x) B[colind[p]][n] ).
 *
 * add_op: 0 = sum, 1 = min, 2 = max.  mul_op: 0 = multiply, 1 = add.  An
 * empty row gives the identity of (+): 0, +infinity, -infinity.  Each (x) is
 * one double-precision operation on two binary32 values (exact: a product of
 * two 24-bit significands fits in 53 bits, and so does a sum whose exponents
 * differ by at most 29; larger gaps round to the same binary32 either way).
 * S_out (sum only, may be NULL) is sum_p |vals[p] (x) B[colind[p]][n]|.
 * B is binary32.  Returns 0, -1 on an argument error, -2 on malformed CSR.
 */
int spmm_semiring_oracle_f64(int32_t M, int32_t K, int32_t N, const int32_t* rowptr,
                             const int32_t* colind, const float* vals, const float* B,
                             int32_t add_op, int32_t mul_op, double* C_out, double* S_out) {
  if (M < 0 || K < 0 || N < 0 || !rowptr || !C_out) return -1;
  if (add_op < 0 || add_op > 2 || mul_op < 0 || mul_op > 1) return -1;
  const double identity = add_op == 0 ? 0.0 : (add_op == 1 ? INFINITY : -INFINITY);
  for (int32_t i = 0; i < M; ++i) {
    double* c = C_out + (int64_t)i * N;
    double* s = S_out ? S_out + (int64_t)i * N : NULL;
    for (int32_t n = 0; n < N; ++n) {
      c[n] = identity;
      if (s) s[n] = 0.0;
    }
    if (rowptr[i + 1] < rowptr[i]) return -2;
    for (int64_t p = rowptr[i]; p < rowptr[i + 1]; ++p) {
      const double a = (double)vals[p];
      const int64_t j = colind[p];
      if (j < 0 || j >= K) return -2;
      for (int32_t n = 0; n < N; ++n) {
        const double b = (double)B[j * N + n];
        const double t = mul_op == 0 ? a * b : a + b;
        if (add_op == 0) {
          c[n] += t;
          if (s) s[n] += fabs(t);
        } else if (add_op == 1) {
          if (t < c[n]) c[n] = t;
        } else {
          if (t > c[n]) c[n] = t;
        }
      }
    }
  }
  return 0;
}
