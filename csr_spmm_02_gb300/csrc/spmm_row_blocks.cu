// Row-block split of one A over several GPUs (host code only).
//
// The merged sequence of A's nonzeros and row ends (M + nnz items; row i's
// end sits at position rowptr[i+1] + i) is cut into `parts` equal diagonals,
// as the balanced kernel's plan cuts it into CTA ranges, but at GPU
// granularity and with every row kept whole: block b holds the rows whose end
// item lies in [d_b, d_{b+1}), d_b = floor(b * (M + nnz) / parts).  A row
// that a diagonal cuts goes wholly to the block that holds its end, so each
// GPU writes a disjoint block of C rows from A's rows and a replicated B, and
// no partial row crosses GPUs.  This is the even split of nonzeros (counting
// output rows too) that the Sgap page's related work credits to Yang et al.,
// applied across devices, as the Intel Max page's introduction scales one
// problem over both stacks of its GPU.
#include <cstdint>

#include "spmm_internal.h"

extern "C" SPMM_API spmm_status spmm_csr_row_blocks(const int32_t* rowptr, int32_t M, int32_t parts,
                                                    int32_t* row_start) {
  if (M < 0 || parts < 1 || !row_start || !rowptr) return SPMM_ERR_INVALID_ARG;
  if (rowptr[0] != 0) return SPMM_ERR_INVALID_CSR;
  for (int32_t i = 0; i < M; ++i)
    if (rowptr[i + 1] < rowptr[i]) return SPMM_ERR_INVALID_CSR;
  const int64_t total = int64_t(M) + int64_t(rowptr[M]);
  for (int32_t b = 0; b <= parts; ++b) {
    const int64_t d = total * b / parts;
    // first row whose end item rowptr[r+1] + r lies at or after d (M if none)
    int32_t lo = 0, hi = M;
    while (lo < hi) {
      const int32_t mid = lo + (hi - lo) / 2;
      if (int64_t(rowptr[mid + 1]) + mid >= d) hi = mid; else lo = mid + 1;
    }
    row_start[b] = lo;
  }
  row_start[parts] = M;  // the last block ends with the last row, whatever rounding did
  return SPMM_OK;
}
