/*
 * csr_spmm_02_gb300 -- C ABI of the GB300 (sm_103a) CSR SpMM library.
 *
 * Operation (SpMM, page "Performance Optimization of Deep Learning Sparse
 * Matrix Kernels on Intel Max Series GPU", SPMM section, Fig. 5 and
 * Algorithm 2; the same reduction over the sparse index j is the core
 * operation named on the page "Sgap: Towards Efficient Sparse Tensor Algebra
 * Compilation for GPU", sparse-dense hybrid algebra section):
 *
 *     C[i][n] = sum_{p = rowptr[i]}^{rowptr[i+1]-1} vals[p] * B[colind[p]][n]
 *
 * for 0 <= i < M, 0 <= n < N.  A is M x K in CSR form; B (K x N) and C
 * (M x N) are dense and row-major.  C is overwritten (never accumulated
 * into); an empty row of A gives a zero row of C.  Duplicate (i, j) entries
 * are summed and column indices need not be sorted.
 *
 * Types and layout
 *   rowptr  int32[M+1], rowptr[0] = 0, non-decreasing, rowptr[M] = nnz
 *   colind  int32[nnz], each in [0, K)
 *   vals    fp32[nnz]
 *   B       fp32[K*N], or bf16[K*N] passed as its raw uint16 bit patterns
 *   C       fp32[M*N]
 *   The bf16 variants widen B exactly to fp32 and accumulate in fp32.
 *
 * Pointers and ownership
 *   Every array pointer is a DEVICE pointer owned by the caller; the library
 *   never frees or retains them, except that a plan remembers `rowptr` and
 *   reads it again on every exec (keep it alive and unchanged while the plan
 *   is used).  The library writes only C and its own plan workspace.
 *   `stream` is a cudaStream_t passed as void* (NULL = the legacy default
 *   stream).  All calls are asynchronous on `stream` unless stated.
 *
 * Sizes
 *   M, K, N >= 0; M <= SPMM_MAX_EXTENT and 0 <= nnz <= SPMM_MAX_EXTENT
 *   (2^31 - 65536: the kernels index rows and nonzeros in 32 bits and step
 *   past the last one by small offsets, which must not overflow); larger M
 *   or nnz return SPMM_ERR_UNSUPPORTED.  M = 0 or N = 0 is a successful no-op.
 *   The nnz-balanced SpMM kernel (SPMM_KERNEL_BALANCED, the semirings and
 *   spmm_csr_f32_noalloc) addresses B with 32-bit offsets of 16-byte vectors
 *   (of single elements on the scalar path): it returns SPMM_ERR_UNSUPPORTED
 *   when K * N / 4 (fp32 B), K * N / 8 (bf16 B) or, on the scalar path, K * N
 *   exceeds 2^32 - 1.
 *   Any N >= 1 is supported.  16-byte vector paths are used when N is a
 *   multiple of 4 (fp32 B) or 8 (bf16 B) and B and C are 16-byte aligned;
 *   otherwise a scalar path runs with the same results.
 *
 * Results and determinism
 *   No floating-point atomics are used: for a given plan, repeated calls give
 *   bitwise-identical C.  The summation order differs from a sequential loop
 *   (rows may be split into pieces that are combined in a fixed order).
 *
 * Non-finite values
 *   Inputs are expected to be finite.  The kernels multiply some B rows by a
 *   zero value instead of skipping them (slots past the end of a row or of a
 *   batch re-read a valid row with value 0; the window kernels multiply the
 *   absent entries inside the window), so an Inf or NaN in B can turn into
 *   NaN: in the row kernel only in a row that references that B row, in the
 *   nnz-balanced kernel also in a row whose nonzeros share a warp step with
 *   such a reference, in the window kernels in every row of the block whose
 *   window holds that B row.
 *
 * Errors
 *   Every call returns a spmm_status; no exception crosses the ABI and no
 *   kernel traps.  Argument errors are detected before any CUDA call.
 *   Column indices outside [0, K) and malformed rowptr are NOT checked on
 *   the fast path (undefined results); run spmm_csr_validate to check them.
 *   A CUDA launch or API failure returns SPMM_ERR_CUDA.  Kernels that wait
 *   on hardware copies give up after a bounded time and record
 *   SPMM_ERR_DEVICE_TIMEOUT in the plan, read by spmm_plan_check_device; the
 *   one-call forms record it in a per-device word read by spmm_check_device.
 */
#ifndef CSR_SPMM_02_GB300_SPMM_H_
#define CSR_SPMM_02_GB300_SPMM_H_

#include <stdint.h>

/* Largest M and nnz the library accepts (2^31 - 65536). */
#define SPMM_MAX_EXTENT 2147418112

/* Only the functions below are exported; everything else in the library is
 * hidden (it is built with -fvisibility=hidden). */
#if defined(__GNUC__)
#define SPMM_API __attribute__((visibility("default")))
#else
#define SPMM_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  SPMM_OK = 0,
  SPMM_ERR_INVALID_ARG = 1,    /* bad size, NULL pointer, unknown option */
  SPMM_ERR_INVALID_CSR = 2,    /* spmm_csr_validate found a malformed CSR */
  SPMM_ERR_UNSUPPORTED = 3,    /* a size the library cannot handle (e.g. nnz > SPMM_MAX_EXTENT) */
  SPMM_ERR_PLAN_MISMATCH = 4,  /* exec called with a plan made for another shape */
  SPMM_ERR_CUDA = 5,           /* a CUDA runtime call or launch failed */
  SPMM_ERR_DEVICE_TIMEOUT = 6, /* a kernel's bounded wait expired (see above) */
  SPMM_ERR_OUT_OF_BOUNDS = 7   /* only in a bounds-checked build: an index pointed outside
                                * its buffer and the access was skipped */
} spmm_status;

/* Kernel family a plan uses. */
typedef enum {
  SPMM_KERNEL_AUTO = 0,      /* chosen from the row-length statistics (rowptr only): skewed
                              * rows -> BALANCED; even rows -> SMALLN for N <= 8, WINDOW_TC
                              * for N >= 128 (which assumes local columns: on scattered
                              * columns force ROW, faster there), else ROW */
  SPMM_KERNEL_ROW = 1,       /* one (sub-)warp group per row: short, uniform rows */
  SPMM_KERNEL_BALANCED = 2,  /* merge-path nnz-balanced split + fixup: skewed rows */
  SPMM_KERNEL_WINDOW = 3,    /* short rows, B rows reused across rows: a CTA of 32 rows
                              * whose columns span few enough B rows stages them in
                              * shared memory and reuses each from registers for 4
                              * rows; other CTAs gather as the row kernel.  Runs when a
                              * warp covers the column tile (N >= 128 fp32 with 4-column
                              * lanes, N >= 256 bf16 with 8-column lanes, 16-byte
                              * aligned B and C); otherwise exec runs the row kernel.
                              * Absent entries inside the window are multiplied as
                              * zeros, so a NaN/Inf in such a B row reaches the row. */
  SPMM_KERNEL_SMALLN = 4,    /* N <= 8: a group of r lanes shares each row, every lane
                              * holding the whole output row (the Sgap page's
                              * {<1/g row, c col>, r} point, atomic parallelism, Table 1);
                              * r from the plan (spmm_plan_set_group_lanes overrides).
                              * For N > 8 exec runs the row kernel instead. */
  SPMM_KERNEL_WINDOW_TC = 5  /* the window kernel's dense product on the tensor cores
                              * (tcgen05, accumulator in tensor memory) for bf16 B with
                              * N a multiple of 16 up to 256: a persistent kernel over
                              * 128-row tiles, A's fp32 values split exactly into three
                              * bf16 terms (exact for |vals| >= 2^-110), B streamed by
                              * TMA in 64-row chunks; tiles with a span over 192
                              * columns, duplicate columns or a nonzero value below
                              * 2^-110 in magnitude gather per row in fp32.  Other B
                              * types or widths run the window kernel.  Absent entries
                              * inside the window are multiplied as zeros, as in the
                              * window kernel. */
} spmm_kernel;

/* Opaque plan: owns its device workspace (merge-path partition, carry rows
 * of split rows, an error word).  Bound to (rowptr, M, nnz, N). */
typedef struct spmm_plan_s* spmm_plan_t;

/* What a plan decided (host copy, filled by spmm_plan_get_info). */
typedef struct {
  int32_t kernel;          /* the spmm_kernel value exec runs (never SPMM_KERNEL_AUTO) */
  int32_t M;
  int64_t nnz;
  int32_t N;
  int32_t max_row_nnz;     /* longest row of A */
  int32_t empty_rows;      /* rows of A with no nonzero */
  int32_t items_per_cta;   /* balanced: merge-path items (row ends + nonzeros) per CTA */
  int32_t num_ctas;        /* balanced: number of merge-path ranges (CTAs) */
  int64_t workspace_bytes; /* device bytes the plan owns */
  int32_t group_lanes;     /* SMALLN: lanes r that share a row (2..32) */
  int32_t column_tile;     /* N-slicing cap set by spmm_plan_set_column_tile (0: none) */
} spmm_plan_info;

/*
 * Build a plan for A's row structure (nnz-balanced row partitioning).
 * Reads rowptr (device, M+1 entries) on `stream` in one pass (one kernel):
 * the row-length statistics and rowptr[M], which are copied to the host
 * (this call synchronises `stream` once), and the merge-path partition -- the
 * merged sequence of row ends and nonzeros cut into equal ranges, the even
 * nnz split the Sgap page's related work attributes to Yang et al. and the
 * element-balanced EB scheme of its DA-SpMM design space; row i's end sits at
 * position rowptr[i+1] + i, so each row writes the range starts that fall in
 * it, with no search.  nnz must equal rowptr[M]: SPMM_ERR_INVALID_CSR
 * otherwise.  The plan's workspace comes stream-ordered on `stream`
 * (cudaMallocFromPoolAsync) from a pool the library creates on each device
 * at its first plan; the pool keeps freed blocks reserved for later plans
 * (spmm_pool_release hands them back).  *plan_out receives the plan (NULL on
 * error).  A plan's workspace (range carry rows, error word) serves one call
 * at a time: calls that may overlap on the device (several streams) need a
 * plan each.
 */
SPMM_API spmm_status spmm_csr_plan(const int32_t* rowptr, int32_t M, int64_t nnz, int32_t N,
                          void* stream, spmm_plan_t* plan_out);

/*
 * As spmm_csr_plan, with the kernel family forced (spmm_kernel value) and
 * the merge-path range size set: items_per_cta = 0 picks the default (3072
 * items for 8 < N <= 32, 3840 for N = 1, 3, 4 and 8, else 2048), otherwise it must be a positive multiple of
 * 256, at most 8192.  The default serves SpMM and FusedMM; a plan used only
 * for SDDMM at N = 8 runs faster on 2048-item ranges (R-MAT patterns: about
 * 5% at scale 20, 20% at scale 22).
 */
SPMM_API spmm_status spmm_csr_plan_ex(const int32_t* rowptr, int32_t M, int64_t nnz, int32_t N,
                             int32_t kernel, int32_t items_per_cta, void* stream,
                             spmm_plan_t* plan_out);

/* Set the lanes r (2, 4, 8, 16 or 32) that share a row in the SMALLN kernel;
 * SPMM_ERR_INVALID_ARG for another value or a plan of another kernel. */
SPMM_API spmm_status spmm_plan_set_group_lanes(spmm_plan_t plan, int32_t lanes);

/*
 * N-slicing (L2-level chunking: the kkmem page's multilevel chunking moved
 * from host/HBM to L2/HBM): cap the column tile of the row and balanced kernels at
 * `columns` (0 removes the cap), so that each tile's slice of B (K x tile
 * columns) is what L2 holds at a time; the tiles run in order.  The plan's
 * own choice is one tile: on the measured workloads narrower tiles were
 * slower (each repeats every nonzero's bookkeeping).  The window and
 * small-N kernels keep their own tiles.  SPMM_ERR_INVALID_ARG if columns < 0.
 */
SPMM_API spmm_status spmm_plan_set_column_tile(spmm_plan_t plan, int32_t columns);

/* Copy the plan's decisions into *info (host memory).  Every plan also holds
 * the merge-path partition used by the balanced SpMM, SDDMM and FusedMM. */
SPMM_API spmm_status spmm_plan_get_info(spmm_plan_t plan, spmm_plan_info* info);

/* Free the plan and its workspace (synchronises the device first, since the
 * plan may be in use on any stream).  NULL is accepted. */
SPMM_API spmm_status spmm_plan_destroy(spmm_plan_t plan);

/*
 * C = A . B with fp32 B, using a plan made for this A (same rowptr, M, nnz,
 * N).  K is B's row count (colind values must lie in [0, K)).  Asynchronous
 * on `stream`.  Returns SPMM_ERR_PLAN_MISMATCH for a NULL plan.
 *
 * CUDA graphs: the exec calls (SpMM, SDDMM, FusedMM, semirings) make no
 * synchronous CUDA call and allocate nothing.  The first call of each
 * kernel on a device sets that kernel's shared-memory attribute; after it,
 * an exec call can be captured on `stream` into a CUDA graph, and every
 * replay reads the captured buffers as they are when it runs.  (Plans and
 * the one-call forms synchronise and cannot be captured.)
 */
SPMM_API spmm_status spmm_csr_f32_exec(spmm_plan_t plan, int32_t K, const int32_t* colind,
                              const float* vals, const float* B, float* C, void* stream);

/* As spmm_csr_f32_exec with B in bf16 (uint16 bit patterns), fp32 accumulate. */
SPMM_API spmm_status spmm_csr_bf16f32_exec(spmm_plan_t plan, int32_t K, const int32_t* colind,
                                  const float* vals, const uint16_t* B, float* C,
                                  void* stream);

/*
 * SDDMM on A's pattern (page "Performance Optimization of Deep Learning Sparse
 * Matrix Kernels on Intel Max Series GPU", SDDMM section, Algorithm 1):
 * out[p] = sum_n C[i][n] * B[colind[p]][n] for every stored position p of
 * row i.  A's values are not used.  C is M x N, B is K x N (fp32, row-major,
 * N the plan's width); out is fp32[nnz] in CSR order.  A plan whose kernel is
 * WINDOW or WINDOW_TC (short rows with local columns) with N <= 512, N a
 * multiple of 4 and 16-byte aligned B and C computes each 32-row block's dense
 * window from shared memory (a block whose columns span more than 96 gathers
 * instead); one whose kernel is ROW or SMALLN with N <= 128 and the same
 * alignment runs one lane group per row with the C row in registers;
 * otherwise the plan's merge-path ranges.
 * Asynchronous on `stream`; every output written once, so results are
 * deterministic.  Tolerance-wise each value is an fp32 dot product.
 */
SPMM_API spmm_status spmm_csr_sddmm_f32(spmm_plan_t plan, int32_t K, const int32_t* colind, const float* C,
                                        const float* B, float* out, void* stream);

/* Operators of the semiring form below. */
typedef enum {
  SPMM_ADD_SUM = 0,  /* (+) = addition, identity 0 */
  SPMM_ADD_MIN = 1,  /* (+) = minimum, identity +infinity */
  SPMM_ADD_MAX = 2   /* (+) = maximum, identity -infinity */
} spmm_add_op;
typedef enum {
  SPMM_MUL_TIMES = 0, /* (x) = multiplication */
  SPMM_MUL_PLUS = 1   /* (x) = addition (with SPMM_ADD_MIN: the tropical semiring) */
} spmm_mul_op;

/*
 * Semiring SpMM (page "Sgap: Towards Efficient Sparse Tensor Algebra
 * Compilation for GPU", sparse-dense hybrid algebra, Eq. 3, where the
 * reduction's (+) may be any commutative operation and (x) any binary one):
 * C[i][n] = (+) over the stored p of row i of vals[p] (x) B[colind[p]][n],
 * with an empty row giving the identity of (+).  fp32 B and C, arguments as
 * in spmm_csr_f32_exec.  (SUM, TIMES) is the ordinary SpMM and runs the
 * plan's own kernel; any other pair runs the nnz-balanced kernel and its
 * fixup with that (+) and (x).  min and max are exact in any order, so those
 * results are bitwise the binary32 rounding of the exact value; sums carry
 * fp32 rounding.  SPMM_ERR_INVALID_ARG for an unknown operator.
 */
SPMM_API spmm_status spmm_csr_semiring_f32_exec(spmm_plan_t plan, int32_t K, const int32_t* colind,
                                                const float* vals, const float* B, float* C,
                                                int32_t add_op, int32_t mul_op, void* stream);

/*
 * FusedMM (same page, FusedMM section, Fig. 6, Algorithm 3, Fig. 11):
 * E[i] = sum over stored j of row i of (C[i] . B[j]) * D[j], the SDDMM values
 * used at once as the sparse values of an SpMM and never stored.  C is M x N,
 * B and D are K x N, E is M x N (fp32, row-major, N the plan's width).  On the
 * plans and widths where SDDMM uses the window (above), both products come
 * from the window in shared memory (the values stay in shared memory, and
 * absent entries inside the window are multiplied as zeros, as in the window
 * SpMM kernel); where SDDMM runs a group per row, one lane group per row
 * keeps C[i] and E[i] in registers; otherwise the nnz-balanced kernel and its
 * fixup run.  Deterministic for a given plan.
 */
SPMM_API spmm_status spmm_csr_fusedmm_f32(spmm_plan_t plan, int32_t K, const int32_t* colind, const float* C,
                                          const float* B, const float* D, float* E, void* stream);

/*
 * One-call form: plans, multiplies and frees on `stream`.  nnz is read from
 * rowptr[M] with the plan's statistics (one copy, which synchronises `stream`
 * once; SPMM_ERR_INVALID_CSR if it is negative).  The plan's workspace comes
 * from the library's pool (see spmm_csr_plan) and is returned to it
 * stream-ordered (cudaFreeAsync) at the end of the call, so repeated calls
 * map no new memory.  The merge-path partition is built
 * only when the chosen kernel is the balanced one.  For repeated products
 * with the same A, build a plan once and call the _exec form.  A bounded
 * wait that gives up in this call's kernels is recorded in the device's
 * one-call error word (see spmm_check_device), not in the returned status.
 * colind and vals must hold rowptr[M] entries: the call cannot check their
 * sizes.
 */
SPMM_API spmm_status spmm_csr_f32(int32_t M, int32_t K, int32_t N, const int32_t* rowptr,
                         const int32_t* colind, const float* vals, const float* B, float* C,
                         void* stream);

/* One-call form with bf16 B (uint16 bit patterns), fp32 accumulate. */
SPMM_API spmm_status spmm_csr_bf16f32(int32_t M, int32_t K, int32_t N, const int32_t* rowptr,
                             const int32_t* colind, const float* vals, const uint16_t* B,
                             float* C, void* stream);

/*
 * Check a CSR structure on the device: rowptr[0] = 0, rowptr non-decreasing,
 * rowptr[M] = nnz, every colind in [0, K).  Synchronous (waits for
 * `stream`).  Returns SPMM_OK or SPMM_ERR_INVALID_CSR.  Uses a 4-byte
 * stream-ordered device allocation from the one-call pool.
 */
SPMM_API spmm_status spmm_csr_validate(const int32_t* rowptr, const int32_t* colind, int32_t M,
                              int32_t K, int64_t nnz, void* stream);

/*
 * Synchronise `stream`, read and clear the plan's device error word.
 * Returns SPMM_ERR_OUT_OF_BOUNDS if (in a library built with
 * -DSPMM_DEBUG_BOUNDS, where every B-row gather and every output store checks
 * its address) an access fell outside its buffer, else
 * SPMM_ERR_DEVICE_TIMEOUT if a kernel run with this plan gave up a bounded
 * wait since the last check, else SPMM_OK.
 */
SPMM_API spmm_status spmm_plan_check_device(spmm_plan_t plan, void* stream);

/*
 * C = A . B with fp32 B, allocating no memory at all (no cudaMalloc,
 * cudaMallocAsync or allocating library call, here or in the kernels).  The
 * pages this library follows have no counterpart to this call: it exists for
 * callers that must not allocate while they multiply -- code inside a memory
 * pool or arena that owns all device memory, real-time loops that cannot
 * accept an allocation's synchronisation or failure, embedders whose own
 * allocator must not be bypassed.
 *
 * It always runs the nnz-balanced kernel and its fixup, with their scratch
 * (range coordinates, carry rows) in one fixed 32 MiB array of device memory
 * that the library itself holds on every device that loads it, until the
 * process exits.  The caller passes all inputs and the output, as for
 * spmm_csr_f32, plus nnz.  A problem whose scratch, 256 + 8 * (P + 1)
 * (rounded up to 256) + 8 * N * P bytes with P = ceil((M + nnz) / 2048),
 * exceeds the array is rejected with SPMM_ERR_UNSUPPORTED before anything is
 * launched.  Every call looks up the array's device address on the current
 * device (cudaGetSymbolAddress, a host-side lookup); the first call on a
 * device also loads the library's device code there, so make it before any
 * stream capture on that device.  Every call reuses the same array and
 * leaves its contents behind: calls whose work can overlap on the GPU (other
 * streams, other threads) race; order them.  Asynchronous on `stream`;
 * results are bitwise reproducible for given inputs.
 *
 * nnz must equal rowptr[M].  The call cannot see rowptr[M] without a
 * synchronisation, so the check runs on the device: on a mismatch no range
 * reads any nonzero, C is left unwritten and spmm_check_device returns
 * SPMM_ERR_INVALID_CSR.  A bounded wait that gives up is reported there too
 * (SPMM_ERR_DEVICE_TIMEOUT).  SPMM_OK from this call means only that the
 * work was launched: call spmm_check_device to learn whether it completed.
 */
SPMM_API spmm_status spmm_csr_f32_noalloc(int32_t M, int32_t K, int32_t N, int64_t nnz,
                                          const int32_t* rowptr, const int32_t* colind,
                                          const float* vals, const float* B, float* C, void* stream);

/*
 * Row-block split of one A over `parts` GPUs (host code; no CUDA call).
 * `rowptr` is a HOST array of M+1 entries; row_start (host, parts+1 entries,
 * owned by the caller) receives the first row of every block, row_start[0] =
 * 0 and row_start[parts] = M.  The merged sequence of nonzeros and row ends
 * (M + nnz items) is cut into `parts` equal diagonals, as the plan cuts it
 * into CTA ranges (the even split of nonzeros the Sgap page's related work
 * credits to Yang et al.), with each row kept whole in the block that holds
 * its end, so every GPU multiplies the rows row_start[b] .. row_start[b+1]-1
 * by a replicated B and writes that block of C, with no exchange of partial
 * rows (the Intel Max page scales one problem over both stacks of its GPU
 * the same way, with one queue per stack).  A block may be empty when one
 * row is longer than a whole share.  SPMM_ERR_INVALID_ARG for M < 0,
 * parts < 1 or a NULL pointer; SPMM_ERR_INVALID_CSR if rowptr[0] != 0 or
 * rowptr decreases.
 */
SPMM_API spmm_status spmm_csr_row_blocks(const int32_t* rowptr, int32_t M, int32_t parts, int32_t* row_start);

/*
 * Synchronise `stream`, then read and clear the error word that the one-call
 * forms (spmm_csr_f32, spmm_csr_bf16f32, spmm_csr_f32_noalloc) share on the
 * current device.  The word collects the bits of every such call on the
 * device since the last check, whatever its stream.  Returns
 * SPMM_ERR_INVALID_CSR if a spmm_csr_f32_noalloc call was given an nnz other
 * than rowptr[M] (that call wrote nothing), else SPMM_ERR_OUT_OF_BOUNDS (a
 * bounds-checked build only, see spmm_plan_check_device), else
 * SPMM_ERR_DEVICE_TIMEOUT if a kernel gave up a bounded wait (its output is
 * incomplete), else SPMM_OK.
 * Allocates nothing.
 */
SPMM_API spmm_status spmm_check_device(void* stream);

/*
 * Optional timing hook.  When `event` (a cudaEvent_t passed as void*) is not
 * NULL, every later exec with this plan records it on the exec stream right
 * after the main SpMM kernel, before the balanced family's fixup kernel, so
 * the main kernel can be timed alone with events.  NULL clears the hook.  The
 * caller owns the event and keeps it alive while it is set.
 */
SPMM_API spmm_status spmm_plan_set_split_event(spmm_plan_t plan, void* event);

/*
 * Return to the system the device memory that the library's pools (one per
 * device, see spmm_csr_plan) keep reserved between plans.  Blocks still in
 * use (live plans), or freed on a stream that has not reached the free yet,
 * stay with the pool: synchronise the streams that ran one-call forms first.
 * Safe to call at any time, from any thread; SPMM_ERR_CUDA if a trim fails.
 */
SPMM_API spmm_status spmm_pool_release(void);

/* Static, human-readable name of a status code. */
SPMM_API const char* spmm_status_string(spmm_status status);

#ifdef __cplusplus
}
#endif

#endif /* CSR_SPMM_02_GB300_SPMM_H_ */
