// C ABI entry points: exec with a plan, the one-call forms, status strings.
#include <algorithm>
#include <cstdint>

#include "spmm_internal.h"

spmm_status spmm_make_plan(const int32_t* rowptr, int32_t M, int64_t nnz, int32_t N, int32_t kernel,
                           int32_t items_per_cta, cudaStream_t stream, bool one_call, spmm_plan_t* plan_out);
void spmm_free_plan(spmm_plan_t plan, cudaStream_t stream);

namespace spmm {

static int pow2_at_least(int x) {
  int p = 1;
  while (p < x) p <<= 1;
  return p;
}

Shape choose_shape(int32_t N, bool bf16, bool vector_ok, int chunks_f32) {
  if (vector_ok) {
    const int vec = bf16 ? 8 : 4;
    const int chunks = bf16 ? (chunks_f32 / 2 > 0 ? chunks_f32 / 2 : 1) : chunks_f32;
    const int L = N / vec;  // 16-byte vectors per row (N is a multiple of vec here)
    if (L <= chunks) return Shape{vec, 1, pow2_at_least(L)};
    // G lanes of `chunks` vectors each; rows wider than 32 lanes run as column tiles
    return Shape{vec, std::min(32, pow2_at_least((L + chunks - 1) / chunks)), chunks};
  }
  return N <= 8 ? Shape{1, 8, 1} : Shape{1, 32, 1};
}

}  // namespace spmm

using namespace spmm;

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

// cudaErrorNotSupported from a launch: a size the kernels cannot address.
spmm_status status_of(cudaError_t e) {
  return e == cudaSuccess ? SPMM_OK : e == cudaErrorNotSupported ? SPMM_ERR_UNSUPPORTED : SPMM_ERR_CUDA;
}

struct DeviceGuard {  // run on the plan's device, restore the caller's afterwards
  int prev = -1;
  bool ok = true;
  explicit DeviceGuard(int dev) {
    if (cudaGetDevice(&prev) != cudaSuccess) { ok = false; return; }
    if (prev != dev && cudaSetDevice(dev) != cudaSuccess) ok = false;
  }
  ~DeviceGuard() {
    int cur;
    if (prev >= 0 && cudaGetDevice(&cur) == cudaSuccess && cur != prev) cudaSetDevice(prev);
  }
};

spmm_status exec(spmm_plan_t plan, int32_t K, const int32_t* colind, const float* vals, const void* B,
                 bool bf16, float* C, cudaStream_t stream) {
  if (!plan) return SPMM_ERR_PLAN_MISMATCH;
  if (K < 0) return SPMM_ERR_INVALID_ARG;
  if (plan->M == 0 || plan->N == 0) return SPMM_OK;
  if (!C || (plan->nnz > 0 && (!colind || !vals || !B || K == 0))) return SPMM_ERR_INVALID_ARG;
  DeviceGuard guard(plan->device);
  if (!guard.ok) return SPMM_ERR_CUDA;

  const bool vector_ok = plan->N % (bf16 ? 8 : 4) == 0 && aligned16(B) && aligned16(C);
  const bool row_family = plan->kernel == SPMM_KERNEL_ROW || plan->kernel == SPMM_KERNEL_WINDOW ||
                          plan->kernel == SPMM_KERNEL_SMALLN || plan->kernel == SPMM_KERNEL_WINDOW_TC;
  const Shape s = cap_tile(row_family ? choose_shape(plan->N, bf16, vector_ok)
                                      : choose_shape_balanced(plan->N, bf16, vector_ok), plan->column_tile);
  const bool window_family = plan->kernel == SPMM_KERNEL_WINDOW || plan->kernel == SPMM_KERNEL_WINDOW_TC;
  const bool window = window_family && s.G == 32 && s.nch == 1 && s.vec == (bf16 ? 8 : 4);
  const bool window_tc = plan->kernel == SPMM_KERNEL_WINDOW_TC && bf16 && plan->N % 16 == 0 && plan->N <= 256 &&
                         aligned16(B) && aligned16(C);
  Launch L{};
  L.M = plan->M;
  L.N = plan->N;
  L.K = K;
  L.nnz = plan->nnz;
  L.rowptr = plan->rowptr;
  L.colind = colind;
  L.vals = vals;
  L.B = B;
  L.C = C;
  L.part = plan->part;
  L.num_ctas = plan->num_ctas;
  L.items_per_cta = plan->items_per_cta;
  L.carry = plan->carry;
  L.err = plan->err;
  L.stream = stream;

  cudaError_t e;
  if (plan->kernel == SPMM_KERNEL_SMALLN && plan->N <= 8) {
    e = bf16 ? launch_rowgroup_bf16(L, plan->group_lanes) : launch_rowgroup_f32(L, plan->group_lanes);
    if (e == cudaSuccess && plan->split_event) e = cudaEventRecord(plan->split_event, stream);
  } else if (window_tc) {
    e = launch_tc_window_bf16(L);
    // no tensor-map encoder in this driver: the row kernel instead
    if (e == cudaErrorNotSupported) e = launch_row_bf16(L, s);
    if (e == cudaSuccess && plan->split_event) e = cudaEventRecord(plan->split_event, stream);
  } else if (window) {
    e = bf16 ? launch_window_bf16(L) : launch_window_f32(L);
    if (e == cudaSuccess && plan->split_event) e = cudaEventRecord(plan->split_event, stream);
  } else if (row_family) {
    e = bf16 ? launch_row_bf16(L, s) : launch_row_f32(L, s);
    if (e == cudaSuccess && plan->split_event) e = cudaEventRecord(plan->split_event, stream);
  } else {
    // narrow rows: a whole output row fits one thread, so each thread takes
    // its own slice of the range (no warp butterfly per row end)
    if (thread_ranges_shape(plan->N, bf16, vector_ok))
      e = launch_thread_ranges(L, bf16, vector_ok);
    else
      e = bf16 ? launch_balanced_bf16(L, s) : launch_balanced_f32(L, s);
    if (e == cudaSuccess && plan->split_event) e = cudaEventRecord(plan->split_event, stream);
    if (e == cudaSuccess) e = launch_fixup(L);
  }
  return status_of(e);
}

Launch plan_launch(spmm_plan_t plan, cudaStream_t stream) {
  Launch L{};
  L.M = plan->M;
  L.N = plan->N;
  L.nnz = plan->nnz;
  L.rowptr = plan->rowptr;
  L.part = plan->part;
  L.num_ctas = plan->num_ctas;
  L.items_per_cta = plan->items_per_cta;
  L.carry = plan->carry;
  L.err = plan->err;
  L.stream = stream;
  return L;
}

spmm_status sddmm(spmm_plan_t plan, int32_t K, const int32_t* colind, const float* Cd, const float* B, float* out,
                  cudaStream_t stream) {
  if (!plan) return SPMM_ERR_PLAN_MISMATCH;
  if (K < 0) return SPMM_ERR_INVALID_ARG;
  if (plan->nnz == 0) return SPMM_OK;
  if (!out || !colind) return SPMM_ERR_INVALID_ARG;
  DeviceGuard guard(plan->device);
  if (!guard.ok) return SPMM_ERR_CUDA;
  if (plan->N == 0)  // empty dot products
    return cudaMemsetAsync(out, 0, size_t(plan->nnz) * sizeof(float), stream) == cudaSuccess ? SPMM_OK : SPMM_ERR_CUDA;
  if (!Cd || !B || K == 0) return SPMM_ERR_INVALID_ARG;
  const bool vector_ok = plan->N % 4 == 0 && aligned16(B) && aligned16(Cd);
  Launch L = plan_launch(plan, stream);
  L.K = K;
  L.colind = colind;
  L.B = B;
  // Window-class plans (rows whose columns are local): the dense window of
  // each 32-row block from shared memory.
  const bool window_family = plan->kernel == SPMM_KERNEL_WINDOW || plan->kernel == SPMM_KERNEL_WINDOW_TC;
  if (window_family && vector_ok && plan->N <= 512) return status_of(launch_window_sddmm_f32(L, Cd, out));
  // Short, even rows (a row-class plan) and one 128-column tile: a group per
  // row keeps the C row in registers.
  const bool row_family = plan->kernel == SPMM_KERNEL_ROW || plan->kernel == SPMM_KERNEL_WINDOW ||
                          plan->kernel == SPMM_KERNEL_SMALLN || plan->kernel == SPMM_KERNEL_WINDOW_TC;
  if (row_family && vector_ok && plan->N <= 128) {
    const int G = std::max(4, pow2_at_least(plan->N / 4));
    const cudaError_t e = launch_sddmm_row_f32(L, G, Cd, out);
    return e == cudaSuccess ? SPMM_OK : SPMM_ERR_CUDA;
  }
  // Rows wider than one 128-column tile: two or four chunks per lane, so the
  // whole dot product comes from batched loads.
  Shape s = choose_shape_balanced(plan->N, false, vector_ok);
  if (vector_ok && s.G == 32 && plan->N > s.tile_width()) {
    int nch = 1;
    while (nch < 4 && 32 * 4 * nch < plan->N) nch <<= 1;
    s = Shape{4, 32, nch};
  }
  // Fewer lanes per dot product, each with more of the row: 8 lanes of N / 32
  // chunks at N = 64 and 128 (4 nonzeros a warp step), 4 lanes of two chunks
  // at N = 32; shorter reductions and more nonzeros per step (rmat20 at
  // N = 128 1,018 -> 572 us, its pattern at N = 64 521 -> 358 us, rmat22 at
  // N = 32 965 -> 924 us).
  if (vector_ok && (plan->N == 32 || plan->N == 64 || plan->N == 128))
    s = plan->N == 32 ? Shape{4, 4, 2} : Shape{4, 8, plan->N / 32};
  const cudaError_t e = launch_sddmm_f32(L, s, Cd, out);
  return e == cudaSuccess ? SPMM_OK : SPMM_ERR_CUDA;
}

spmm_status semiring(spmm_plan_t plan, int32_t K, const int32_t* colind, const float* vals, const float* B,
                     float* C, int32_t add_op, int32_t mul_op, cudaStream_t stream) {
  if (add_op < SPMM_ADD_SUM || add_op > SPMM_ADD_MAX || mul_op < SPMM_MUL_TIMES || mul_op > SPMM_MUL_PLUS)
    return SPMM_ERR_INVALID_ARG;
  const int sr = 2 * add_op + mul_op;
  if (sr == 0) return exec(plan, K, colind, vals, B, false, C, stream);
  if (!plan) return SPMM_ERR_PLAN_MISMATCH;
  if (K < 0) return SPMM_ERR_INVALID_ARG;
  if (plan->M == 0 || plan->N == 0) return SPMM_OK;
  if (!C || (plan->nnz > 0 && (!colind || !vals || !B || K == 0))) return SPMM_ERR_INVALID_ARG;
  DeviceGuard guard(plan->device);
  if (!guard.ok) return SPMM_ERR_CUDA;
  const bool vector_ok = plan->N % 4 == 0 && aligned16(B) && aligned16(C);
  Launch L = plan_launch(plan, stream);
  L.K = K;
  L.colind = colind;
  L.vals = vals;
  L.B = B;
  L.C = C;
  cudaError_t e = launch_semiring_f32(L, cap_tile(choose_shape_balanced(plan->N, false, vector_ok), plan->column_tile), sr);
  if (e == cudaSuccess && plan->split_event) e = cudaEventRecord(plan->split_event, stream);
  if (e == cudaSuccess) e = launch_fixup(L, sr);
  return status_of(e);
}

spmm_status fusedmm(spmm_plan_t plan, int32_t K, const int32_t* colind, const float* Cd, const float* B,
                    const float* D, float* E, cudaStream_t stream) {
  if (!plan) return SPMM_ERR_PLAN_MISMATCH;
  if (K < 0) return SPMM_ERR_INVALID_ARG;
  if (plan->M == 0 || plan->N == 0) return SPMM_OK;
  if (!E || (plan->nnz > 0 && (!colind || !Cd || !B || !D || K == 0))) return SPMM_ERR_INVALID_ARG;
  DeviceGuard guard(plan->device);
  if (!guard.ok) return SPMM_ERR_CUDA;
  const bool vector_ok = plan->N % 4 == 0 && aligned16(B) && aligned16(Cd) && aligned16(D) && aligned16(E);
  Launch L = plan_launch(plan, stream);
  L.K = K;
  L.colind = colind;
  L.B = D;  // gathered and accumulated
  L.C = E;
  // Window-class plans (rows whose columns are local): the dense window of
  // each 32-row block from shared memory, for both products.
  const bool window_family = plan->kernel == SPMM_KERNEL_WINDOW || plan->kernel == SPMM_KERNEL_WINDOW_TC;
  if (window_family && vector_ok && plan->N <= 512) {
    cudaError_t e = launch_window_fusedmm_f32(L, Cd, B);
    if (e == cudaSuccess && plan->split_event) e = cudaEventRecord(plan->split_event, stream);
    return status_of(e);
  }
  // Short, even rows (a row-class plan) and one 128-column tile: a group per
  // row keeps the C row and the E row in registers.
  const bool row_family = plan->kernel == SPMM_KERNEL_ROW || plan->kernel == SPMM_KERNEL_WINDOW ||
                          plan->kernel == SPMM_KERNEL_SMALLN || plan->kernel == SPMM_KERNEL_WINDOW_TC;
  if (row_family && vector_ok && plan->N <= 128) {
    cudaError_t e = launch_fusedmm_row_f32(L, std::max(4, pow2_at_least(plan->N / 4)), Cd, B);
    if (e == cudaSuccess && plan->split_event) e = cudaEventRecord(plan->split_event, stream);
    return e == cudaSuccess ? SPMM_OK : SPMM_ERR_CUDA;
  }
  // Narrow rows: one thread per slice of each range, the dot products in the thread.
  if (thread_ranges_shape(plan->N, false, vector_ok)) {
    cudaError_t e = launch_thread_ranges_fused(L, vector_ok, Cd, B);
    if (e == cudaSuccess && plan->split_event) e = cudaEventRecord(plan->split_event, stream);
    if (e == cudaSuccess) e = launch_fixup(L);
    return e == cudaSuccess ? SPMM_OK : SPMM_ERR_CUDA;
  }
  // Every column tile recomputes the dot products over all N columns, so wide
  // rows take one tile of up to 512 columns (two or four chunks per lane).
  Shape s = choose_shape_balanced(plan->N, false, vector_ok);
  if (vector_ok && s.G == 32 && plan->N > s.tile_width()) {
    int nch = 1;
    while (nch < 4 && 32 * 4 * nch < plan->N) nch <<= 1;
    s = Shape{4, 32, nch};
  }
  cudaError_t e = launch_fusedmm_f32(L, s, Cd, B);
  if (e == cudaSuccess && plan->split_event) e = cudaEventRecord(plan->split_event, stream);
  if (e == cudaSuccess) e = launch_fixup(L);
  return e == cudaSuccess ? SPMM_OK : SPMM_ERR_CUDA;
}

spmm_status one_call(int32_t M, int32_t K, int32_t N, const int32_t* rowptr, const int32_t* colind,
                     const float* vals, const void* B, bool bf16, float* C, void* stream) {
  if (M < 0 || K < 0 || N < 0) return SPMM_ERR_INVALID_ARG;
  if (M == 0 || N == 0) return SPMM_OK;
  if (!rowptr) return SPMM_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // nnz = rowptr[M] comes back with the row statistics (one synchronisation).
  spmm_plan_t plan = nullptr;
  spmm_status st = spmm_make_plan(rowptr, M, -1, N, SPMM_KERNEL_AUTO, 0, s, true, &plan);
  if (st != SPMM_OK) return st;
  // The kernels report to the one-call forms' shared error word, which
  // outlives this plan (spmm_check_device reads it).
  if (plan->err && call_error_word(&plan->err) != cudaSuccess) {
    spmm_free_plan(plan, s);
    return SPMM_ERR_CUDA;
  }
  st = exec(plan, K, colind, vals, B, bf16, C, s);
  spmm_free_plan(plan, s);
  return st;
}

}  // namespace

extern "C" {

spmm_status spmm_csr_f32_exec(spmm_plan_t plan, int32_t K, const int32_t* colind, const float* vals,
                              const float* B, float* C, void* stream) {
  return exec(plan, K, colind, vals, B, false, C, static_cast<cudaStream_t>(stream));
}

spmm_status spmm_csr_bf16f32_exec(spmm_plan_t plan, int32_t K, const int32_t* colind, const float* vals,
                                  const uint16_t* B, float* C, void* stream) {
  return exec(plan, K, colind, vals, B, true, C, static_cast<cudaStream_t>(stream));
}

spmm_status spmm_csr_f32(int32_t M, int32_t K, int32_t N, const int32_t* rowptr, const int32_t* colind,
                         const float* vals, const float* B, float* C, void* stream) {
  return one_call(M, K, N, rowptr, colind, vals, B, false, C, stream);
}

spmm_status spmm_csr_bf16f32(int32_t M, int32_t K, int32_t N, const int32_t* rowptr, const int32_t* colind,
                             const float* vals, const uint16_t* B, float* C, void* stream) {
  return one_call(M, K, N, rowptr, colind, vals, B, true, C, stream);
}

spmm_status spmm_csr_sddmm_f32(spmm_plan_t plan, int32_t K, const int32_t* colind, const float* C, const float* B,
                               float* out, void* stream) {
  return sddmm(plan, K, colind, C, B, out, static_cast<cudaStream_t>(stream));
}

spmm_status spmm_csr_semiring_f32_exec(spmm_plan_t plan, int32_t K, const int32_t* colind, const float* vals,
                                       const float* B, float* C, int32_t add_op, int32_t mul_op, void* stream) {
  return semiring(plan, K, colind, vals, B, C, add_op, mul_op, static_cast<cudaStream_t>(stream));
}

spmm_status spmm_csr_fusedmm_f32(spmm_plan_t plan, int32_t K, const int32_t* colind, const float* C,
                                 const float* B, const float* D, float* E, void* stream) {
  return fusedmm(plan, K, colind, C, B, D, E, static_cast<cudaStream_t>(stream));
}

spmm_status spmm_plan_set_split_event(spmm_plan_t plan, void* event) {
  if (!plan) return SPMM_ERR_INVALID_ARG;
  plan->split_event = static_cast<cudaEvent_t>(event);
  return SPMM_OK;
}

const char* spmm_status_string(spmm_status status) {
  switch (status) {
    case SPMM_OK: return "SPMM_OK";
    case SPMM_ERR_INVALID_ARG: return "SPMM_ERR_INVALID_ARG";
    case SPMM_ERR_INVALID_CSR: return "SPMM_ERR_INVALID_CSR";
    case SPMM_ERR_UNSUPPORTED: return "SPMM_ERR_UNSUPPORTED";
    case SPMM_ERR_PLAN_MISMATCH: return "SPMM_ERR_PLAN_MISMATCH";
    case SPMM_ERR_CUDA: return "SPMM_ERR_CUDA";
    case SPMM_ERR_DEVICE_TIMEOUT: return "SPMM_ERR_DEVICE_TIMEOUT";
    case SPMM_ERR_OUT_OF_BOUNDS: return "SPMM_ERR_OUT_OF_BOUNDS";
  }
  return "SPMM_ERR_UNKNOWN";
}

}  // extern "C"
