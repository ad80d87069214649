// One-call SpMM that allocates no memory, and the error word that the
// one-call forms share.
//
// Some callers cannot call cudaMalloc or any other allocator at the moment
// they need a product: code running inside a memory pool or arena that owns
// all device memory, real-time loops where an allocation's implicit
// synchronisation or failure is not acceptable, and embedders whose own
// allocator must not be bypassed.  For them spmm_csr_f32_noalloc runs the
// nnz-balanced path with its scratch (merge-path range coordinates, carry
// rows of rows that cross ranges) carved from one fixed-size array in the
// library's own device memory instead.
//
// The array is a file-scope static __device__ object, so every GPU that
// loads the library holds it (kNoallocScratchBytes) until the process
// exits.  Host code cannot use the array's name as a device address: every
// call looks the address up with cudaGetSymbolAddress while the caller's
// device is current (a host-side lookup), so the address stays right even
// after the device's context has been reset and the library's device code
// loaded again.  All calls share the array and each call overwrites it:
// calls that may overlap on the GPU (different streams, or different host
// threads) race and must be ordered by the caller.
//
// The array's first 256 bytes hold the error word of the one-call forms
// (spmm_csr_f32, spmm_csr_bf16f32 and this one): their kernels OR a bit into
// it when a bounded wait gives up, and this form's partition kernel when the
// caller's nnz differs from rowptr[M].  The word is sticky; spmm_check_device
// reads and clears it.
#include <cstdint>

#include "spmm_device.cuh"
#include "spmm_internal.h"

namespace {

constexpr size_t kNoallocScratchBytes = size_t(32) << 20;  // 32 MiB per device
constexpr size_t kErrBytes = 256;                           // the shared error word, padded
constexpr int kNoallocItemsPerCta = spmm::kDefaultItemsPerCta;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];

// Device address of the scratch array on the current device.
cudaError_t noalloc_scratch(unsigned char** out) {
  void* p = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
  if (e != cudaSuccess) return e;
  *out = static_cast<unsigned char*>(p);
  return cudaSuccess;
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

}  // namespace

namespace spmm {

cudaError_t call_error_word(int** out) {
  unsigned char* base = nullptr;
  const cudaError_t e = noalloc_scratch(&base);
  if (e == cudaSuccess) *out = reinterpret_cast<int*>(base);
  return e;
}

}  // namespace spmm

extern "C" SPMM_API spmm_status spmm_csr_f32_noalloc(int32_t M, int32_t K, int32_t N, int64_t nnz,
                                                     const int32_t* rowptr, const int32_t* colind,
                                                     const float* vals, const float* B, float* C, void* stream) {
  using namespace spmm;
  if (M < 0 || K < 0 || N < 0 || nnz < 0) return SPMM_ERR_INVALID_ARG;
  if (M > SPMM_MAX_EXTENT || nnz > SPMM_MAX_EXTENT) return SPMM_ERR_UNSUPPORTED;
  if (M == 0 || N == 0) return SPMM_OK;
  if (!rowptr || !C || (nnz > 0 && (!colind || !vals || !B || K == 0))) return SPMM_ERR_INVALID_ARG;

  // Scratch layout: [error word | range coordinates (P+1) | carry rows (P x 2 x N)].
  const int64_t P = (int64_t(M) + nnz + kNoallocItemsPerCta - 1) / kNoallocItemsPerCta;
  const size_t part_bytes = align256(size_t(P + 1) * sizeof(int2));
  const size_t carry_bytes = size_t(P) * 2 * size_t(N) * sizeof(float);
  if (P > INT32_MAX - 1 || kErrBytes + part_bytes + carry_bytes > kNoallocScratchBytes)
    return SPMM_ERR_UNSUPPORTED;  // the problem needs more scratch than the fixed array holds

  unsigned char* scratch = nullptr;
  if (noalloc_scratch(&scratch) != cudaSuccess) return SPMM_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int* err = reinterpret_cast<int*>(scratch);
  int2* part = reinterpret_cast<int2*>(scratch + kErrBytes);
  float* carry = reinterpret_cast<float*>(scratch + kErrBytes + part_bytes);

  // Nothing in the array needs to start at zero: the ranges and the carry
  // rows are written before they are read, and the error word keeps earlier
  // calls' bits until spmm_check_device clears it.  The partition kernel
  // checks rowptr[M] == nnz and empties every range if not.
  if (launch_partition(rowptr, M, nnz, kNoallocItemsPerCta, int32_t(P), part, s, err) != cudaSuccess)
    return SPMM_ERR_CUDA;

  const bool vector_ok = N % 4 == 0 && (reinterpret_cast<uintptr_t>(B) & 15) == 0 &&
                         (reinterpret_cast<uintptr_t>(C) & 15) == 0;
  Launch L{};
  L.M = M;
  L.N = N;
  L.K = K;
  L.nnz = nnz;
  L.rowptr = rowptr;
  L.colind = colind;
  L.vals = vals;
  L.B = B;
  L.C = C;
  L.part = part;
  L.num_ctas = int32_t(P);
  L.items_per_cta = kNoallocItemsPerCta;
  L.carry = carry;
  L.err = err;
  L.stream = s;
  cudaError_t e = launch_balanced_f32(L, choose_shape_balanced(N, false, vector_ok));
  if (e == cudaSuccess) e = launch_fixup(L);
  return e == cudaSuccess ? SPMM_OK : e == cudaErrorNotSupported ? SPMM_ERR_UNSUPPORTED : SPMM_ERR_CUDA;
}

extern "C" SPMM_API spmm_status spmm_check_device(void* stream) {
  int* word = nullptr;
  if (spmm::call_error_word(&word) != cudaSuccess) return SPMM_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int host = 0;
  if (cudaMemcpyAsync(&host, word, sizeof host, cudaMemcpyDeviceToHost, s) != cudaSuccess) return SPMM_ERR_CUDA;
  if (cudaMemsetAsync(word, 0, sizeof host, s) != cudaSuccess) return SPMM_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return SPMM_ERR_CUDA;
  if (host & spmm::kErrInvalidCsr) return SPMM_ERR_INVALID_CSR;
  if (host & spmm::kErrBounds) return SPMM_ERR_OUT_OF_BOUNDS;
  if (host & spmm::kErrStageTimeout) return SPMM_ERR_DEVICE_TIMEOUT;
  return SPMM_OK;
}
