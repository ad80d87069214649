// Instantiations of the thread-range SpMM (and FusedMM) kernel: the shapes where it beats the
// balanced kernel's lane groups (library A/B on the rmat20 and rmat22 patterns,
// CUDA events, L2 flushed): N = 1 and 2 (scalar loads, fp32 or bf16 B), N = 4
// with 16-byte aligned fp32 B and N = 8 with 16-byte aligned bf16 B (one 16-byte
// load per nonzero in both).  At N = 3 and 5..7, and at N = 8 in fp32, the
// thread's row takes several scalar loads per nonzero, or two vectors, and the
// lane groups were faster.
#include "spmm_thread_ranges.cuh"

namespace spmm {

bool thread_ranges_shape(int32_t N, bool bf16, bool vector_ok) {
  return N <= 2 || (N == 4 && !bf16 && vector_ok) || (N == 8 && bf16 && vector_ok);
}

cudaError_t launch_thread_ranges(const Launch& L, bool bf16, bool vector_ok) {
  if (!thread_ranges_shape(L.N, bf16, vector_ok) || L.N < 1) return cudaErrorInvalidConfiguration;
  if (L.N == 4) return launch_thread_ranges_t<float, 4, 1>(L);
  if (L.N == 8) return launch_thread_ranges_t<uint16_t, 8, 1>(L);
  if (!bf16) return L.N == 1 ? launch_thread_ranges_t<float, 1, 1>(L) : launch_thread_ranges_t<float, 1, 2>(L);
  return L.N == 1 ? launch_thread_ranges_t<uint16_t, 1, 1>(L) : launch_thread_ranges_t<uint16_t, 1, 2>(L);
}

cudaError_t launch_thread_ranges_fused(const Launch& L, bool vector_ok, const float* Cd, const float* Bd) {
  if (!thread_ranges_shape(L.N, false, vector_ok) || L.N < 1) return cudaErrorInvalidConfiguration;
  if (L.N == 4) return launch_thread_ranges_t<float, 4, 1, true>(L, Cd, Bd);
  return L.N == 1 ? launch_thread_ranges_t<float, 1, 1, true>(L, Cd, Bd)
                  : launch_thread_ranges_t<float, 1, 2, true>(L, Cd, Bd);
}

}  // namespace spmm
