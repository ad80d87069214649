// Instantiations of the window SDDMM and FusedMM kernels (fp32).
#include "spmm_window_sddmm.cuh"

namespace spmm {

cudaError_t launch_window_sddmm_f32(const Launch& L, const float* Cd, float* out) {
  return launch_window_sddmm_t<false>(L, Cd, static_cast<const float*>(L.B), out);
}

cudaError_t launch_window_fusedmm_f32(const Launch& L, const float* Cd, const float* Bd) {
  return launch_window_sddmm_t<true>(L, Cd, Bd, L.C);
}

}  // namespace spmm
