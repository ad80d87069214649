// Instantiations of the FusedMM kernels (fp32): the balanced kernel in
// FusedMM mode and the group-per-row form.
#include "spmm_balanced.cuh"
#include "spmm_sddmm_row.cuh"

namespace spmm {

cudaError_t launch_fusedmm_f32(const Launch& L, Shape s, const float* Cd, const float* Bd) {
#define X(V, GG, NC) \
  if (s.vec == V && s.G == GG && s.nch == NC) return launch_balanced_t<float, V, GG, NC, true>(L, Cd, Bd);
  SPMM_VECTOR_SHAPES(X, 4, SPMM_BAL_CHUNKS)
  SPMM_SCALAR_SHAPES(X)
  X(4, 32, 2) X(4, 32, 4)  // one tile for wide rows
#undef X
  return cudaErrorInvalidConfiguration;
}

cudaError_t launch_fusedmm_row_f32(const Launch& L, int G, const float* Cd, const float* Bd) {
  switch (G) {
    case 4: return launch_fusedmm_row_t<4>(L, Cd, Bd);
    case 8: return launch_fusedmm_row_t<8>(L, Cd, Bd);
    case 16: return launch_fusedmm_row_t<16>(L, Cd, Bd);
    case 32: return launch_fusedmm_row_t<32>(L, Cd, Bd);
    default: return cudaErrorInvalidConfiguration;
  }
}

}  // namespace spmm
