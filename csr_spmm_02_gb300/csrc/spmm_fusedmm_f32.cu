// Instantiations of the balanced kernel in FusedMM mode (fp32).
#include "spmm_balanced.cuh"

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

}  // namespace spmm
