// Balanced-kernel instantiations for semiring code 3 (fp32 B).
#include "spmm_balanced.cuh"

namespace spmm {

cudaError_t launch_semiring_f32_sr3(const Launch& L, Shape s) {
#define X(V, GG, NC) \
  if (s.vec == V && s.G == GG && s.nch == NC) return launch_balanced_t<float, V, GG, NC, false, 3>(L);
  SPMM_VECTOR_SHAPES(X, 4, SPMM_BAL_CHUNKS)
  SPMM_SCALAR_SHAPES(X)
#undef X
  return cudaErrorInvalidConfiguration;
}

}  // namespace spmm
