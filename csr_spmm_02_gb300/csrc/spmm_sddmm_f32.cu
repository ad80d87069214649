// Instantiations of the SDDMM kernel (fp32).
#include "spmm_sddmm.cuh"

namespace spmm {

cudaError_t launch_sddmm_f32(const Launch& L, Shape s, const float* Cd, float* out) {
#define X(V, GG, NC) \
  if (s.vec == V && s.G == GG && s.nch == NC) return launch_sddmm_t<V, GG, NC>(L, Cd, out);
  SPMM_VECTOR_SHAPES(X, 4, SPMM_BAL_CHUNKS)
  SPMM_SCALAR_SHAPES(X)
  X(4, 32, 2) X(4, 32, 4)  // wide rows
#undef X
  return cudaErrorInvalidConfiguration;
}

}  // namespace spmm
