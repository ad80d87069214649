// Instantiations of the balanced kernel for bf16 B.
#include "spmm_balanced.cuh"

namespace spmm {

cudaError_t launch_balanced_bf16(const Launch& L, Shape s) {
#define X(V, GG, NC) \
  if (s.vec == V && s.G == GG && s.nch == NC) return launch_balanced_t<uint16_t, V, GG, NC>(L);
  SPMM_VECTOR_SHAPES(X, 8, SPMM_BAL_BF16_CHUNKS)
  SPMM_SCALAR_SHAPES(X)
#undef X
  return cudaErrorInvalidConfiguration;
}

}  // namespace spmm
