// Instantiations of the balanced kernel for bf16 B.
#include "spmm_balanced.cuh"

namespace spmm {

cudaError_t launch_balanced_bf16(const Launch& L, Shape s) {
#define X(V, GG, NC) \
  if (s.vec == V && s.G == GG && s.nch == NC) return launch_balanced_t<uint16_t, V, GG, NC>(L);
  X(8, 1, 1) X(8, 2, 1) X(8, 4, 1) X(8, 8, 1) X(8, 16, 1) X(8, 32, 1) X(8, 32, 2)
  X(1, 8, 1) X(1, 32, 1)
#undef X
  return cudaErrorInvalidConfiguration;
}

}  // namespace spmm
