// Instantiations of the row kernel for f32 B.
#include "spmm_row.cuh"

namespace spmm {

cudaError_t launch_row_f32(const Launch& L, Shape s) {
#define X(V, GG, NC) \
  if (s.vec == V && s.G == GG && s.nch == NC) return launch_row_t<float, V, GG, NC>(L);
  X(4, 1, 1) X(4, 2, 1) X(4, 4, 1) X(4, 8, 1) X(4, 16, 1) X(4, 32, 1) X(4, 32, 2)
  X(1, 8, 1) X(1, 32, 1) X(4, 32, 4)
#undef X
  return cudaErrorInvalidConfiguration;
}

}  // namespace spmm
