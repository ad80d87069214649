// Instantiations of the SDDMM kernels (fp32): merge-path ranges and row groups.
#include "spmm_sddmm.cuh"
#include "spmm_sddmm_row.cuh"

namespace spmm {

cudaError_t launch_sddmm_f32(const Launch& L, Shape s, const float* Cd, float* out) {
#define X(V, GG, NC) \
  if (s.vec == V && s.G == GG && s.nch == NC) return launch_sddmm_t<V, GG, NC>(L, Cd, out);
  SPMM_VECTOR_SHAPES(X, 4, SPMM_BAL_CHUNKS)
  SPMM_SCALAR_SHAPES(X)
  X(4, 32, 2) X(4, 32, 4)  // wide rows
  X(4, 4, 2) X(4, 8, 2) X(4, 8, 4)  // two or four chunks per lane at N = 32, 64, 128
#undef X
  return cudaErrorInvalidConfiguration;
}

cudaError_t launch_sddmm_row_f32(const Launch& L, int G, const float* Cd, float* out) {
  switch (G) {
    case 4: return launch_sddmm_row_t<4>(L, Cd, out);
    case 8: return launch_sddmm_row_t<8>(L, Cd, out);
    case 16: return launch_sddmm_row_t<16>(L, Cd, out);
    case 32: return launch_sddmm_row_t<32>(L, Cd, out);
    default: return cudaErrorInvalidConfiguration;
  }
}

}  // namespace spmm
