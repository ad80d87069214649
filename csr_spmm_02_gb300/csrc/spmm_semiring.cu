// Semiring dispatch: one translation unit per semiring code keeps the build parallel.
#include "spmm_internal.h"

namespace spmm {

cudaError_t launch_semiring_f32_sr1(const Launch& L, Shape s);
cudaError_t launch_semiring_f32_sr2(const Launch& L, Shape s);
cudaError_t launch_semiring_f32_sr3(const Launch& L, Shape s);
cudaError_t launch_semiring_f32_sr4(const Launch& L, Shape s);
cudaError_t launch_semiring_f32_sr5(const Launch& L, Shape s);

cudaError_t launch_semiring_f32(const Launch& L, Shape s, int sr) {
  switch (sr) {
    case 1: return launch_semiring_f32_sr1(L, s);
    case 2: return launch_semiring_f32_sr2(L, s);
    case 3: return launch_semiring_f32_sr3(L, s);
    case 4: return launch_semiring_f32_sr4(L, s);
    case 5: return launch_semiring_f32_sr5(L, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace spmm
