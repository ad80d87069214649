// Instantiations of the window kernel: fp32 B (4-column lanes, 128-column
// tiles) and bf16 B (8-column lanes, 256-column tiles).
#include "spmm_window.cuh"

namespace spmm {

cudaError_t launch_window_f32(const Launch& L) { return launch_window_t<float, 4>(L); }
cudaError_t launch_window_bf16(const Launch& L) { return launch_window_t<uint16_t, 8>(L); }

}  // namespace spmm
