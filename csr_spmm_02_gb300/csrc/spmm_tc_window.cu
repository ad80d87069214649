// The tensor-core window kernel (bf16 B).
#include "spmm_tc_window.cuh"

namespace spmm {

cudaError_t launch_tc_window_bf16(const Launch& L) { return launch_tc_window(L); }

}  // namespace spmm
