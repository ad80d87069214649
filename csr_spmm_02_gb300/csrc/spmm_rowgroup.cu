// Instantiations of the row-group kernel (N <= 8): 4 or 8 fp32 columns as
// 16-byte vectors, 8 bf16 columns as one vector, else up to 8 scalar columns;
// r = 2 .. 32 lanes per row.
#include "spmm_rowgroup.cuh"

namespace spmm {

namespace {

template <typename BT, int VEC, int NCH>
cudaError_t by_lanes(const Launch& L, int lanes) {
  switch (lanes) {
    case 2: return launch_rowgroup_t<BT, VEC, NCH, 2>(L);
    case 4: return launch_rowgroup_t<BT, VEC, NCH, 4>(L);
    case 8: return launch_rowgroup_t<BT, VEC, NCH, 8>(L);
    case 16: return launch_rowgroup_t<BT, VEC, NCH, 16>(L);
    case 32: return launch_rowgroup_t<BT, VEC, NCH, 32>(L);
    default: return cudaErrorInvalidValue;
  }
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

}  // namespace

cudaError_t launch_rowgroup_f32(const Launch& L, int lanes) {
  const bool vec = aligned16(L.B) && aligned16(L.C);
  if (vec && L.N == 4) return by_lanes<float, 4, 1>(L, lanes);
  if (vec && L.N == 8) return by_lanes<float, 4, 2>(L, lanes);
  return by_lanes<float, 1, 8>(L, lanes);
}

cudaError_t launch_rowgroup_bf16(const Launch& L, int lanes) {
  if (aligned16(L.B) && aligned16(L.C) && L.N == 8) return by_lanes<uint16_t, 8, 1>(L, lanes);
  return by_lanes<uint16_t, 1, 8>(L, lanes);
}

}  // namespace spmm
