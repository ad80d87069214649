// Row-group kernel for narrow B (N <= 8): R lanes share one row.
//
// The Sgap page ("Sgap: Towards Efficient Sparse Tensor Algebra Compilation
// for GPU", atomic parallelism, Figs. 7-8, Table 1) studies SpMM with few
// dense columns, where the work is bound by balance rather than by the dense
// accesses, and names the point {<1/g row, c col>, r}: g threads share a row,
// each owns c columns, and r threads synchronise in the reduction; its Table 1
// finds r = 4 or 8 faster than the fixed r = 32.  Here a whole output row fits
// one lane (VEC * NCH >= N columns), so a group of R lanes takes one row:
// lane l takes the row's nonzeros l, l + R, l + 2R, ... (the group's colind
// and vals loads are coalesced), keeps U gathers in flight, and accumulates
// all N columns; at the row end log2(R) shuffle levels sum the R partial rows
// and the group's first lane stores the row.  R is chosen by the plan from the
// mean row length (and can be set); the summation order is fixed.
#pragma once

#include "spmm_device.cuh"
#include "spmm_internal.h"

#ifndef SPMM_RG_LOADS
#define SPMM_RG_LOADS 4  // nonzeros a lane has in flight
#endif

namespace spmm {

// VEC * NCH columns per lane; VEC == 1 serves any N <= NCH with column guards.
template <typename BT, int VEC, int NCH, int R>
__global__ void __launch_bounds__(kThreads)
    spmm_rowgroup_kernel(int32_t M, int32_t N, const int32_t* __restrict__ rowptr,
                         const int32_t* __restrict__ colind, const float* __restrict__ vals,
                         const BT* __restrict__ B, float* __restrict__ C) {
  constexpr int kRowsPerCta = kThreads / R;
  constexpr int U = SPMM_RG_LOADS;
  const int gl = threadIdx.x & (R - 1);
  const int64_t row = int64_t(blockIdx.x) * kRowsPerCta + threadIdx.x / R;
  const bool live = row < M;  // groups past M still take part in the shuffles
  const uint64_t stream_pol = policy_evict_first();
  const int start = live ? ld_stream(rowptr + row, stream_pol) : 0;
  const int end = live ? ld_stream(rowptr + row + 1, stream_pol) : 0;

  // column offsets of the lane's chunks, clamped into the row for loads
  int coff[NCH];
#pragma unroll
  for (int ch = 0; ch < NCH; ++ch) coff[ch] = min(ch * VEC, N - VEC);
  FVec<VEC> acc[NCH];
#pragma unroll
  for (int ch = 0; ch < NCH; ++ch) acc[ch].zero();

  for (int base = start; base < end; base += R * U) {
    BSlice<BT, VEC> bs[U][NCH];
    float v[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {  // past the row: the row's first nonzero again, value 0
      const int idx = base + u * R + gl;
      const bool ok = idx < end;
      const int k = ok ? idx : start;
      const int c = ld_stream(colind + k, stream_pol);
      const float x = ld_stream(vals + k, stream_pol);
      v[u] = ok ? x : 0.f;
      const BT* brow = B + size_t(c) * N;
#pragma unroll
      for (int ch = 0; ch < NCH; ++ch) bs[u][ch].load(brow + coff[ch]);
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const float2 vv = pair(v[u]);
#pragma unroll
      for (int ch = 0; ch < NCH; ++ch) {
        FVec<VEC> b;
        bs[u][ch].widen(b);
        acc[ch].fma(vv, b);
      }
    }
  }
  // the group's R partial rows (every lane of the warp takes part)
#pragma unroll
  for (int o = R / 2; o > 0; o >>= 1)
#pragma unroll
    for (int ch = 0; ch < NCH; ++ch) acc[ch].add_shfl_xor(o);
  if (live && gl == 0) {
    float* crow = C + size_t(row) * N;
    if constexpr (VEC == 1) {
#pragma unroll
      for (int ch = 0; ch < NCH; ++ch)
        if (ch < N) st_stream1(crow + ch, acc[ch].x);
    } else {
#pragma unroll
      for (int ch = 0; ch < NCH; ++ch) store_c<VEC>(crow + ch * VEC, acc[ch]);
    }
  }
}

template <typename BT, int VEC, int NCH, int R>
cudaError_t launch_rowgroup_t(const Launch& L) {
  constexpr int kRowsPerCta = kThreads / R;
  const unsigned grid = unsigned((int64_t(L.M) + kRowsPerCta - 1) / kRowsPerCta);
  SPMM_DEBUG_RANGES(L.stream, L.err, {{L.B, size_t(L.K) * L.N * sizeof(BT)}}, {{L.C, size_t(L.M) * L.N * 4}});
  spmm_rowgroup_kernel<BT, VEC, NCH, R><<<grid, kThreads, 0, L.stream>>>(
      L.M, L.N, L.rowptr, L.colind, L.vals, static_cast<const BT*>(L.B), L.C);
  return cudaGetLastError();
}

}  // namespace spmm
