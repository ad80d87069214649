// Row kernel: one group of G lanes per row of A (G a power of two <= 32).
//
// The SPMM section of "Performance Optimization of Deep Learning Sparse
// Matrix Kernels on Intel Max Series GPU" (Figs. 9-10) gives each output row
// to one work-item that stages a chunk of the row's column indices and values,
// gathers the B row of every nonzero and accumulates the output row in
// registers before storing it once.  On sm_103a the work-item becomes a group
// of G lanes that together hold the row's N outputs (the sub-warp-per-row
// mapping the kkmem page describes for GPUs, and Sgap's {<1/g row, c col>, r}
// point): each lane owns NCH chunks of VEC consecutive columns, so every B
// gather is one 16-byte load per lane, coalesced across the group.
//
// Per chunk of G nonzeros the group loads G (colind, vals) pairs with one
// coalesced load per lane and broadcasts them with warp shuffles; U B-row
// gathers are issued before the FMAs that consume them, so each lane keeps U
// 16-byte loads in flight.  Rows are summed in index order by one group, so
// results are deterministic.  C rows are stored once with streaming stores.
#pragma once

#include "spmm_device.cuh"
#include "spmm_internal.h"

namespace spmm {

template <int G, int NCH>
struct RowUnroll {
  static constexpr int kBase = NCH >= 4 ? 2 : (NCH == 2 ? 4 : 8);
  static constexpr int value = kBase < G ? kBase : G;
};

template <typename BT, int VEC, int G, int NCH>
__global__ void __launch_bounds__(kThreads)
    spmm_row_kernel(int32_t M, int32_t N, const int32_t* __restrict__ rowptr,
                    const int32_t* __restrict__ colind, const float* __restrict__ vals,
                    const BT* __restrict__ B, float* __restrict__ C) {
  constexpr int kGroups = kThreads / G;
  constexpr int U = RowUnroll<G, NCH>::value;
  const int lane = threadIdx.x & (G - 1);
  const int64_t row = int64_t(blockIdx.x) * kGroups + threadIdx.x / G;
  if (row >= M) return;  // the whole group leaves together
  const unsigned gmask = G == 32 ? 0xffffffffu : (((1u << G) - 1u) << ((threadIdx.x & 31) & ~(G - 1)));

  const int col0 = blockIdx.y * (G * VEC * NCH);
  int coff[NCH];
  bool cok[NCH];
#pragma unroll
  for (int ch = 0; ch < NCH; ++ch) {
    coff[ch] = col0 + (ch * G + lane) * VEC;
    cok[ch] = coff[ch] < N;
  }
  float acc[NCH][VEC];
#pragma unroll
  for (int ch = 0; ch < NCH; ++ch)
#pragma unroll
    for (int j = 0; j < VEC; ++j) acc[ch][j] = 0.f;

  const int start = __ldg(rowptr + row);
  const int end = __ldg(rowptr + row + 1);
  for (int base = start; base < end; base += G) {
    const int cnt = min(G, end - base);
    int my_c = 0;
    float my_v = 0.f;
    if (lane < cnt) {
      my_c = __ldg(colind + base + lane);
      my_v = __ldg(vals + base + lane);
    }
    for (int t = 0; t < cnt; t += U) {
      BSlice<BT, VEC> bs[U][NCH];
      float v[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int src = (t + u) & (G - 1);
        const int c = __shfl_sync(gmask, my_c, src, G);
        v[u] = __shfl_sync(gmask, my_v, src, G);
        if (t + u < cnt) {
          const BT* brow = B + size_t(c) * N;
#pragma unroll
          for (int ch = 0; ch < NCH; ++ch)
            if (cok[ch]) bs[u][ch].load(brow + coff[ch]);
        }
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        if (t + u < cnt) {
#pragma unroll
          for (int ch = 0; ch < NCH; ++ch) {
            if (cok[ch]) {
              float b[VEC];
              bs[u][ch].widen(b);
              axpy<VEC>(acc[ch], v[u], b);
            }
          }
        }
      }
    }
  }
  float* crow = C + size_t(row) * N;
#pragma unroll
  for (int ch = 0; ch < NCH; ++ch)
    if (cok[ch]) store_c<VEC>(crow + coff[ch], acc[ch]);
}

template <typename BT, int VEC, int G, int NCH>
cudaError_t launch_row_t(const Launch& L) {
  constexpr int kGroups = kThreads / G;
  constexpr int TW = G * VEC * NCH;
  const dim3 grid(unsigned((int64_t(L.M) + kGroups - 1) / kGroups), unsigned((L.N + TW - 1) / TW));
  spmm_row_kernel<BT, VEC, G, NCH><<<grid, kThreads, 0, L.stream>>>(
      L.M, L.N, L.rowptr, L.colind, L.vals, static_cast<const BT*>(L.B), L.C);
  return cudaGetLastError();
}

}  // namespace spmm
