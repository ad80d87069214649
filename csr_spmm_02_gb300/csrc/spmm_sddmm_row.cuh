// SDDMM and FusedMM for short, even rows: one group of G lanes per row,
// persistent.
//
// The SDDMM section of "Performance Optimization of Deep Learning Sparse
// Matrix Kernels on Intel Max Series GPU" (Algorithm 1, Figs. 3-4) keeps the
// row C_i in registers and produces each nonzero of the row as a dot product
// with the B row it selects.  Here a group of G lanes (4 columns each, N <=
// 4G) does that for one row at a time: the C row is loaded once per row, each
// nonzero costs one 16-byte B gather per lane, and every G consecutive
// nonzeros are summed over the group by a transposed butterfly (G-1 shuffles
// for G results) after which lane l holds nonzero l's value and the group
// stores them with one coalesced store.  Groups walk rows with the stride of
// all groups in the grid and load the next row's bounds and first column
// indices while the current row's gathers run (the row SpMM kernel's scheme).
// The summation order is fixed, so results are deterministic.
#pragma once

#include <algorithm>

#include "spmm_device.cuh"
#include "spmm_internal.h"
#include "spmm_sddmm.cuh"

namespace spmm {

// group_reduce_transposed restricted to the G lanes of `gmask` (groups of a
// warp may be on different rows, so the full-warp form cannot be used).
template <int G>
__device__ __forceinline__ float group_reduce_transposed_masked(float (&v)[G], int gl, unsigned gmask) {
#pragma unroll
  for (int o = G / 2; o >= 1; o >>= 1) {
    const bool upper = (gl & o) != 0;
#pragma unroll
    for (int i = 0; i < o; ++i) {
      const float send = upper ? v[i] : v[i + o];
      const float keep = upper ? v[i + o] : v[i];
      v[i] = keep + __shfl_xor_sync(gmask, send, o, G);
    }
  }
  return v[0];
}

template <int G>
__global__ void __launch_bounds__(kThreads)
    spmm_sddmm_row_kernel(int32_t M, int32_t N, const int32_t* __restrict__ rowptr,
                          const int32_t* __restrict__ colind, const float* __restrict__ Cd,
                          const float* __restrict__ B, float* __restrict__ out) {
  constexpr int VEC = 4;
  constexpr int kGroups = kThreads / G;
  constexpr int U = 4;  // B gathers in flight per lane
  __shared__ int s_c[kGroups * G];  // group g's block of G column indices

  const int lane = threadIdx.x & (G - 1);
  const int grp = threadIdx.x / G;
  const int64_t stride = int64_t(gridDim.x) * kGroups;
  int64_t row = int64_t(blockIdx.x) * kGroups + grp;
  if (row >= M) return;  // the whole group leaves together
  const unsigned gmask = G == 32 ? 0xffffffffu : (((1u << G) - 1u) << ((threadIdx.x & 31) & ~(G - 1)));
  int* cb = s_c + grp * G;

  const int coff = lane * VEC;
  const bool valid = coff < N;
  const int cl = min(coff, N - VEC);  // lanes past N read a valid slice and add nothing
  const float* bl = B + cl;
  const uint64_t stream_pol = policy_evict_first();

  int start = ld_stream(rowptr + row, stream_pol);
  int end = ld_stream(rowptr + row + 1, stream_pol);
  int pc = start + lane < end ? ld_stream(colind + start + lane, stream_pol) : 0;
  for (; row < M; row += stride) {
    const int64_t nrow = row + stride;
    int nstart = 0, nend = 0;
    if (nrow < M) {
      nstart = ld_stream(rowptr + nrow, stream_pol);
      nend = ld_stream(rowptr + nrow + 1, stream_pol);
    }
    FVec<VEC> c;
    if (end > start) {
      BSlice<float, VEC> cs;
      cs.load(Cd + size_t(row) * N + cl);
      cs.widen(c);
    }
    for (int base = start; base < end; base += G) {  // rounds of G nonzeros
      const int cnt = min(G, end - base);
      __syncwarp(gmask);  // the group has finished with the previous block
      cb[lane] = pc;
      __syncwarp(gmask);
      // the next block's columns, or the next row's first block
      if (base + G < end) pc = base + G + lane < end ? ld_stream(colind + base + G + lane, stream_pol) : 0;
      else pc = nstart + lane < nend ? ld_stream(colind + nstart + lane, stream_pol) : 0;
      float d[G];
#pragma unroll
      for (int t0 = 0; t0 < G; t0 += U) {
        BSlice<float, VEC> bs[U];
#pragma unroll
        for (int u = 0; u < U; ++u) bs[u].load(bl + size_t(cb[min(t0 + u, cnt - 1)]) * N);
#pragma unroll
        for (int u = 0; u < U; ++u) {
          FVec<VEC> b;
          bs[u].widen(b);
          float2 t = __fmul2_rn(c.p[0], b.p[0]);
          t = __ffma2_rn(c.p[1], b.p[1], t);
          d[t0 + u] = valid ? t.x + t.y : 0.f;
        }
      }
      const float x = group_reduce_transposed_masked<G>(d, lane, gmask);
      // plain store: a group writes 64 bytes of a 128-byte line per round, and
      // both halves must meet in L2 (an evict-first store let half-written
      // lines reach DRAM, about 17x the output's bytes)
#ifdef SPMM_DEBUG_BOUNDS
      if (lane < cnt) st_plain1(out + base + lane, x);
#else
      // written out rather than through st_plain1: with the helper the
      // compiler schedules this loop differently and uniform64k (N = 64)
      // takes 48 instead of 40 us
      if (lane < cnt) out[base + lane] = x;
#endif
    }
    if (start == end) pc = nstart + lane < nend ? ld_stream(colind + nstart + lane, stream_pol) : 0;
    start = nstart;
    end = nend;
  }
}

template <int G>
int sddmm_row_blocks(int dev) {
  static int cached[kMaxDevices] = {};
  if (dev < 0 || dev >= kMaxDevices) return 1;
  if (!cached[dev]) {
    int per_sm = 0, sms = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, spmm_sddmm_row_kernel<G>, kThreads, 0) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return 1;
    cached[dev] = std::max(1, per_sm) * std::max(1, sms);
  }
  return cached[dev];
}

template <int G>
cudaError_t launch_sddmm_row_t(const Launch& L, const float* Cd, float* out) {
  constexpr int kGroups = kThreads / G;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const int64_t need = (int64_t(L.M) + kGroups - 1) / kGroups;
  const unsigned grid = unsigned(std::min<int64_t>(need, sddmm_row_blocks<G>(dev)));
  SPMM_DEBUG_RANGES(L.stream, L.err, {{L.B, size_t(L.K) * L.N * 4}, {Cd, size_t(L.M) * L.N * 4}},
                    {{out, size_t(L.nnz) * 4}});
  spmm_sddmm_row_kernel<G><<<grid, kThreads, 0, L.stream>>>(L.M, L.N, L.rowptr, L.colind, Cd,
                                                            static_cast<const float*>(L.B), out);
  return cudaGetLastError();
}

}  // namespace spmm

namespace spmm {

// FusedMM for short, even rows (the FusedMM section of the same page, Fig. 6,
// Algorithm 3): E_i = sum_j (C_i . B_j) D_j with one group of G lanes per
// row, persistent as above.  A round of G nonzeros first gathers their B rows
// for the dot products (C_i in registers), sums them over the group with the
// transposed butterfly, then gathers their D rows and accumulates each with
// its value, handed from lane t by a group shuffle.  E_i stays in registers
// and is stored once; the values never reach memory.
template <int G>
__global__ void __launch_bounds__(kThreads)
    spmm_fusedmm_row_kernel(int32_t M, int32_t N, const int32_t* __restrict__ rowptr,
                            const int32_t* __restrict__ colind, const float* __restrict__ Cd,
                            const float* __restrict__ B, const float* __restrict__ D, float* __restrict__ E) {
  constexpr int VEC = 4;
  constexpr int kGroups = kThreads / G;
  constexpr int U = 4;  // gathers in flight per lane
  __shared__ int s_c[kGroups * G];

  const int lane = threadIdx.x & (G - 1);
  const int grp = threadIdx.x / G;
  const int64_t stride = int64_t(gridDim.x) * kGroups;
  int64_t row = int64_t(blockIdx.x) * kGroups + grp;
  if (row >= M) return;
  const unsigned gmask = G == 32 ? 0xffffffffu : (((1u << G) - 1u) << ((threadIdx.x & 31) & ~(G - 1)));
  int* cb = s_c + grp * G;

  const int coff = lane * VEC;
  const bool valid = coff < N;
  const int cl = min(coff, N - VEC);
  const uint64_t stream_pol = policy_evict_first();

  int start = ld_stream(rowptr + row, stream_pol);
  int end = ld_stream(rowptr + row + 1, stream_pol);
  int pc = start + lane < end ? ld_stream(colind + start + lane, stream_pol) : 0;
  for (; row < M; row += stride) {
    const int64_t nrow = row + stride;
    int nstart = 0, nend = 0;
    if (nrow < M) {
      nstart = ld_stream(rowptr + nrow, stream_pol);
      nend = ld_stream(rowptr + nrow + 1, stream_pol);
    }
    FVec<VEC> c, acc;
    acc.zero();
    if (end > start) {
      BSlice<float, VEC> cs;
      cs.load(Cd + size_t(row) * N + cl);
      cs.widen(c);
    }
    for (int base = start; base < end; base += G) {
      const int cnt = min(G, end - base);
      __syncwarp(gmask);
      cb[lane] = pc;
      __syncwarp(gmask);
      if (base + G < end) pc = base + G + lane < end ? ld_stream(colind + base + G + lane, stream_pol) : 0;
      else pc = nstart + lane < nend ? ld_stream(colind + nstart + lane, stream_pol) : 0;
      float d[G];
#pragma unroll
      for (int t0 = 0; t0 < G; t0 += U) {  // dot products with the round's B rows
        BSlice<float, VEC> bs[U];
#pragma unroll
        for (int u = 0; u < U; ++u) bs[u].load(B + size_t(cb[min(t0 + u, cnt - 1)]) * N + cl);
#pragma unroll
        for (int u = 0; u < U; ++u) {
          FVec<VEC> b;
          bs[u].widen(b);
          float2 t = __fmul2_rn(c.p[0], b.p[0]);
          t = __ffma2_rn(c.p[1], b.p[1], t);
          d[t0 + u] = valid ? t.x + t.y : 0.f;
        }
      }
      const float x = group_reduce_transposed_masked<G>(d, lane, gmask);  // lane t: value of nonzero t
#pragma unroll
      for (int t0 = 0; t0 < G; t0 += U) {  // accumulate the round's D rows
        if (t0 >= cnt) break;
        BSlice<float, VEC> ds[U];
#pragma unroll
        for (int u = 0; u < U; ++u) ds[u].load(D + size_t(cb[min(t0 + u, cnt - 1)]) * N + cl);
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const float v = __shfl_sync(gmask, x, t0 + u, G);
          FVec<VEC> dv;
          ds[u].widen(dv);
          acc.fma(pair(t0 + u < cnt ? v : 0.f), dv);
        }
      }
    }
    if (start == end) pc = nstart + lane < nend ? ld_stream(colind + nstart + lane, stream_pol) : 0;
    if (valid) store_c<VEC>(E + size_t(row) * N + coff, acc);
    start = nstart;
    end = nend;
  }
}

template <int G>
int fusedmm_row_blocks(int dev) {
  static int cached[kMaxDevices] = {};
  if (dev < 0 || dev >= kMaxDevices) return 1;
  if (!cached[dev]) {
    int per_sm = 0, sms = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, spmm_fusedmm_row_kernel<G>, kThreads, 0) !=
            cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return 1;
    cached[dev] = std::max(1, per_sm) * std::max(1, sms);
  }
  return cached[dev];
}

template <int G>
cudaError_t launch_fusedmm_row_t(const Launch& L, const float* Cd, const float* Bd) {
  constexpr int kGroups = kThreads / G;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const int64_t need = (int64_t(L.M) + kGroups - 1) / kGroups;
  const unsigned grid = unsigned(std::min<int64_t>(need, fusedmm_row_blocks<G>(dev)));
  SPMM_DEBUG_RANGES(L.stream, L.err,
                    {{L.B, size_t(L.K) * L.N * 4}, {Cd, size_t(L.M) * L.N * 4}, {Bd, size_t(L.K) * L.N * 4}},
                    {{L.C, size_t(L.M) * L.N * 4}});
  spmm_fusedmm_row_kernel<G><<<grid, kThreads, 0, L.stream>>>(L.M, L.N, L.rowptr, L.colind, Cd, Bd,
                                                              static_cast<const float*>(L.B), L.C);
  return cudaGetLastError();
}

}  // namespace spmm
