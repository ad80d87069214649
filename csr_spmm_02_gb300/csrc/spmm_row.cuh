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
// A group stages a chunk of its row's (colind, vals) pairs in shared memory
// with coalesced loads; every lane then reads each pair with a broadcast
// shared load.  U gathers of B rows are issued before the FMAs that consume
// them; a short last batch is zero-extended (it re-reads a valid row and adds
// it with value 0, the zero extension the Sgap page describes), so the inner
// loop has no branches.  Each lane owns NCH 16-byte chunks, so the per-nonzero
// bookkeeping (shared loads, address arithmetic) is paid by few lanes for
// many columns.  The summation order is fixed, so results are deterministic.
#pragma once

#include <algorithm>

#include "spmm_device.cuh"
#include "spmm_internal.h"

#ifndef SPMM_ROW_LOADS
#define SPMM_ROW_LOADS 4  // 16-byte B loads in flight per lane (U nonzeros x NCH chunks)
#endif
#ifndef SPMM_ROW_MIN_BLOCKS
#define SPMM_ROW_MIN_BLOCKS 1
#endif

namespace spmm {

template <int G, int NCH>
struct RowTiling {
  static constexpr int kChunk = G > 16 ? G : 16;  // (col, val) pairs a group stages at a time
  static constexpr int kU0 = SPMM_ROW_LOADS / NCH > 0 ? SPMM_ROW_LOADS / NCH : 1;
  static constexpr int U = kU0 < kChunk ? kU0 : kChunk;  // nonzeros per batch; divides kChunk
};

// B-slice loads of the row kernel with an L2 policy: B rows get evict-last
// priority, since every B row is gathered again by other rows (the bytes
// loaded are those of BSlice::load).
__device__ __forceinline__ uint4 ld_b16_policy(const void* p, uint64_t pol) {
  uint4 v;
#ifdef SPMM_DEBUG_BOUNDS
  if (!debug_load_ok(p, 16)) return make_uint4(0u, 0u, 0u, 0u);
#endif
  asm volatile("ld.global.nc.L2::cache_hint.v4.u32 {%0,%1,%2,%3}, [%4], %5;"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p), "l"(pol));
  return v;
}
__device__ __forceinline__ void gather_keep(BSlice<float, 4>& s, const float* p, uint64_t pol) {
  const uint4 v = ld_b16_policy(p, pol);
  s.r = make_float4(__uint_as_float(v.x), __uint_as_float(v.y), __uint_as_float(v.z), __uint_as_float(v.w));
}
__device__ __forceinline__ void gather_keep(BSlice<uint16_t, 8>& s, const uint16_t* p, uint64_t pol) {
  s.r = ld_b16_policy(p, pol);
}
template <typename BT>
__device__ __forceinline__ void gather_keep(BSlice<BT, 1>& s, const BT* p, uint64_t) {  // scalar path
  s.load(p);
}

// The group's pairs for staging slots [base, base + CH) of a row ending at
// `end`: lane l holds slots base + l + G p (p < CH / G); slots past the end
// hold (0, 0).
template <int G, int PPL>
__device__ __forceinline__ void load_pairs(int2 (&pr)[PPL], const int32_t* __restrict__ colind,
                                           const float* __restrict__ vals, int base, int end, int lane,
                                           uint64_t pol) {
#pragma unroll
  for (int p = 0; p < PPL; ++p) {
    const int j = base + lane + G * p;
    pr[p] = j < end ? make_int2(ld_stream(colind + j, pol), ld_stream(reinterpret_cast<const int*>(vals) + j, pol))
                    : make_int2(0, 0);
  }
}

template <typename BT, int VEC, int G, int NCH>
__global__ void __launch_bounds__(kThreads, SPMM_ROW_MIN_BLOCKS)
    spmm_row_kernel(int32_t M, int32_t N, const int32_t* __restrict__ rowptr,
                    const int32_t* __restrict__ colind, const float* __restrict__ vals,
                    const BT* __restrict__ B, float* __restrict__ C) {
  constexpr int kGroups = kThreads / G;
  constexpr int CH = RowTiling<G, NCH>::kChunk;
  constexpr int U = RowTiling<G, NCH>::U;
  constexpr int PPL = CH / G;  // staged pairs per lane
  __shared__ int2 s_cv[kGroups * CH];  // group g stages (col, val bits) in s_cv[g*CH, g*CH+CH)

  const int lane = threadIdx.x & (G - 1);
  const int grp = threadIdx.x / G;
  // Persistent: group g of CTA b takes rows b*kGroups + g, then every
  // gridDim.x*kGroups rows further.  The next row's bounds and first pairs
  // are loaded while the current row's gathers run, so a row's chain is its
  // gathers alone.
  const int64_t stride = int64_t(gridDim.x) * kGroups;
  int64_t row = int64_t(blockIdx.x) * kGroups + grp;
  if (row >= M) return;  // the whole group leaves together
  const unsigned gmask = G == 32 ? 0xffffffffu : (((1u << G) - 1u) << ((threadIdx.x & 31) & ~(G - 1)));
  int2* cv = s_cv + grp * CH;

  // Columns of this lane: NCH chunks of VEC, chunk ch at col0 + (ch*G + lane)*VEC.
  // Loads use offsets clamped into the row (a lane past N re-reads a valid
  // slice it never stores), so the inner loop needs no column predicate.
  const int col0 = blockIdx.y * (G * VEC * NCH);
  int coff[NCH];
  const BT* bl[NCH];  // this lane's slice of B row 0; row c is bl[ch] + c*N
#pragma unroll
  for (int ch = 0; ch < NCH; ++ch) {
    coff[ch] = col0 + (ch * G + lane) * VEC;
    bl[ch] = B + min(coff[ch], N - VEC);
  }

  const uint64_t stream_pol = policy_evict_first();
  const uint64_t keep_pol = policy_evict_last();  // B rows: reused by many rows
  int start = ld_stream(rowptr + row, stream_pol);
  int end = ld_stream(rowptr + row + 1, stream_pol);
  int2 pr[PPL];
  load_pairs<G, PPL>(pr, colind, vals, start, end, lane, stream_pol);
  for (; row < M; row += stride) {
    const int64_t nrow = row + stride;
    int nstart = 0, nend = 0;
    if (nrow < M) {
      nstart = ld_stream(rowptr + nrow, stream_pol);
      nend = ld_stream(rowptr + nrow + 1, stream_pol);
    }
    FVec<VEC> acc[NCH];
#pragma unroll
    for (int ch = 0; ch < NCH; ++ch) acc[ch].zero();
    for (int base = start; base < end; base += CH) {
      const int cnt = min(CH, end - base);
      __syncwarp(gmask);  // every lane has finished with the previous chunk
#pragma unroll
      for (int p = 0; p < PPL; ++p) cv[lane + G * p] = pr[p];
      __syncwarp(gmask);
      // the pairs of the next chunk, or of the next row's first chunk
      if (base + CH < end) load_pairs<G, PPL>(pr, colind, vals, base + CH, end, lane, stream_pol);
      else load_pairs<G, PPL>(pr, colind, vals, nstart, nend, lane, stream_pol);
      int t = 0;
      for (; t + U <= cnt; t += U) {  // full batches: gathers first, then the FMAs
        BSlice<BT, VEC> bs[U][NCH];
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const size_t roff = size_t(cv[t + u].x) * N;
#pragma unroll
          for (int ch = 0; ch < NCH; ++ch) gather_keep(bs[u][ch], bl[ch] + roff, keep_pol);
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const float2 vv = pair(__int_as_float(cv[t + u].y));  // re-read: frees registers
#pragma unroll
          for (int ch = 0; ch < NCH; ++ch) {
            FVec<VEC> b;
            bs[u][ch].widen(b);
            acc[ch].fma(vv, b);
          }
        }
      }
      if (t < cnt) {  // short last batch: padded slots re-read the last row with value 0
        BSlice<BT, VEC> bs[U][NCH];
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const size_t roff = size_t(cv[min(t + u, cnt - 1)].x) * N;
#pragma unroll
          for (int ch = 0; ch < NCH; ++ch) gather_keep(bs[u][ch], bl[ch] + roff, keep_pol);
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const float2 vv = pair(t + u < cnt ? __int_as_float(cv[t + u].y) : 0.f);
#pragma unroll
          for (int ch = 0; ch < NCH; ++ch) {
            FVec<VEC> b;
            bs[u][ch].widen(b);
            acc[ch].fma(vv, b);
          }
        }
      }
    }
    if (start == end) load_pairs<G, PPL>(pr, colind, vals, nstart, nend, lane, stream_pol);  // empty row
    float* crow = C + size_t(row) * N;
#pragma unroll
    for (int ch = 0; ch < NCH; ++ch)
      if (coff[ch] < N) store_c<VEC>(crow + coff[ch], acc[ch]);
    start = nstart;
    end = nend;
  }
}

// Resident CTAs per SM of one instantiation, looked up once per device.
template <typename BT, int VEC, int G, int NCH>
int row_blocks_per_sm(int dev) {
  static int cached[kMaxDevices] = {};
  if (dev < 0 || dev >= kMaxDevices) return 1;
  if (!cached[dev]) {
    int per_sm = 0, sms = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, spmm_row_kernel<BT, VEC, G, NCH>, kThreads, 0) !=
            cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return 1;
    cached[dev] = std::max(1, per_sm) * std::max(1, sms);
  }
  return cached[dev];
}

template <typename BT, int VEC, int G, int NCH>
cudaError_t launch_row_t(const Launch& L) {
  constexpr int kGroups = kThreads / G;
  constexpr int TW = G * VEC * NCH;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned tiles = unsigned((L.N + TW - 1) / TW);
  // one wave of resident CTAs over all column tiles
  const int64_t need = (int64_t(L.M) + kGroups - 1) / kGroups;
  const int64_t wave = std::max<int64_t>(1, row_blocks_per_sm<BT, VEC, G, NCH>(dev) / int64_t(tiles));
  const dim3 grid(unsigned(std::min(need, wave)), tiles);
  SPMM_DEBUG_RANGES(L.stream, L.err, {{L.B, size_t(L.K) * L.N * sizeof(BT)}}, {{L.C, size_t(L.M) * L.N * 4}});
  spmm_row_kernel<BT, VEC, G, NCH><<<grid, kThreads, 0, L.stream>>>(
      L.M, L.N, L.rowptr, L.colind, L.vals, static_cast<const BT*>(L.B), L.C);
  return cudaGetLastError();
}

}  // namespace spmm
