// Window kernel: B rows staged once per CTA and reused from registers across
// rows, for matrices whose consecutive rows touch a narrow range of columns
// (banded, block-diagonal, mesh-like); any other CTA falls back to gathers.
//
// The [Intel Max] SPMM kernel (Figs. 9-10) and the row kernel read the B row
// of every nonzero again, from L2 on this GPU: for a band of 63 nonzeros per
// row and N = 256 that is 8.6 GB of L2->SM traffic for 0.54 GB of compulsory
// bytes, and the L2 gather rate (about 20 TB/s here) sets the time.  Here a
// CTA takes R = 8 * RW consecutive rows and, after staging their colind/vals
// (bulk copy into shared memory), finds the span [cmin, cmax] of columns they
// touch.  If the span's B rows fit the shared-memory window budget:
//
//  1. the window B[cmin..cmax][tile] is copied into shared memory with 16-byte
//     cp.async copies (each B row once per CTA instead of once per nonzero);
//  2. warp w owns RW consecutive rows and scatters their values into its own
//     dense tile A_w[j - cmin][r] (zeros elsewhere, RW values per column
//     contiguous): lane-parallel when a row's columns strictly increase (one
//     warp vote), else lane 0 adds the row's values in CSR order, so duplicate
//     columns are summed deterministically; only the warp itself reads it;
//  3. the warp walks the columns j its rows touch and, per column, reads the
//     lane's B slice once and the RW values once (one broadcast load) and
//     issues RW packed FMAs into RW accumulators: every B slice is reused RW
//     times from registers.
//
// The walk multiplies the explicit zeros of A_w too (for a band of width 63 and
// RW = 4 rows, 4 x 63 useful of 4 x 67 products), so a non-finite B value in a
// column inside the window but outside a row's pattern reaches that row
// (0 * inf = NaN); IEEE special values are outside the accepted inputs.
//
// Otherwise (the span does not fit, or the rows hold more nonzeros than the
// staging area) each warp computes its rows one by one with gathers, as the
// row kernel with one warp per row does.  The summation order of a row is
// fixed either way, so results are deterministic.
#pragma once

#include <climits>

#include "spmm_device.cuh"
#include "spmm_internal.h"

#ifndef SPMM_WIN_RW
#define SPMM_WIN_RW 4  // rows per warp (accumulator sets per lane)
#endif
#ifndef SPMM_WIN_B_BYTES
#define SPMM_WIN_B_BYTES (64 * 1024)  // shared-memory budget of the B window
#endif
#ifndef SPMM_WIN_STAGE
#define SPMM_WIN_STAGE 2048  // nonzeros a CTA can stage (larger CTAs use the gather path)
#endif

namespace spmm {

constexpr int kWinWarps = kThreads / 32;

template <typename BT, int TW>
struct WindowGeometry {
  static constexpr int R = kWinWarps * SPMM_WIN_RW;           // rows per CTA
  static constexpr int kRowBytes = TW * int(sizeof(BT));      // one B row of the tile
  static constexpr int kMaxSpan = SPMM_WIN_B_BYTES / kRowBytes;  // B rows the window holds
  static constexpr int kStage = SPMM_WIN_STAGE;
  static constexpr size_t smem_bytes() {
    return size_t(2) * (kStage + 8) * 4       // colind, vals
           + size_t(R + 8) * 4                // rowptr slice
           + size_t(kMaxSpan) * R * 4         // dense value tiles, one per warp
           + size_t(kMaxSpan) * kRowBytes     // B window
           + 64;                              // mbarrier, reductions
  }
};

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
#ifdef SPMM_DEBUG_BOUNDS
  if (!debug_load_ok(src, 16)) return;
#endif
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

template <typename BT, int VEC>
__global__ void __launch_bounds__(kThreads)
    spmm_window_kernel(int32_t M, int32_t N, const int32_t* __restrict__ rowptr,
                       const int32_t* __restrict__ colind, const float* __restrict__ vals,
                       const BT* __restrict__ B, float* __restrict__ C, int* __restrict__ err) {
  constexpr int G = 32, RW = SPMM_WIN_RW;
  constexpr int TW = G * VEC;
  using Geo = WindowGeometry<BT, TW>;
  constexpr int R = Geo::R;
  constexpr int kSpan = Geo::kMaxSpan;
  constexpr int kStage = Geo::kStage;
  static_assert(RW == 4 || RW == 8, "the value tile is read 4 rows at a time");

  extern __shared__ __align__(16) unsigned char smem[];
  int* s_col = reinterpret_cast<int*>(smem);
  float* s_val = reinterpret_cast<float*>(s_col + kStage + 8);
  int* s_rp = reinterpret_cast<int*>(s_val + kStage + 8);
  float* s_A = reinterpret_cast<float*>(s_rp + R + 8);                  // [warp][kSpan][RW]
  unsigned char* s_B = reinterpret_cast<unsigned char*>(s_A + kSpan * R);  // [kSpan][TW] of BT
  int* s_red = reinterpret_cast<int*>(s_B + size_t(kSpan) * Geo::kRowBytes);  // [4]
  uint64_t* s_bar = reinterpret_cast<uint64_t*>(s_red + 4);

  const int tid = threadIdx.x, w = tid >> 5, lane = tid & 31;
  const int i0 = blockIdx.x * R;
  const int nrows = min(R, M - i0);
  const int col0 = blockIdx.y * TW;
  const uint64_t stream_pol = policy_evict_first();

  // ---- rowptr slice, staging decision -----------------------------------
  if (tid <= nrows) s_rp[tid] = ld_stream(rowptr + i0 + tid, stream_pol);
  if (tid == 0) {
    s_red[0] = INT_MAX;  // column min
    s_red[1] = -1;       // column max
    mbar_init(smem_addr(s_bar), 1);
  }
  __syncthreads();
  const int p0 = s_rp[0], p1 = s_rp[nrows];
  const int nbase = p0 & ~3;
  const bool stage = p1 - nbase <= kStage;
  bool window = false;
  int cmin = 0;
  if (stage) {
    const uint32_t bar = smem_addr(s_bar);
    const bool bulk_ok = ((reinterpret_cast<uintptr_t>(colind) | reinterpret_cast<uintptr_t>(vals)) & 15) == 0;
    const int ca = (p0 + 3) & ~3, cb = p1 & ~3;
    const bool c_bulk = bulk_ok && cb > ca;
    if (tid == 0) {
      mbar_arrive_expect_tx(bar, c_bulk ? 8u * uint32_t(cb - ca) : 0u);
      if (c_bulk) {
        bulk_g2s(smem_addr(s_col + (ca - nbase)), colind + ca, 4u * uint32_t(cb - ca), bar);
        bulk_g2s(smem_addr(s_val + (ca - nbase)), vals + ca, 4u * uint32_t(cb - ca), bar);
      }
    }
    if (c_bulk) {
      const int g = tid < 4 ? p0 + tid : cb + (tid - 4);
      if (tid < 8 && ((tid < 4 && g < ca) || (tid >= 4 && g < p1))) {
        s_col[g - nbase] = ld_stream(colind + g, stream_pol);
        s_val[g - nbase] = ld_stream(vals + g, stream_pol);
      }
    } else {
      for (int g = p0 + tid; g < p1; g += kThreads) {
        s_col[g - nbase] = ld_stream(colind + g, stream_pol);
        s_val[g - nbase] = ld_stream(vals + g, stream_pol);
      }
    }
    const bool staged = mbar_wait_bounded(bar, 0, kSpinLimit);
    if (__syncthreads_or(!staged)) {
      if (tid == 0) atomicOr(err, kErrStageTimeout);
      mbar_wait_bounded(bar, 0, kSpinLimit);
      return;
    }
    // column span of the CTA's nonzeros
    int lo = INT_MAX, hi = -1;
    for (int g = p0 + tid; g < p1; g += kThreads) {
      const int c = s_col[g - nbase];
      lo = min(lo, c);
      hi = max(hi, c);
    }
    lo = __reduce_min_sync(0xffffffffu, lo);
    hi = __reduce_max_sync(0xffffffffu, hi);
    if (lane == 0) {
      atomicMin(s_red + 0, lo);
      atomicMax(s_red + 1, hi);
    }
    __syncthreads();
    cmin = s_red[0];
    window = s_red[1] < 0 || s_red[1] - cmin < kSpan;  // no nonzeros, or a narrow span
  }

  // lane's columns of the tile (clamped into the row for loads; stores guarded)
  const int coff = col0 + lane * VEC;
  const bool col_ok = coff < N;

  if (window) {
    const int span = p1 > p0 ? s_red[1] - cmin + 1 : 0;
    // 1. the B window, 16-byte copies (columns past N are copied from the
    //    clamped slice; they only feed lanes whose stores are skipped)
    constexpr int kChunksPerRow = Geo::kRowBytes / 16;
    constexpr int kElemsPerChunk = 16 / int(sizeof(BT));
    for (int c = tid; c < span * kChunksPerRow; c += kThreads) {
      const int jj = c / kChunksPerRow, k = c - jj * kChunksPerRow;
      const int col = min(col0 + k * kElemsPerChunk, N - kElemsPerChunk);
      cp_async16(smem_addr(s_B + size_t(jj) * Geo::kRowBytes + k * 16), B + size_t(cmin + jj) * N + col);
    }
    // 2. this warp's value tile: zero the columns its rows touch, scatter
    const int r0 = w * RW;
    const int rend = min(r0 + RW, nrows);
    int jlo = INT_MAX, jhi = -1;
    if (r0 < nrows) {
      for (int g = s_rp[r0] + lane; g < s_rp[rend]; g += 32) {
        const int c = s_col[g - nbase] - cmin;
        jlo = min(jlo, c);
        jhi = max(jhi, c);
      }
    }
    jlo = __reduce_min_sync(0xffffffffu, jlo);
    jhi = __reduce_max_sync(0xffffffffu, jhi);
    if (jhi < 0) jlo = 0;  // no nonzeros in the warp's rows: the empty range [0, -1]
    float* const aw = s_A + w * (kSpan * RW);  // aw[j * RW + r]
    for (int j = jlo + lane; j <= jhi; j += 32) {
#pragma unroll
      for (int r4 = 0; r4 < RW; r4 += 4) *reinterpret_cast<float4*>(aw + j * RW + r4) = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    __syncwarp();
    for (int r = r0; r < rend; ++r) {
      const int start = s_rp[r], end = s_rp[r + 1];
      bool increasing = true;
      for (int g = start + 1 + lane; g < end; g += 32) increasing &= s_col[g - nbase] > s_col[g - 1 - nbase];
      if (__all_sync(0xffffffffu, increasing)) {
        for (int g = start + lane; g < end; g += 32) aw[(s_col[g - nbase] - cmin) * RW + (r - r0)] = s_val[g - nbase];
      } else if (lane == 0) {
        for (int g = start; g < end; ++g) aw[(s_col[g - nbase] - cmin) * RW + (r - r0)] += s_val[g - nbase];
      }
      __syncwarp();
    }
    cp_async_wait_all();
    __syncthreads();  // the B window is complete for every warp

    // 3. walk the columns
    FVec<VEC> acc[RW];
#pragma unroll
    for (int r = 0; r < RW; ++r) acc[r].zero();
    const BT* bw = reinterpret_cast<const BT*>(s_B) + lane * VEC;
#pragma unroll 2
    for (int j = jlo; j <= jhi; ++j) {
      BSlice<BT, VEC> bs;
      bs.load_shared(bw + j * TW);
      FVec<VEC> b;
      bs.widen(b);
#pragma unroll
      for (int r4 = 0; r4 < RW; r4 += 4) {
        const float4 a = *reinterpret_cast<const float4*>(aw + j * RW + r4);
        acc[r4 + 0].fma(pair(a.x), b);
        acc[r4 + 1].fma(pair(a.y), b);
        acc[r4 + 2].fma(pair(a.z), b);
        acc[r4 + 3].fma(pair(a.w), b);
      }
    }
    if (col_ok) {
#pragma unroll
      for (int r = 0; r < RW; ++r)
        if (r0 + r < nrows) store_c<VEC>(C + size_t(i0 + r0 + r) * N + coff, acc[r]);
    }
    return;
  }

  // ---- gather path: warp w computes rows w, w + 8, ... one at a time --------
  constexpr int U = 4;  // gathers in flight per lane
  const BT* bl = B + min(coff, N - VEC);
  for (int r = w; r < nrows; r += kWinWarps) {
    FVec<VEC> acc;
    acc.zero();
    const int start = s_rp[r], end = s_rp[r + 1];
    for (int base = start; base < end; base += 32) {
      const int cnt = min(32, end - base);
      int myc = 0;
      float myv = 0.f;
      if (lane < cnt) {
        myc = stage ? s_col[base + lane - nbase] : ld_stream(colind + base + lane, stream_pol);
        myv = stage ? s_val[base + lane - nbase] : ld_stream(vals + base + lane, stream_pol);
      }
      for (int t = 0; t < cnt; t += U) {
        BSlice<BT, VEC> bs[U];
        float v[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {  // past cnt: lane 0's column with value 0
          const int src = t + u < cnt ? t + u : 0;
          const int c = __shfl_sync(0xffffffffu, myc, src);
          const float x = __shfl_sync(0xffffffffu, myv, src);
          v[u] = t + u < cnt ? x : 0.f;
          bs[u].load(bl + size_t(c) * N);
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
          FVec<VEC> b;
          bs[u].widen(b);
          acc.fma(pair(v[u]), b);
        }
      }
    }
    if (col_ok) store_c<VEC>(C + size_t(i0 + r) * N + coff, acc);
  }
}

template <typename BT, int VEC>
cudaError_t launch_window_t(const Launch& L) {
  constexpr int TW = 32 * VEC;
  using Geo = WindowGeometry<BT, TW>;
  const size_t smem = Geo::smem_bytes();
  static bool attr_set[kMaxDevices] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= kMaxDevices || !attr_set[dev]) {
    e = cudaFuncSetAttribute(spmm_window_kernel<BT, VEC>, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
    if (e != cudaSuccess) return e;
    if (dev < kMaxDevices) attr_set[dev] = true;
  }
  const dim3 grid(unsigned((int64_t(L.M) + Geo::R - 1) / Geo::R), unsigned((L.N + TW - 1) / TW));
  SPMM_DEBUG_RANGES(L.stream, L.err, {{L.B, size_t(L.K) * L.N * sizeof(BT)}}, {{L.C, size_t(L.M) * L.N * 4}});
  spmm_window_kernel<BT, VEC><<<grid, kThreads, smem, L.stream>>>(
      L.M, L.N, L.rowptr, L.colind, L.vals, static_cast<const BT*>(L.B), L.C, L.err);
  return cudaGetLastError();
}

}  // namespace spmm
