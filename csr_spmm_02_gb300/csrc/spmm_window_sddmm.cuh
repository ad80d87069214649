// Window SDDMM and FusedMM: the dense window of a row block, from shared memory.
//
// SDDMM (page "Performance Optimization of Deep Learning Sparse Matrix Kernels
// on Intel Max Series GPU", SDDMM section, Algorithm 1) gives every stored
// (i, j) the dot product C_i . B_j, and FusedMM (same page, FusedMM section,
// Fig. 6, Algorithm 3) uses those values at once as the sparse values of an
// SpMM with a third matrix D: E_i = sum_j (C_i . B_j) D_j.  The group-per-row
// and merge-path kernels read the B row (and the D row) of every nonzero
// again from L2; for a band of 63 nonzeros per row and N = 256 that is 1-2 KB
// per nonzero.  When consecutive rows touch a narrow range of columns the
// products form a dense window instead, and this kernel computes it from
// shared memory, as the SpMM window kernel does for A . B:
//
//  * a CTA takes 32 rows, stages their column indices and finds the span
//    [cmin, cmax] of columns they touch; if it holds at most 96 columns:
//  * phase 1, 128 columns of N at a time: the B rows of the window and the
//    CTA's C rows are copied into shared memory (16-byte cp.async); warps g
//    and g + 4 compute the dot products of rows 8g .. 8g+7 with all 96 window
//    columns over the first and the second half of the pass's columns (lane
//    l owns columns l, l + 32, l + 64: 24 sums, each B slice reused for 8 rows
//    and each C slice for 3 columns, 16-byte shared loads, rows padded to 132
//    floats so that those loads are free of bank conflicts); the halves are
//    added and each value goes to the tile of the warp that owns its row;
//  * SDDMM: each stored (i, j) takes its dot product from the warp's tile;
//    FusedMM: the tile is masked by the pattern (a stored (i, j) counts once
//    per occurrence, so duplicate entries add their product again, as in the
//    row form) and, 128 columns of N at a time, the D rows of the window are
//    staged and each warp walks the window columns its rows touch: one D slice
//    and one broadcast of 4 values feed 4 rows' accumulators.
//
// A CTA whose span is wider, or that holds more nonzeros than the staging
// area, computes its rows with gathers: per round of 32 nonzeros each lane
// adds its columns' products for all 32, a transposed butterfly leaves
// nonzero l's value in lane l, and FusedMM accumulates the D rows from there.
// Every value's summation order is fixed, so results are deterministic.  The
// window product multiplies non-pattern entries of the window as zeros, so a
// non-finite D value inside the window reaches the block's rows (IEEE special
// values are outside the accepted inputs).
#pragma once

#include <climits>

#include "spmm_device.cuh"
#include "spmm_internal.h"
#include "spmm_sddmm.cuh"
#include "spmm_window.cuh"

namespace spmm {

namespace wsd {
constexpr int kRows = 32;              // rows per CTA
constexpr int kRW = 4;                 // rows per warp
constexpr int kWarps = kThreads / 32;  // 8
constexpr int kChunk = 128;            // columns of N per pass (32 lanes x 4)
constexpr int kSpan = 96;              // window columns
constexpr int kPerLane = kSpan / 32;   // window columns a lane owns
constexpr int kStride = kChunk + 4;    // floats per staged row (528 bytes: 16-byte aligned, odd in 16-byte units)
constexpr int kStage = 2048;           // nonzeros a CTA stages
constexpr int kMaxN = 512;             // widest N (the gather path keeps N / 128 slices per lane)
constexpr int kMaxChunks = kMaxN / kChunk;
__host__ __device__ constexpr size_t smem_bytes() {
  return size_t(kStage + 8) * 4                  // column indices
         + size_t(kRows + 8) * 4                 // rowptr slice
         + size_t(kWarps) * kSpan * kRW * 4      // one value tile per warp, [j][r]
         + size_t(kSpan) * kStride * 4           // window rows of B (phase 1) or D (phase 2)
         + size_t(kRows) * kStride * 4           // the CTA's C rows (phase 1)
         + 32;                                   // reductions, mbarrier
}
}  // namespace wsd

template <bool FUSED>
__global__ void __launch_bounds__(kThreads, 2)
    spmm_window_sddmm_kernel(int32_t M, int32_t N, const int32_t* __restrict__ rowptr,
                             const int32_t* __restrict__ colind, const float* __restrict__ Cd,
                             const float* __restrict__ Bd, const float* __restrict__ Dd, float* __restrict__ out,
                             int* __restrict__ err) {
  // SDDMM: out[p] for every stored p.  FusedMM: out is E (M x N).
  using namespace wsd;
  extern __shared__ __align__(16) unsigned char smem[];
  int* s_col = reinterpret_cast<int*>(smem);
  int* s_rp = s_col + kStage + 8;
  float* s_A = reinterpret_cast<float*>(s_rp + kRows + 8);  // [warp][kSpan][kRW]
  float* s_win = s_A + kWarps * kSpan * kRW;                // [kSpan][kStride]
  float* s_C = s_win + kSpan * kStride;                     // [kRows][kStride]
  int* s_red = reinterpret_cast<int*>(s_C + kRows * kStride);
  uint64_t* s_bar = reinterpret_cast<uint64_t*>(s_red + 4);

  const int tid = threadIdx.x, w = tid >> 5, lane = tid & 31;
  const int i0 = blockIdx.x * kRows;
  const int nrows = min(kRows, M - i0);
  const uint64_t stream_pol = policy_evict_first();

  // ---- rowptr slice, column indices, span ---------------------------------
  if (tid <= nrows) s_rp[tid] = ld_stream(rowptr + i0 + tid, stream_pol);
  if (tid == 0) {
    s_red[0] = INT_MAX;
    s_red[1] = -1;
    mbar_init(smem_addr(s_bar), 1);
  }
  __syncthreads();
  const int p0 = s_rp[0], p1 = s_rp[nrows];
  const int nbase = p0 & ~3;
  const bool stage = p1 - nbase <= kStage;
  bool window = false;
  int cmin = 0, span = 0;
  if (stage) {
    const uint32_t bar = smem_addr(s_bar);
    const bool bulk_ok = (reinterpret_cast<uintptr_t>(colind) & 15) == 0;
    const int ca = (p0 + 3) & ~3, cb = p1 & ~3;  // 16-byte aligned interior of [p0, p1)
    const bool c_bulk = bulk_ok && cb > ca;
    if (tid == 0) {
      mbar_arrive_expect_tx(bar, c_bulk ? 4u * uint32_t(cb - ca) : 0u);
      if (c_bulk) bulk_g2s(smem_addr(s_col + (ca - nbase)), colind + ca, 4u * uint32_t(cb - ca), bar);
    }
    if (c_bulk) {  // at most 3 leading and 3 trailing indices
      const int g = tid < 4 ? p0 + tid : cb + (tid - 4);
      if (tid < 8 && ((tid < 4 && g < ca) || (tid >= 4 && g < p1))) s_col[g - nbase] = ld_stream(colind + g, stream_pol);
    } else {
      for (int g = p0 + tid; g < p1; g += kThreads) s_col[g - nbase] = ld_stream(colind + g, stream_pol);
    }
    const bool staged = mbar_wait_bounded(bar, 0, kSpinLimit);
    if (__syncthreads_or(!staged)) {
      if (tid == 0) atomicOr(err, kErrStageTimeout);
      mbar_wait_bounded(bar, 0, kSpinLimit);  // let copies in flight land before leaving
      return;
    }
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
    span = s_red[1] < 0 ? 0 : s_red[1] - cmin + 1;
    window = span <= kSpan;
  }
  const int r0 = w * kRW;
  const int rend = min(r0 + kRW, nrows);

  if (window) {
    float* const aw = s_A + w * (kSpan * kRW);  // aw[j * kRW + r]
    // the window columns this warp's rows touch
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
    if constexpr (FUSED) {  // occurrences of every stored (row, window column) of the warp
      for (int t = lane; t < kSpan * kRW; t += 32) aw[t] = 0.f;
      __syncwarp();
      for (int r = r0; r < rend; ++r)
        for (int g = s_rp[r] + lane; g < s_rp[r + 1]; g += 32)
          atomicAdd(aw + (s_col[g - nbase] - cmin) * kRW + (r - r0), 1.f);  // small integers: exact in any order
      __syncwarp();
    }

    // ---- phase 1: dot products of the block's rows with the window columns --
    // Warps g and g + 4 take rows 8g .. 8g+7 (kRW2 rows a lane), the first and
    // second half of each pass's columns of N: per 4 columns a lane loads 8 C
    // slices (broadcasts) and 3 B slices for 24 products.
    constexpr int kRW2 = 2 * kRW;
    const int g8 = w & 3, half = w >> 2, r8 = g8 * kRW2;
    float2 dd[kRW2][kPerLane];
#pragma unroll
    for (int r = 0; r < kRW2; ++r)
#pragma unroll
      for (int k = 0; k < kPerLane; ++k) dd[r][k] = make_float2(0.f, 0.f);
    for (int n0 = 0; n0 < N; n0 += kChunk) {
      const int q4 = min(kChunk, N - n0) / 4;  // 16-byte pieces per row in this pass
      __syncthreads();  // every warp is done with the previous pass's rows
      for (int c = tid; c < span * q4; c += kThreads) {
        const int jj = c / q4, k = c - jj * q4;
        cp_async16(smem_addr(s_win + jj * kStride + 4 * k), Bd + size_t(cmin + jj) * N + n0 + 4 * k);
      }
      for (int c = tid; c < nrows * q4; c += kThreads) {
        const int rr = c / q4, k = c - rr * q4;
        cp_async16(smem_addr(s_C + rr * kStride + 4 * k), Cd + size_t(i0 + rr) * N + n0 + 4 * k);
      }
      cp_async_wait_all();
      __syncthreads();
      if (r8 < nrows) {
        // rows past the block and window rows past the span read stale shared
        // memory; their sums are never used (masked or not stored)
        const int kh = (q4 + 1) >> 1, k4a = half ? kh : 0, k4b = half ? q4 : kh;
        for (int k4 = k4a; k4 < k4b; ++k4) {
          float4 c[kRW2], b[kPerLane];
#pragma unroll
          for (int r = 0; r < kRW2; ++r) c[r] = *reinterpret_cast<const float4*>(s_C + (r8 + r) * kStride + 4 * k4);
#pragma unroll
          for (int k = 0; k < kPerLane; ++k)
            b[k] = *reinterpret_cast<const float4*>(s_win + (lane + 32 * k) * kStride + 4 * k4);
#pragma unroll
          for (int r = 0; r < kRW2; ++r)
#pragma unroll
            for (int k = 0; k < kPerLane; ++k) {
              dd[r][k] = __ffma2_rn(make_float2(c[r].x, c[r].y), make_float2(b[k].x, b[k].y), dd[r][k]);
              dd[r][k] = __ffma2_rn(make_float2(c[r].z, c[r].w), make_float2(b[k].z, b[k].w), dd[r][k]);
            }
        }
      }
    }
    // the second half's sums reach the first half's warp through the window
    // buffer (laid out [g][r][k][lane]); lane l owns window columns l, l + 32,
    // l + 64; each value goes to the tile of the warp that owns its row
    __syncthreads();  // every warp is done with the window rows
    float* const xch = s_win;
    if (half) {
#pragma unroll
      for (int r = 0; r < kRW2; ++r)
#pragma unroll
        for (int k = 0; k < kPerLane; ++k) xch[((g8 * kRW2 + r) * kPerLane + k) * 32 + lane] = dd[r][k].x + dd[r][k].y;
    }
    __syncthreads();
    if (!half) {
#pragma unroll
      for (int r = 0; r < kRW2; ++r) {
        float* const ow = s_A + (2 * g8 + r / kRW) * (kSpan * kRW);  // the owning warp's tile
        const int rr = r % kRW;
#pragma unroll
        for (int k = 0; k < kPerLane; ++k) {
          const int j = lane + 32 * k;
          const float v = (dd[r][k].x + dd[r][k].y) + xch[((g8 * kRW2 + r) * kPerLane + k) * 32 + lane];
          if constexpr (FUSED) {
            const float cnt = ow[j * kRW + rr];
            ow[j * kRW + rr] = cnt > 0.f ? cnt * v : 0.f;
          } else {
            ow[j * kRW + rr] = v;
          }
        }
      }
    }
    __syncthreads();  // every tile is complete
    if constexpr (!FUSED) {  // every stored (i, j) takes its dot product
      for (int r = r0; r < rend; ++r)
        for (int g = s_rp[r] + lane; g < s_rp[r + 1]; g += 32)
          st_plain1(out + g, aw[(s_col[g - nbase] - cmin) * kRW + (r - r0)]);
      return;
    } else {
      // ---- phase 2: E rows from the D rows of the window ---------------------
      for (int t0 = 0; t0 < N; t0 += kChunk) {
        const int q4 = min(kChunk, N - t0) / 4;
        __syncthreads();  // every warp is done with the window rows in shared memory
        for (int c = tid; c < span * q4; c += kThreads) {
          const int jj = c / q4, k = c - jj * q4;
          cp_async16(smem_addr(s_win + jj * kStride + 4 * k), Dd + size_t(cmin + jj) * N + t0 + 4 * k);
        }
        cp_async_wait_all();
        __syncthreads();
        if (r0 < nrows) {
          FVec<4> acc[kRW];
#pragma unroll
          for (int r = 0; r < kRW; ++r) acc[r].zero();
          const float* dw = s_win + 4 * min(lane, q4 - 1);  // lanes past the pass read a valid slice
#pragma unroll 2
          for (int j = jlo; j <= jhi; ++j) {
            const float4 a = *reinterpret_cast<const float4*>(aw + j * kRW);
            BSlice<float, 4> ds;
            ds.load_shared(dw + j * kStride);
            FVec<4> d;
            ds.widen(d);
            acc[0].fma(pair(a.x), d);
            acc[1].fma(pair(a.y), d);
            acc[2].fma(pair(a.z), d);
            acc[3].fma(pair(a.w), d);
          }
          if (lane < q4) {
#pragma unroll
            for (int r = 0; r < kRW; ++r)
              if (r0 + r < nrows) store_c<4>(out + size_t(i0 + r0 + r) * N + t0 + 4 * lane, acc[r]);
          }
        }
      }
      return;
    }
  }

  // ---- gather path: warp w computes rows r0 .. rend-1 one at a time ---------
  const int nch = (N + kChunk - 1) / kChunk;
  for (int r = r0; r < rend; ++r) {
    const int row = i0 + r, start = s_rp[r], end = s_rp[r + 1];
    FVec<4> c[kMaxChunks], e[kMaxChunks];
#pragma unroll
    for (int ch = 0; ch < kMaxChunks; ++ch) {
      c[ch].zero();
      e[ch].zero();
      if (ch < nch && ch * kChunk + 4 * lane < N) {
        BSlice<float, 4> cs;
        cs.load(Cd + size_t(row) * N + ch * kChunk + 4 * lane);
        cs.widen(c[ch]);
      }
    }
    for (int base = start; base < end; base += 32) {
      const int cnt = min(32, end - base);
      const int myc = lane < cnt ? (stage ? s_col[base + lane - nbase] : ld_stream(colind + base + lane, stream_pol)) : 0;
      float d[32];
#pragma unroll
      for (int t = 0; t < 32; ++t) {
        const int ct = __shfl_sync(0xffffffffu, myc, t);  // past cnt: lane t's column 0, value discarded
        float s = 0.f;
#pragma unroll
        for (int ch = 0; ch < kMaxChunks; ++ch) {
          if (ch < nch && ch * kChunk + 4 * lane < N) {
            BSlice<float, 4> bs;
            bs.load(Bd + size_t(ct) * N + ch * kChunk + 4 * lane);
            FVec<4> b;
            bs.widen(b);
            float2 p = __fmul2_rn(c[ch].p[0], b.p[0]);
            p = __ffma2_rn(c[ch].p[1], b.p[1], p);
            s += p.x + p.y;
          }
        }
        d[t] = t < cnt ? s : 0.f;
      }
      const float x = group_reduce_transposed<32, 32>(d, lane);  // nonzero base + lane's value
      if constexpr (!FUSED) {
        if (lane < cnt) st_plain1(out + base + lane, x);
      } else {
        for (int t = 0; t < cnt; ++t) {
          const float a = __shfl_sync(0xffffffffu, x, t);
          const int ct = __shfl_sync(0xffffffffu, myc, t);
#pragma unroll
          for (int ch = 0; ch < kMaxChunks; ++ch) {
            if (ch < nch && ch * kChunk + 4 * lane < N) {
              BSlice<float, 4> ds;
              ds.load(Dd + size_t(ct) * N + ch * kChunk + 4 * lane);
              FVec<4> dv;
              ds.widen(dv);
              e[ch].fma(pair(a), dv);
            }
          }
        }
      }
    }
    if constexpr (FUSED) {
#pragma unroll
      for (int ch = 0; ch < kMaxChunks; ++ch)
        if (ch < nch && ch * kChunk + 4 * lane < N) store_c<4>(out + size_t(row) * N + ch * kChunk + 4 * lane, e[ch]);
    }
  }
}

// FUSED: L.B is D, Cd and Bd the dot-product operands, out is E; else out is the nnz values.
// N a multiple of 4, at most 512, Cd/Bd/D/out 16-byte aligned (checked by the caller).
template <bool FUSED>
cudaError_t launch_window_sddmm_t(const Launch& L, const float* Cd, const float* Bd, float* out) {
  const size_t smem = wsd::smem_bytes();
  static bool attr_set[kMaxDevices] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= kMaxDevices || !attr_set[dev]) {
    e = cudaFuncSetAttribute(spmm_window_sddmm_kernel<FUSED>, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
    if (e != cudaSuccess) return e;
    if (dev < kMaxDevices) attr_set[dev] = true;
  }
  const float* D = FUSED ? static_cast<const float*>(L.B) : nullptr;
  const unsigned grid = unsigned((int64_t(L.M) + wsd::kRows - 1) / wsd::kRows);
  SPMM_DEBUG_RANGES(L.stream, L.err,
                    {{Bd, size_t(L.K) * L.N * 4}, {Cd, size_t(L.M) * L.N * 4}, {D, FUSED ? size_t(L.K) * L.N * 4 : 0}},
                    {{out, FUSED ? size_t(L.M) * L.N * 4 : size_t(L.nnz) * 4}});
  spmm_window_sddmm_kernel<FUSED><<<grid, kThreads, smem, L.stream>>>(L.M, L.N, L.rowptr, L.colind, Cd, Bd, D, out,
                                                                       L.err);
  return cudaGetLastError();
}

}  // namespace spmm
