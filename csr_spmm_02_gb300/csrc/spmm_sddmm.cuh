// SDDMM on the CSR pattern of A: out[p] = C_i . B_j for every stored (i, j).
//
// The SDDMM section of "Performance Optimization of Deep Learning Sparse
// Matrix Kernels on Intel Max Series GPU" (Algorithm 1, Figs. 3-4, 7) assigns
// each row of the sparse output to one or more work-items (NT per row), keeps
// the row C_i in registers and produces every nonzero of the row as a dot
// product with the row B_j it selects.  Here the rows of a CTA come from the
// same merge-path ranges as the SpMM kernels (balanced in rows + nonzeros), a
// warp takes a sub-range, and its S = 32/G lane groups take consecutive
// nonzeros: a group keeps the C row of its current nonzero's row in registers
// (reloaded when the row changes), gathers the B row with 16-byte loads, and
// its G lanes add their partial dot products with shuffles before one lane
// stores the value.  Each output is written once; no reduction crosses CTAs.
#pragma once

#include <climits>

#include "spmm_device.cuh"
#include "spmm_internal.h"

namespace spmm {

__host__ __device__ constexpr size_t sddmm_smem_layout_bytes(int T) {
  return size_t(2) * (T + 8) * 4 + 16;  // colind and rowptr slices, mbarrier
}

// A lane's share of a dot product: chunks whose columns lie past N (their
// loads were clamped into the row) contribute nothing.
template <int VEC, int NCH>
__device__ __forceinline__ float dot_lane(const FVec<VEC> (&c)[NCH], const FVec<VEC> (&b)[NCH],
                                          const bool (&valid)[NCH], float d) {
#pragma unroll
  for (int ch = 0; ch < NCH; ++ch) {
    float t = 0.f;
    if constexpr (VEC == 1) {
      t = c[ch].x * b[ch].x;
    } else {
#pragma unroll
      for (int j = 0; j < VEC / 2; ++j) {
        t = fmaf(c[ch].p[j].x, b[ch].p[j].x, t);
        t = fmaf(c[ch].p[j].y, b[ch].p[j].y, t);
      }
    }
    d += valid[ch] ? t : 0.f;
  }
  return d;
}

// Dot-product share of a lane over the column tiles after the first
// (rows wider than one tile of G*VEC*NCH columns); loads are not batched.
template <int VEC, int G, int NCH>
__device__ __forceinline__ float dot_tail_tiles(const float* crow, const float* brow, int N, int gl, float d) {
  constexpr int TW = G * VEC * NCH;
  for (int t0 = TW; t0 < N; t0 += TW) {
    FVec<VEC> c[NCH], b[NCH];
    bool valid[NCH];
#pragma unroll
    for (int ch = 0; ch < NCH; ++ch) {
      const int col = t0 + (ch * G + gl) * VEC;
      valid[ch] = col < N;
      const int cl = min(col, N - VEC);
      BSlice<float, VEC> x, y;
      x.load(crow + cl);
      y.load(brow + cl);
      x.widen(c[ch]);
      y.widen(b[ch]);
    }
    d = dot_lane<VEC, NCH>(c, b, valid, d);
  }
  return d;
}

// Sum over the G lanes of each group (every lane of the warp takes part).
template <int G>
__device__ __forceinline__ float group_sum(float d) {
#pragma unroll
  for (int o = G / 2; o > 0; o >>= 1) d += __shfl_xor_sync(0xffffffffu, d, o);
  return d;
}

template <int VEC, int G, int NCH>
__global__ void __launch_bounds__(kThreads)
    spmm_sddmm_kernel(int32_t M, int32_t N, const int32_t* __restrict__ rowptr, const int32_t* __restrict__ colind,
                      const float* __restrict__ Cd, const float* __restrict__ B, float* __restrict__ out,
                      const int2* __restrict__ part, int32_t T, int* __restrict__ err) {
  constexpr int S = 32 / G;
  constexpr int W = kThreads / 32;
  constexpr int U = 8 / NCH > 0 ? 8 / NCH : 1;  // steps per batch

  extern __shared__ __align__(16) unsigned char smem[];
  const int Tpad = T + 8;
  int* s_col = reinterpret_cast<int*>(smem);
  int* s_rp = s_col + Tpad;
  uint64_t* s_bar = reinterpret_cast<uint64_t*>(s_col + 2 * Tpad);

  const int tid = threadIdx.x;
  const int2 beg = __ldg(part + blockIdx.x);
  const int2 fin = __ldg(part + blockIdx.x + 1);
  const int i0 = beg.x, p0 = beg.y, i1 = fin.x, p1 = fin.y;
  const int nbase = p0 & ~3, rbase = i0 & ~3;
  const uint64_t stream_pol = policy_evict_first();

  // ---- stage colind[p0, p1) and rowptr[i0, i1] ------------------------------
  const uint32_t bar = smem_addr(s_bar);
  const bool bulk_ok = ((reinterpret_cast<uintptr_t>(colind) | reinterpret_cast<uintptr_t>(rowptr)) & 15) == 0;
  const int ca = (p0 + 3) & ~3, cb = p1 & ~3;
  const int ra = (i0 + 3) & ~3, rb = (i1 + 1) & ~3;
  const bool c_bulk = bulk_ok && cb > ca;
  const bool r_bulk = bulk_ok && rb > ra;
  if (tid == 0) mbar_init(bar, 1);
  __syncthreads();
  if (tid == 0) {
    mbar_arrive_expect_tx(bar, (c_bulk ? 4u * uint32_t(cb - ca) : 0u) + (r_bulk ? 4u * uint32_t(rb - ra) : 0u));
    if (c_bulk) bulk_g2s(smem_addr(s_col + (ca - nbase)), colind + ca, 4u * uint32_t(cb - ca), bar);
    if (r_bulk) bulk_g2s(smem_addr(s_rp + (ra - rbase)), rowptr + ra, 4u * uint32_t(rb - ra), bar);
  }
  if (c_bulk) {
    const int g = tid < 4 ? p0 + tid : cb + (tid - 4);
    if (tid < 8 && ((tid < 4 && g < ca) || (tid >= 4 && g < p1))) s_col[g - nbase] = ld_stream(colind + g, stream_pol);
  } else {
    for (int g = p0 + tid; g < p1; g += kThreads) s_col[g - nbase] = ld_stream(colind + g, stream_pol);
  }
  if (r_bulk) {
    const int g = tid < 4 ? i0 + tid : rb + (tid - 4);
    if (tid < 8 && ((tid < 4 && g < ra) || (tid >= 4 && g <= i1))) s_rp[g - rbase] = ld_stream(rowptr + g, stream_pol);
  } else {
    for (int g = i0 + tid; g <= i1; g += kThreads) s_rp[g - rbase] = ld_stream(rowptr + g, stream_pol);
  }
  const bool staged = mbar_wait_bounded(bar, 0, kSpinLimit);
  if (__syncthreads_or(!staged)) {
    if (tid == 0) atomicOr(err, kErrStageTimeout);
    mbar_wait_bounded(bar, 0, kSpinLimit);
    return;
  }

  // ---- this warp's sub-range --------------------------------------------------
  const int w = tid >> 5, lane = tid & 31, grp = lane / G, gl = lane & (G - 1);
  const int* rp = s_rp + (i0 - rbase);
  const int items = (i1 - i0) + (p1 - p0);
  const int Tw = T / W;
  auto find_row = [&](int dl) {
    int lo = 0, hi = i1 - i0;
    while (lo < hi) {
      const int mid = (lo + hi) >> 1;
      if (rp[mid + 1] - p0 + mid >= dl) hi = mid; else lo = mid + 1;
    }
    return lo;
  };
  const int dl0 = min(w * Tw, items), dl1 = min(dl0 + Tw, items);
  const int rw0 = find_row(dl0), rw1 = find_row(dl1);
  const int pw0 = p0 + dl0 - rw0, pw1 = p0 + dl1 - rw1;
  if (pw0 >= pw1) return;  // no nonzeros in this sub-range (uniform in the warp)

  int coffl[NCH];
  bool valid[NCH];
  const float* bl[NCH];
#pragma unroll
  for (int ch = 0; ch < NCH; ++ch) {
    const int col = (ch * G + gl) * VEC;  // first column tile
    valid[ch] = col < N;
    coffl[ch] = min(col, N - VEC);
    bl[ch] = B + coffl[ch];
  }
  const int last_row = i1 - i0;  // rows past it hold no nonzero of this CTA
  const int* colw = s_col - nbase + grp;
  int rg = rw0;      // row of this group's current nonzero (local)
  int loaded = -1;   // row whose C slice is in c
  FVec<VEC> c[NCH];
  for (int q = pw0; q < pw1; q += U * S) {
    BSlice<float, VEC> bs[U][NCH];
#pragma unroll
    for (int s = 0; s < U; ++s) {
      const size_t roff = size_t(colw[min(q + s * S, pw1 - 1 - grp)]) * N;
#pragma unroll
      for (int ch = 0; ch < NCH; ++ch) bs[s][ch].load(bl[ch] + roff);
    }
#pragma unroll
    for (int s = 0; s < U; ++s) {
      const int a = q + s * S;
      if (a >= pw1) break;
      const int n = a + grp;
      float d = 0.f;
      if (n < pw1) {
        while (rg < last_row && rp[rg + 1] <= n) ++rg;  // rows only advance along the sub-range
        if (rg != loaded) {
          const float* crow = Cd + size_t(i0 + rg) * N;
#pragma unroll
          for (int ch = 0; ch < NCH; ++ch) {
            BSlice<float, VEC> t;
            t.load(crow + coffl[ch]);
            t.widen(c[ch]);
          }
          loaded = rg;
        }
        FVec<VEC> b[NCH];
#pragma unroll
        for (int ch = 0; ch < NCH; ++ch) bs[s][ch].widen(b[ch]);
        d = dot_lane<VEC, NCH>(c, b, valid, 0.f);
        if (N > G * VEC * NCH)
          d = dot_tail_tiles<VEC, G, NCH>(Cd + size_t(i0 + rg) * N, B + size_t(colw[a]) * N, N, gl, d);
      }
      d = group_sum<G>(d);
      if (gl == 0 && n < pw1) st_stream1(out + n, d);
    }
  }
}

template <int VEC, int G, int NCH>
cudaError_t launch_sddmm_t(const Launch& L, const float* Cd, float* out) {
  const size_t smem = sddmm_smem_layout_bytes(L.items_per_cta);
  static bool attr_set[kMaxDevices] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= kMaxDevices || !attr_set[dev]) {
    e = cudaFuncSetAttribute(spmm_sddmm_kernel<VEC, G, NCH>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             int(sddmm_smem_layout_bytes(kMaxItemsPerCta)));
    if (e != cudaSuccess) return e;
    if (dev < kMaxDevices) attr_set[dev] = true;
  }
  spmm_sddmm_kernel<VEC, G, NCH><<<unsigned(L.num_ctas), kThreads, smem, L.stream>>>(
      L.M, L.N, L.rowptr, L.colind, Cd, static_cast<const float*>(L.B), out, L.part, L.items_per_cta, L.err);
  return cudaGetLastError();
}

}  // namespace spmm
