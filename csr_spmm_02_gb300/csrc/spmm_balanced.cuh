// nnz-balanced (merge-path) SpMM kernel and its deterministic fixup.
//
// Work items.  The row ends of A (M items) and its nonzeros (nnz items) are
// merged into one sequence: row i's nonzeros rowptr[i]..rowptr[i+1]-1, then
// row i's end, so row i's end sits at position rowptr[i+1] + i.  Cutting this
// sequence into equal ranges balances both the B gathers (one per nonzero)
// and the C-row stores (one per row end), whatever the row lengths: the even
// split of nonzeros that the Sgap page's related work credits to Yang et al.
// and the element-balanced (EB) choice in its DA-SpMM design space, made to
// count output rows too.  A range starting at diagonal d begins at row
// r(d) = #{rows whose end lies before d} and nonzero d - r(d); the plan
// computes these coordinates once per CTA by binary search over rowptr.
//
// One CTA per range of T items:
//  1. stages the range's colind and vals and the rowptr entries of its rows
//     into shared memory with 1-D bulk copies (the TMA engine; the ESIMD
//     kernel's chunked colind/vals loads and prefetch, Figs. 8-10 of the
//     Intel Max page, and the coalesced row caching the Sgap page cites from
//     Ge-SpMM), plain loads covering the unaligned ends;
//  2. splits the range again among its W worker groups (G lanes each) by the
//     same search in shared memory;
//  3. each worker walks its items in order: U gathers of B rows in flight,
//     FMAs into per-lane registers, and at each row end either a streaming
//     store of the finished C row or, for the row it entered mid-way, a
//     partial in shared memory; the row it leaves unfinished is a second
//     partial;
//  4. after a barrier, partials of one row are summed in worker order (the
//     segmented reduction keyed by row the Sgap page describes; here through
//     shared memory, with no atomics) and stored to C when the row lies inside
//     the CTA, else written to the CTA's two carry slots: slot 0 for the row
//     that began before the range, slot 1 for the row that continues after it.
//
// The fixup kernel then adds, for every row that crosses CTAs, its carry
// slots in CTA order and writes the C row.  No floating-point atomics
// anywhere, so C is bitwise reproducible for a given plan.
#pragma once

#include <climits>

#include "spmm_device.cuh"
#include "spmm_internal.h"

namespace spmm {

constexpr int kFlagCoversStart = 1;  // partial includes the row's first nonzero
constexpr int kFlagCoversEnd = 2;    // partial includes the row's end

template <int G, int NCH>
struct BalancedUnroll {
  static constexpr int value = NCH >= 4 ? 2 : (NCH == 2 ? 4 : 8);
};

__host__ __device__ constexpr size_t balanced_smem_layout_bytes(int W, int TW, int T) {
  return size_t(3) * (T + 8) * 4   // colind, vals, rowptr slices
         + size_t(2) * W * TW * 4  // two partial slots per worker
         + size_t(2) * W * 8       // slot metadata (row, flags)
         + 16;                     // mbarrier
}

template <typename BT, int VEC, int G, int NCH>
__global__ void __launch_bounds__(kThreads)
    spmm_balanced_kernel(int32_t M, int32_t N, const int32_t* __restrict__ rowptr,
                         const int32_t* __restrict__ colind, const float* __restrict__ vals,
                         const BT* __restrict__ B, float* __restrict__ C,
                         const int2* __restrict__ part, int32_t T, float* __restrict__ carry,
                         int* __restrict__ err) {
  constexpr int W = kThreads / G;
  constexpr int TW = G * VEC * NCH;
  constexpr int U = BalancedUnroll<G, NCH>::value;

  extern __shared__ __align__(16) unsigned char smem[];
  const int Tpad = T + 8;
  int* s_col = reinterpret_cast<int*>(smem);
  float* s_val = reinterpret_cast<float*>(s_col + Tpad);
  int* s_rp = reinterpret_cast<int*>(s_val + Tpad);
  float* s_slot = reinterpret_cast<float*>(s_rp + Tpad);      // [W][2][TW]
  int2* s_meta = reinterpret_cast<int2*>(s_slot + 2 * W * TW);  // [W][2] (row, flags)
  uint64_t* s_bar = reinterpret_cast<uint64_t*>(s_meta + 2 * W);

  const int tid = threadIdx.x;
  const int cta = blockIdx.x;
  const int2 beg = __ldg(part + cta);
  const int2 fin = __ldg(part + cta + 1);
  const int i0 = beg.x, p0 = beg.y, i1 = fin.x, p1 = fin.y;
  const int nbase = p0 & ~3;  // s_col[k], s_val[k] hold nonzero nbase + k
  const int rbase = i0 & ~3;  // s_rp[k] holds rowptr[rbase + k]; rows i0..i1 are staged

  // ---- 1. stage the range -------------------------------------------------
  const uint32_t bar = smem_addr(s_bar);
  const bool bulk_ok =
      ((reinterpret_cast<uintptr_t>(colind) | reinterpret_cast<uintptr_t>(vals) |
        reinterpret_cast<uintptr_t>(rowptr)) & 15) == 0;
  const int ca = (p0 + 3) & ~3, cb = p1 & ~3;      // 16-byte aligned interior of [p0, p1)
  const int ra = (i0 + 3) & ~3, rb = (i1 + 1) & ~3;  // ... of [i0, i1 + 1)
  const bool c_bulk = bulk_ok && cb > ca;
  const bool r_bulk = bulk_ok && rb > ra;
  if (tid == 0) mbar_init(bar, 1);
  for (int k = tid; k < 2 * W; k += kThreads) s_meta[k] = make_int2(-1, 0);
  __syncthreads();
  if (tid == 0) {
    const uint32_t bytes = (c_bulk ? 8u * uint32_t(cb - ca) : 0u) + (r_bulk ? 4u * uint32_t(rb - ra) : 0u);
    mbar_arrive_expect_tx(bar, bytes);
    if (c_bulk) {
      bulk_g2s(smem_addr(s_col + (ca - nbase)), colind + ca, 4u * uint32_t(cb - ca), bar);
      bulk_g2s(smem_addr(s_val + (ca - nbase)), vals + ca, 4u * uint32_t(cb - ca), bar);
    }
    if (r_bulk) bulk_g2s(smem_addr(s_rp + (ra - rbase)), rowptr + ra, 4u * uint32_t(rb - ra), bar);
  }
  if (c_bulk) {  // at most 3 leading and 3 trailing nonzeros
    const int g = tid < 4 ? p0 + tid : cb + (tid - 4);
    if (tid < 8 && ((tid < 4 && g < ca) || (tid >= 4 && g < p1))) {
      s_col[g - nbase] = __ldg(colind + g);
      s_val[g - nbase] = __ldg(vals + g);
    }
  } else {
    for (int g = p0 + tid; g < p1; g += kThreads) {
      s_col[g - nbase] = __ldg(colind + g);
      s_val[g - nbase] = __ldg(vals + g);
    }
  }
  if (r_bulk) {
    const int g = tid < 4 ? i0 + tid : rb + (tid - 4);
    if (tid < 8 && ((tid < 4 && g < ra) || (tid >= 4 && g <= i1))) s_rp[g - rbase] = __ldg(rowptr + g);
  } else {
    for (int g = i0 + tid; g <= i1; g += kThreads) s_rp[g - rbase] = __ldg(rowptr + g);
  }
  const bool staged = mbar_wait_bounded(bar, 0, kSpinLimit);
  if (__syncthreads_or(!staged)) {
    if (tid == 0) atomicOr(err, kErrStageTimeout);
    mbar_wait_bounded(bar, 0, kSpinLimit);  // let copies in flight land before leaving
    return;
  }

  // ---- 2. this worker's sub-range -----------------------------------------
  const int w = tid / G;
  const int lane = tid & (G - 1);
  const int* rp = s_rp + (i0 - rbase);  // rp[r] = rowptr[i0 + r], 0 <= r <= i1 - i0
  const int items = (i1 - i0) + (p1 - p0);
  const int Tw = T / W;
  const int dl0 = min(w * Tw, items);
  const int dl1 = min(dl0 + Tw, items);
  auto find_row = [&](int dl) {  // first local row whose end lies at or after dl
    int lo = 0, hi = i1 - i0;
    while (lo < hi) {
      const int mid = (lo + hi) >> 1;
      if (rp[mid + 1] - p0 + mid >= dl) hi = mid; else lo = mid + 1;
    }
    return lo;
  };
  const int rw0 = find_row(dl0);
  const int rw1 = find_row(dl1);
  const int pw0 = p0 + dl0 - rw0;
  const int pw1 = p0 + dl1 - rw1;

  const int col0 = blockIdx.y * TW;
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

  auto slot_ptr = [&](int worker, int slot, int ch) {
    return s_slot + (worker * 2 + slot) * TW + (ch * G + lane) * VEC;
  };
  // Row r (local) ends inside this worker: store it, or park it as this
  // worker's head partial when the row began before the worker's range.
  auto emit = [&](int r, bool began_before) {
    const int grow = i0 + r;
    if (began_before) {
#pragma unroll
      for (int ch = 0; ch < NCH; ++ch) store_f4<VEC>(slot_ptr(w, 0, ch), acc[ch]);
      if (lane == 0) s_meta[w * 2] = make_int2(grow, kFlagCoversEnd);
    } else {
      float* crow = C + size_t(grow) * N;
#pragma unroll
      for (int ch = 0; ch < NCH; ++ch)
        if (cok[ch]) store_c<VEC>(crow + coff[ch], acc[ch]);
    }
#pragma unroll
    for (int ch = 0; ch < NCH; ++ch)
#pragma unroll
      for (int j = 0; j < VEC; ++j) acc[ch][j] = 0.f;
  };

  // ---- 3. walk the sub-range ----------------------------------------------
  int r = rw0;
  bool began_before = rp[r] < pw0;
  int next_end = r < rw1 ? rp[r + 1] : INT_MAX;
  for (int p = pw0; p < pw1;) {
    const int nb = min(U, pw1 - p);
    BSlice<BT, VEC> bs[U][NCH];
    float v[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      if (u < nb) {
        const int k = p + u - nbase;
        const int c = s_col[k];
        v[u] = s_val[k];
        const BT* brow = B + size_t(c) * N;
#pragma unroll
        for (int ch = 0; ch < NCH; ++ch)
          if (cok[ch]) bs[u][ch].load(brow + coff[ch]);
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      if (u < nb) {
        while (p + u == next_end) {  // rows ending before this nonzero (empty rows too)
          emit(r, began_before);
          ++r;
          began_before = false;
          next_end = r < rw1 ? rp[r + 1] : INT_MAX;
        }
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
    p += nb;
  }
  while (r < rw1) {  // rows ending exactly at the end of the sub-range
    emit(r, began_before);
    ++r;
    began_before = false;
  }
  if (i0 + r < M && rp[r] < pw1) {  // row r continues past this worker: tail partial
#pragma unroll
    for (int ch = 0; ch < NCH; ++ch) store_f4<VEC>(slot_ptr(w, 1, ch), acc[ch]);
    if (lane == 0) s_meta[w * 2 + 1] = make_int2(i0 + r, rp[r] >= pw0 ? kFlagCoversStart : 0);
  }
  __syncthreads();

  // ---- 4. combine partials of rows split between workers -------------------
#pragma unroll
  for (int slot = 0; slot < 2; ++slot) {
    const int2 m = s_meta[w * 2 + slot];
    if (m.x < 0) continue;
    const bool covers_start = m.y & kFlagCoversStart;
    const bool first_of_cta = w == 0 && (slot == 0 || s_meta[0].x < 0);
    if (!covers_start && !first_of_cta) continue;  // not the first piece of its row here
    const int row = m.x;
    float sum[NCH][VEC];
#pragma unroll
    for (int ch = 0; ch < NCH; ++ch) load_f4<VEC>(slot_ptr(w, slot, ch), sum[ch]);
    bool covers_end = slot == 0;
    for (int w2 = w + 1; !covers_end && w2 < W; ++w2) {
      int take;
      if (s_meta[w2 * 2].x >= 0) {  // the row ends in worker w2
        take = 0;
        covers_end = true;
      } else if (s_meta[w2 * 2 + 1].x == row) {  // worker w2 lies inside the row
        take = 1;
      } else {
        break;  // past the end of this CTA's items
      }
#pragma unroll
      for (int ch = 0; ch < NCH; ++ch) {
        float part_sum[VEC];
        load_f4<VEC>(slot_ptr(w2, take, ch), part_sum);
#pragma unroll
        for (int j = 0; j < VEC; ++j) sum[ch][j] += part_sum[j];
      }
    }
    if (covers_start && covers_end) {
      float* crow = C + size_t(row) * N;
#pragma unroll
      for (int ch = 0; ch < NCH; ++ch)
        if (cok[ch]) store_c<VEC>(crow + coff[ch], sum[ch]);
    } else {
      float* dst = carry + (size_t(cta) * 2 + (covers_start ? 1 : 0)) * N;
#pragma unroll
      for (int ch = 0; ch < NCH; ++ch)
        if (cok[ch]) store_f4<VEC>(dst + coff[ch], sum[ch]);
    }
  }
}

template <typename BT, int VEC, int G, int NCH>
cudaError_t launch_balanced_t(const Launch& L) {
  constexpr int W = kThreads / G;
  constexpr int TW = G * VEC * NCH;
  const size_t smem = balanced_smem_layout_bytes(W, TW, L.items_per_cta);
  static bool attr_set[kMaxDevices] = {};  // per instantiation and device
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= kMaxDevices || !attr_set[dev]) {
    e = cudaFuncSetAttribute(spmm_balanced_kernel<BT, VEC, G, NCH>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             int(balanced_smem_layout_bytes(W, TW, kMaxItemsPerCta)));
    if (e != cudaSuccess) return e;
    if (dev < kMaxDevices) attr_set[dev] = true;
  }
  const dim3 grid(unsigned(L.num_ctas), unsigned((L.N + TW - 1) / TW));
  spmm_balanced_kernel<BT, VEC, G, NCH><<<grid, kThreads, smem, L.stream>>>(
      L.M, L.N, L.rowptr, L.colind, L.vals, static_cast<const BT*>(L.B), L.C, L.part,
      L.items_per_cta, L.carry, L.err);
  return cudaGetLastError();
}

}  // namespace spmm
