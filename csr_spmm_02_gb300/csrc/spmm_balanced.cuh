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
// One CTA per range [(i0, p0), (i1, p1)) of T items:
//  1. stages the range's colind and vals in shared memory with 1-D bulk
//     copies (the TMA engine; the ESIMD kernel's chunked colind/vals loads and
//     prefetch, Figs. 8-10 of the Intel Max page, and the coalesced row caching
//     the Sgap page cites from Ge-SpMM), plain loads covering unaligned ends;
//  2. meanwhile reads rowptr[i0..i1+1] once: marks where each row's
//     nonzeros start, lists the empty rows whose end lies in the range, and a
//     block max-scan turns the marks into a row id per staged nonzero; the
//     empty rows' C rows are stored as zeros, coalesced;
//  3. splits its nonzeros evenly among W worker groups of G lanes; each
//     worker streams its nonzeros in batches of U (gathers of B rows issued
//     before the FMAs that use them; short batches zero-extended), and when
//     the row id changes stores the finished C row (streaming store) -- or
//     parks it as a partial in shared memory when the row started before the
//     worker's nonzeros (slot 0) or continues after them (slot 1);
//  4. after a barrier, the partials of each row are summed in worker order
//     (the segmented reduction keyed by row of the Sgap page, done through
//     shared memory without atomics) and stored to C when the row lies inside
//     the CTA, else written to the CTA's carry slot 0 (row began before the
//     range) or 1 (row began inside and continues after it).
//
// The fixup kernel then adds, for every row whose nonzeros cross CTAs, its
// carry slots in CTA order and writes the C row.  No floating-point atomics
// anywhere, so C is bitwise reproducible for a given plan.
#pragma once

#include <climits>

#include "spmm_device.cuh"
#include "spmm_internal.h"

#ifndef SPMM_BAL_LOADS
#define SPMM_BAL_LOADS 4  // 16-byte B loads in flight per lane (U nonzeros x NCH chunks)
#endif
#ifndef SPMM_BAL_MIN_BLOCKS
#define SPMM_BAL_MIN_BLOCKS 1
#endif

namespace spmm {

// Kinds of a worker's parked partial row (its shared-memory slot).
constexpr int kSlotHead = 1;    // the row began before the worker and ends in it
constexpr int kSlotMiddle = 2;  // the worker lies entirely inside the row

template <int NCH>
struct BalancedUnroll {
  static constexpr int value = SPMM_BAL_LOADS / NCH > 0 ? SPMM_BAL_LOADS / NCH : 1;
};

__host__ __device__ constexpr size_t balanced_smem_layout_bytes(int W, int TW, int T) {
  return size_t(4) * (T + 8) * 4   // colind, vals, row ids, empty-row list
         + size_t(1) * W * TW * 4  // one parked partial row per worker
         + size_t(1) * W * 8       // slot metadata (local row, kind)
         + 64 * 4                  // scan scratch, counters, flags
         + 16;                     // mbarrier
}

template <typename BT, int VEC, int G, int NCH>
__global__ void __launch_bounds__(kThreads, SPMM_BAL_MIN_BLOCKS)
    spmm_balanced_kernel(int32_t M, int32_t N, const int32_t* __restrict__ rowptr,
                         const int32_t* __restrict__ colind, const float* __restrict__ vals,
                         const BT* __restrict__ B, float* __restrict__ C,
                         const int2* __restrict__ part, int32_t T, float* __restrict__ carry,
                         int* __restrict__ err) {
  constexpr int W = kThreads / G;
  constexpr int TW = G * VEC * NCH;
  constexpr int U = BalancedUnroll<NCH>::value;

  extern __shared__ __align__(16) unsigned char smem[];
  const int Tpad = T + 8;
  int* s_col = reinterpret_cast<int*>(smem);
  float* s_val = reinterpret_cast<float*>(s_col + Tpad);
  int* s_row = s_col + 2 * Tpad;    // local row id of each staged nonzero
  int* s_empty = s_col + 3 * Tpad;  // local ids of empty rows ending in this range
  float* s_slot = reinterpret_cast<float*>(s_col + 4 * Tpad);  // [W][TW] parked partial rows
  int2* s_meta = reinterpret_cast<int2*>(s_slot + W * TW);     // [W] (local row, kind)
  int* s_misc = reinterpret_cast<int*>(s_meta + W);            // [0..7] scan, [8] #empty, [9..10] flags
  uint64_t* s_bar = reinterpret_cast<uint64_t*>(s_misc + 64);

  const int tid = threadIdx.x;
  const int warp = tid >> 5, wl = tid & 31;
  const int cta = blockIdx.x;
  const uint64_t stream_pol = policy_evict_first();
  const int2 beg = __ldg(part + cta);
  const int2 fin = __ldg(part + cta + 1);
  const int i0 = beg.x, p0 = beg.y, i1 = fin.x, p1 = fin.y;
  const int nbase = p0 & ~3;  // s_col[k], s_val[k], s_row[k] describe nonzero nbase + k
  const int nnz_here = p1 - p0;
  const int col0 = blockIdx.y * TW;

  // ---- 1. launch the bulk copies; init row ids ------------------------------
  const uint32_t bar = smem_addr(s_bar);
  const bool bulk_ok = ((reinterpret_cast<uintptr_t>(colind) | reinterpret_cast<uintptr_t>(vals)) & 15) == 0;
  const int ca = (p0 + 3) & ~3, cb = p1 & ~3;  // 16-byte aligned interior of [p0, p1)
  const bool c_bulk = bulk_ok && cb > ca;
  if (tid == 0) {
    mbar_init(bar, 1);
    s_misc[8] = 0;
  }
  for (int k = p0 - nbase + tid; k < p1 - nbase; k += kThreads) s_row[k] = -1;
  for (int k = tid; k < W; k += kThreads) s_meta[k] = make_int2(-1, 0);
  __syncthreads();
  if (tid == 0) {
    mbar_arrive_expect_tx(bar, c_bulk ? 8u * uint32_t(cb - ca) : 0u);
    if (c_bulk) {
      bulk_g2s(smem_addr(s_col + (ca - nbase)), colind + ca, 4u * uint32_t(cb - ca), bar);
      bulk_g2s(smem_addr(s_val + (ca - nbase)), vals + ca, 4u * uint32_t(cb - ca), bar);
    }
    // Does the first nonzero belong to a row that began before the range, and
    // does the last nonzero's row continue after it?
    const int rs0 = ld_stream(rowptr + i0, stream_pol);
    const int re0 = i0 < M ? ld_stream(rowptr + i0 + 1, stream_pol) : rs0;
    const bool first_before = nnz_here > 0 && rs0 < p0 && p0 < re0;
    if (first_before) s_row[p0 - nbase] = 0;
    s_misc[9] = first_before;
    const int rs1 = ld_stream(rowptr + i1, stream_pol);
    const int re1 = i1 < M ? ld_stream(rowptr + i1 + 1, stream_pol) : rs1;
    s_misc[10] = nnz_here > 0 && rs1 < p1 && re1 > p1;
  }
  if (c_bulk) {  // at most 3 leading and 3 trailing nonzeros
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
  // ---- 2. row starts and empty rows -----------------------------------------
  for (int r = i0 + tid; r <= i1 && r < M; r += kThreads) {
    const int rs = ld_stream(rowptr + r, stream_pol);
    const int re = ld_stream(rowptr + r + 1, stream_pol);
    if (rs < re) {
      if (rs >= p0 && rs < p1) s_row[rs - nbase] = r - i0;
    } else if (r < i1) {
      s_empty[atomicAdd(s_misc + 8, 1)] = r;
    }
  }
  __syncthreads();
  {  // zero the empty rows' C tiles: consecutive threads store consecutive 16-byte pieces
    constexpr int kPieces = TW / (VEC >= 4 ? 4 : 1);
    const int n_empty = s_misc[8];
    for (int u = tid; u < n_empty * kPieces; u += kThreads) {
      const int e = u / kPieces;
      const int col = col0 + (u - e * kPieces) * (VEC >= 4 ? 4 : 1);
      if (col < N) {
        float* dst = C + size_t(s_empty[e]) * N + col;
        if constexpr (VEC >= 4) {
          st_stream4(dst, 0.f, 0.f, 0.f, 0.f);
        } else {
          st_stream1(dst, 0.f);
        }
      }
    }
  }
  {  // inclusive max-scan of the row-start marks -> row id of every nonzero
    const int per_t = (nnz_here + kThreads - 1) / kThreads;
    const int a = p0 - nbase + tid * per_t;
    const int b = min(a + per_t, p1 - nbase);
    int run = -1;
    for (int k = a; k < b; ++k) run = max(run, s_row[k]);
    int incl = run;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, o);
      if (wl >= o) incl = max(incl, y);
    }
    if (wl == 31) s_misc[warp] = incl;
    __syncthreads();
    int prefix = __shfl_up_sync(0xffffffffu, incl, 1);
    if (wl == 0) prefix = -1;
    for (int x = 0; x < warp; ++x) prefix = max(prefix, s_misc[x]);
    for (int k = a; k < b; ++k) {
      prefix = max(prefix, s_row[k]);
      s_row[k] = prefix;
    }
  }
  const bool staged = mbar_wait_bounded(bar, 0, kSpinLimit);
  if (__syncthreads_or(!staged)) {
    if (tid == 0) atomicOr(err, kErrStageTimeout);
    mbar_wait_bounded(bar, 0, kSpinLimit);  // let copies in flight land before leaving
    return;
  }

  // ---- 3. stream this worker's nonzeros -------------------------------------
  const int w = tid / G;
  const int lane = tid & (G - 1);
  const int per_w = (nnz_here + W - 1) / W;
  const int q0 = p0 + min(w * per_w, nnz_here);
  const int q1 = p0 + min((w + 1) * per_w, nnz_here);
  int coff[NCH], coffl[NCH];  // store offsets; load offsets clamped into the row
  bool cok[NCH];
#pragma unroll
  for (int ch = 0; ch < NCH; ++ch) {
    coff[ch] = col0 + (ch * G + lane) * VEC;
    coffl[ch] = min(coff[ch], N - VEC);
    cok[ch] = coff[ch] < N;
  }
  auto slot_ptr = [&](int worker, int ch) { return s_slot + worker * TW + (ch * G + lane) * VEC; };
  // The worker's unfinished last row, when the row also began in this worker:
  // kept in registers across the barrier and completed by this worker.
  bool has_tail = false;
  int tail_row = -1;
  float acc[NCH][VEC];
#pragma unroll
  for (int ch = 0; ch < NCH; ++ch)
#pragma unroll
    for (int j = 0; j < VEC; ++j) acc[ch][j] = 0.f;

  if (q0 < q1) {
    const int first = s_row[q0 - nbase];
    const bool head_partial = q0 > p0 ? s_row[q0 - 1 - nbase] == first : s_misc[9] != 0;
    // Finished row `r`: C row, or a parked head partial when it began before q0.
    auto flush = [&](int r) {
      if (r == first && head_partial) {
#pragma unroll
        for (int ch = 0; ch < NCH; ++ch) store_f4<VEC>(slot_ptr(w, ch), acc[ch]);
        if (lane == 0) s_meta[w] = make_int2(r, kSlotHead);
      } else {
        float* crow = C + size_t(i0 + r) * N;
#pragma unroll
        for (int ch = 0; ch < NCH; ++ch)
          if (cok[ch]) store_c<VEC>(crow + coff[ch], acc[ch]);
      }
#pragma unroll
      for (int ch = 0; ch < NCH; ++ch)
#pragma unroll
        for (int j = 0; j < VEC; ++j) acc[ch][j] = 0.f;
    };

    int cur = first;
    for (int q = q0; q < q1; q += U) {
      // Issue the batch's gathers first (a padded slot re-reads the worker's
      // last row); values and row ids are re-read from shared memory
      // afterwards, so only the B slices occupy registers while loads fly.
      BSlice<BT, VEC> bs[U][NCH];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const BT* brow = B + size_t(s_col[min(q + u, q1 - 1) - nbase]) * N;
#pragma unroll
        for (int ch = 0; ch < NCH; ++ch) bs[u][ch].load(brow + coffl[ch]);
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int k = min(q + u, q1 - 1) - nbase;
        const int r = s_row[k];  // a padded slot repeats the last row: no flush
        const float v = q + u < q1 ? s_val[k] : 0.f;
        if (r != cur) {
          flush(cur);
          cur = r;
        }
        const uint64_t vv = pack_pair(v);
#pragma unroll
        for (int ch = 0; ch < NCH; ++ch) {
          float b[VEC];
          bs[u][ch].widen(b);
          axpy<VEC>(acc[ch], v, vv, b);
        }
      }
    }
    const bool tail_partial = q1 < p1 ? s_row[q1 - nbase] == cur : s_misc[10] != 0;
    if (!tail_partial) {
      flush(cur);
    } else if (cur == first && head_partial) {  // the worker lies inside one row
#pragma unroll
      for (int ch = 0; ch < NCH; ++ch) store_f4<VEC>(slot_ptr(w, ch), acc[ch]);
      if (lane == 0) s_meta[w] = make_int2(cur, kSlotMiddle);
    } else {  // row `cur` began here and continues after this worker
      has_tail = true;
      tail_row = cur;
    }
  }
  __syncthreads();

  // ---- 4. complete rows split between workers -------------------------------
  // A chain is a row's partials in worker order: a start (worker 0's parked
  // partial of the CTA's first row, or a worker's register tail), then parked
  // middles, then possibly a parked head where the row ends.
  auto walk = [&](int row, int from) {  // add the parked pieces of `row` from worker `from` on
    for (int w2 = from; w2 < W; ++w2) {
      const int2 m = s_meta[w2];
      if (m.x != row) return false;  // the row continues past this CTA's nonzeros
#pragma unroll
      for (int ch = 0; ch < NCH; ++ch) {
        float piece[VEC];
        load_f4<VEC>(slot_ptr(w2, ch), piece);
#pragma unroll
        for (int j = 0; j < VEC; ++j) acc[ch][j] += piece[j];
      }
      if (m.y == kSlotHead) return true;
    }
    return false;
  };
  if (w == 0 && s_meta[0].x >= 0) {  // the CTA's first row began before the CTA
    const int2 m0 = s_meta[0];
    float keep[NCH][VEC];  // worker 0 may also hold a register tail
#pragma unroll
    for (int ch = 0; ch < NCH; ++ch)
#pragma unroll
      for (int j = 0; j < VEC; ++j) {
        keep[ch][j] = acc[ch][j];
        acc[ch][j] = 0.f;
      }
    walk(m0.x, 0);
    float* dst = carry + size_t(cta) * 2 * N;  // slot 0: completed by the fixup
#pragma unroll
    for (int ch = 0; ch < NCH; ++ch) {
      if (cok[ch]) store_f4<VEC>(dst + coff[ch], acc[ch]);
#pragma unroll
      for (int j = 0; j < VEC; ++j) acc[ch][j] = keep[ch][j];
    }
  }
  if (has_tail) {
    const bool covers_end = walk(tail_row, w + 1);
    if (covers_end) {
      float* crow = C + size_t(i0 + tail_row) * N;
#pragma unroll
      for (int ch = 0; ch < NCH; ++ch)
        if (cok[ch]) store_c<VEC>(crow + coff[ch], acc[ch]);
    } else {
      float* dst = carry + (size_t(cta) * 2 + 1) * N;  // slot 1: row continues after the CTA
#pragma unroll
      for (int ch = 0; ch < NCH; ++ch)
        if (cok[ch]) store_f4<VEC>(dst + coff[ch], acc[ch]);
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
