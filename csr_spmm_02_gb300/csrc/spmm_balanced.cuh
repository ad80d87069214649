// nnz-balanced (merge-path) SpMM kernel.
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
// computes these coordinates once per CTA (spmm_plan.cu).
//
// One CTA per range [(i0, p0), (i1, p1)) of T items:
//  1. stages the range's colind and vals and rowptr[i0..i1] in shared memory
//     with 1-D bulk copies (the TMA engine; the ESIMD kernel's chunked
//     colind/vals loads and prefetch, Figs. 8-10 of the Intel Max page, and the
//     coalesced row caching the Sgap page cites from Ge-SpMM), plain loads for
//     the unaligned ends;
//  2. cuts the range again into one sub-range per warp with the same search
//     in shared memory, a row end weighing as much as the nonzeros of two
//     warp steps (the work it costs a warp).  A warp is one worker: its 32 lanes form S = 32/G
//     groups of G lanes, each lane owning NCH 16-byte chunks of the output
//     row; a step gives S consecutive nonzeros to the S groups (Sgap's
//     {<1 nnz, c col>, r = S} point), so every branch is uniform in the warp;
//  3. per batch, issues the gathers of U steps, then accumulates with packed
//     FMAs.  Where a row ends inside a step, each group only adds the nonzeros
//     on its side of the end (value 0 otherwise: zero extension), and the S
//     groups' partial rows are combined by a shuffle butterfly in a fixed
//     order -- the warp-shuffle segmented reduction keyed by row -- before
//     group 0 stores the finished C row with a streaming store.  Rows the warp
//     entered mid-way (head) or that lie across the whole warp (middle) are
//     parked in shared memory; the row it leaves unfinished stays in registers;
//  4. after a barrier, each row's pieces are summed in warp order: rows that
//     lie inside the CTA go to C, the CTA's first and last rows to its carry
//     slots 0 and 1, which the fixup kernel adds across CTAs in CTA order.
//
// FusedMM mode (same page, FusedMM section, Fig. 6, Algorithm 3, Fig. 11):
// the sparse value of each nonzero (i, j) is not read from vals but computed
// as the SDDMM dot product C_i . B_j of two dense fp32 matrices, and the
// gathered rows belong to a third matrix D.  After staging, the CTA computes
// the values of all its nonzeros into the shared-memory slots that vals
// would fill (the SDDMM kernel's rounds, spmm_sddmm.cuh, with the SDDMM
// kernel's lane shape for the width), then streams the range exactly as for
// SpMM; the values never leave the CTA.
//
// No floating-point atomics anywhere, so C is bitwise reproducible for a given
// plan.
#pragma once

#include <climits>

#include "spmm_device.cuh"
#include "spmm_internal.h"
#include "spmm_sddmm.cuh"

#ifndef SPMM_BAL_LOADS
#define SPMM_BAL_LOADS 8  // 16-byte B loads in flight per lane (U steps x NCH chunks)
#endif
#ifndef SPMM_BAL_MIN_BLOCKS
#define SPMM_BAL_MIN_BLOCKS 4  // resident CTAs asked of the compiler (fp32, one chunk per lane)
#endif
#ifndef SPMM_BAL_ROW_WEIGHT
#define SPMM_BAL_ROW_WEIGHT 0  // items a row end counts for in the warps' split (0: by shape, below)
#endif


namespace spmm {

// Kinds of a warp's parked partial row (its shared-memory slot).
constexpr int kSlotHead = 1;    // the row began before the warp and ends in it
constexpr int kSlotMiddle = 2;  // the warp lies entirely inside the row

template <int NCH>
struct BalancedSteps {
  static constexpr int value = SPMM_BAL_LOADS / NCH > 0 ? SPMM_BAL_LOADS / NCH : 1;
};

// FusedMM's value pass: the lane shape the SDDMM kernel takes for the same
// width (fewer lanes per dot product, each with more of the row).
template <int VEC, int G, int NCH>
struct FusedValueShape {
  static constexpr bool narrow = VEC == 4 && NCH == 1 && (G == 8 || G == 16 || G == 32);
  static constexpr int g = !narrow ? G : G == 8 ? 4 : 8;
  static constexpr int nch = !narrow ? NCH : G == 8 ? 2 : G / 8;
};

// The 64-register budget of 4 resident CTAs fits the fp32 one-chunk SpMM
// shapes without spills; wider or bf16 lanes keep the compiler's choice.
// FusedMM (value pass and walk in one kernel): 4 CTAs for 8-lane groups
// (rmat22, N = 32: 1,974 -> 1,840 us against 3 CTAs), 3 of 80 registers for
// the other one-chunk shapes (rmat20, N = 128: 1,424 -> 1,416 us; its pattern
// at N = 64: 817 -> 790 us), no spills there.
template <typename BT, int G, int NCH, bool FUSED>
struct BalancedMinBlocks {
  static constexpr int fused = G == 8 ? 4 : 3;
  static constexpr int value = (sizeof(BT) == 4 && NCH == 1) ? (FUSED ? fused : SPMM_BAL_MIN_BLOCKS) : 1;
};

__host__ __device__ constexpr size_t balanced_smem_layout_bytes(int W, int TW, int T) {
  return size_t(3) * (T + 8) * 4   // colind, vals, rowptr slices
         + size_t(1) * W * TW * 4  // one parked partial row per warp
         + size_t(1) * W * 8       // slot metadata (local row, kind)
         + 16;                     // mbarrier
}

template <typename BT, int VEC, int G, int NCH, bool FUSED, int SR>
__global__ void __launch_bounds__(kThreads, BalancedMinBlocks<BT, G, NCH, FUSED>::value)
    spmm_balanced_kernel(int32_t M, int32_t N, const int32_t* __restrict__ rowptr,
                         const int32_t* __restrict__ colind, const float* __restrict__ vals,
                         const BT* __restrict__ B, float* __restrict__ C,
                         const int2* __restrict__ part, int32_t T, float* __restrict__ carry,
                         int* __restrict__ err, const float* __restrict__ Cd, const float* __restrict__ Bd) {
  // FUSED: B is D (gathered and accumulated), Cd and Bd the SDDMM operands, vals
  // unused (its staging area holds the local row ids, then the computed values).
  // SR: semiring code (spmm_device.cuh); 0 = ordinary SpMM.
  static_assert(!FUSED || sizeof(BT) == 4, "FusedMM is fp32");
  static_assert(SR == 0 || (!FUSED && sizeof(BT) == 4), "semirings: fp32 SpMM only");
  constexpr int S = 32 / G;                // nonzeros per warp step
  constexpr int W = kThreads / 32;         // warps (workers) per CTA
  constexpr int TW = G * VEC * NCH;        // columns per tile
  constexpr int U = BalancedSteps<NCH>::value;  // steps per batch

  extern __shared__ __align__(16) unsigned char smem[];
  const int Tpad = T + 8;
  int* s_col = reinterpret_cast<int*>(smem);
  float* s_val = reinterpret_cast<float*>(s_col + Tpad);
  int* s_rp = s_col + 2 * Tpad;
  float* s_slot = reinterpret_cast<float*>(s_col + 3 * Tpad);  // [W][TW]
  int2* s_meta = reinterpret_cast<int2*>(s_slot + W * TW);     // [W] (local row, kind)
  uint64_t* s_bar = reinterpret_cast<uint64_t*>(s_meta + W);

  const int tid = threadIdx.x;
  const int cta = blockIdx.x;
  const int2 beg = __ldg(part + cta);
  const int2 fin = __ldg(part + cta + 1);
  const int i0 = beg.x, p0 = beg.y, i1 = fin.x, p1 = fin.y;
  const int nbase = p0 & ~3;  // s_col[k], s_val[k] hold nonzero nbase + k
  const int rbase = i0 & ~3;  // s_rp[k] holds rowptr[rbase + k]; rows i0..i1 are staged
  const uint64_t stream_pol = policy_evict_first();

  // ---- 1. stage the range -------------------------------------------------
  if (!stage_range<!FUSED>(colind, vals, rowptr, i0, p0, i1, p1, s_col, s_val, s_rp, s_bar, err,
                           [&] { for (int k = tid; k < W; k += kThreads) s_meta[k] = make_int2(-1, 0); }))
    return;
  const int w = tid >> 5;
  const int lane = tid & 31;
  const int grp = lane / G;       // which nonzero of a step this lane's group takes
  const int gl = lane & (G - 1);  // lane within its group
  const int* rp = s_rp + (i0 - rbase);  // rp[r] = rowptr[i0 + r], 0 <= r <= i1 - i0
  // FusedMM: the value of every staged nonzero.  The local row ids go into the
  // value slots first; each warp's rounds read the ids of their nonzeros
  // before storing the values over them.
  if constexpr (FUSED) {
    int* const s_row = reinterpret_cast<int*>(s_val);
    fill_row_ids(rp, i1 - i0, p0, p1, nbase, s_row);
    using VS = FusedValueShape<VEC, G, NCH>;
    sddmm_rounds<VEC, VS::g, VS::nch>(N, s_col, s_row, nbase, p0, p1, Cd + size_t(i0) * N, Bd, w, lane,
                                      [&](int n, float x) { s_val[n - nbase] = x; });
    __syncthreads();
  }
  // Column indices become the offsets of their B (FusedMM: D) rows in
  // VEC-element units (c * N / VEC < 2^32, which the launch checks), so that a
  // gather's address is one multiply-add on a 32-bit offset (rmat22 826 -> 818
  // us, rmat20 543 -> 525 us).
  {
    const uint32_t nv = uint32_t(N / VEC);
    for (int k = p0 - nbase + tid; k < p1 - nbase; k += kThreads) s_col[k] = int(uint32_t(s_col[k]) * nv);
    __syncthreads();
  }

  // ---- 2. this warp's sub-range ---------------------------------------------
  // The warps split the range's merged sequence with each row end counted as
  // kRowWeight items: row r's end sits at cost E(r) = (rowptr[r+1] - p0) +
  // kRowWeight * r, and a warp starting at cost c begins at the first row with
  // E(r) >= c and at the nonzeros of that row whose cost lies below c.  A row
  // end costs a warp about two steps (its butterfly and store) and a step
  // takes S nonzeros, so a row end weighs 2S nonzeros (capped at 16; measured
  // best on rmat22 at S = 4 and rmat20 at S = 1).
  constexpr int kRowWeight = SPMM_BAL_ROW_WEIGHT > 0 ? SPMM_BAL_ROW_WEIGHT : (2 * S < 16 ? 2 * S : 16);
  const int cost = (p1 - p0) + kRowWeight * (i1 - i0);
  auto find_row = [&](int c) {  // first local row whose end costs c or more
    int lo = 0, hi = i1 - i0;
    while (lo < hi) {
      const int mid = (lo + hi) >> 1;
      if (rp[mid + 1] - p0 + kRowWeight * mid >= c) hi = mid; else lo = mid + 1;
    }
    return lo;
  };
  auto nz_start = [&](int c, int r) {  // first nonzero of the warp starting at cost c in row r
    const int hi = r < i1 - i0 ? rp[r + 1] : p1;
    return p0 + min(max(c - kRowWeight * r, rp[r] - p0), hi - p0);
  };
  const int c0 = int((int64_t(cost) * w) / W), c1 = int((int64_t(cost) * (w + 1)) / W);
  const int rw0 = find_row(c0), rw1 = find_row(c1);
  const int pw0 = nz_start(c0, rw0), pw1 = nz_start(c1, rw1);

  const int col0 = blockIdx.y * TW;
  int coff[NCH];
  const BT* bl[NCH];  // this lane's slice of B row 0 (clamped into the row); row c is bl[ch] + c*N
#pragma unroll
  for (int ch = 0; ch < NCH; ++ch) {
    coff[ch] = col0 + (ch * G + gl) * VEC;
    bl[ch] = B + min(coff[ch], N - VEC);
  }
  const int* colw = s_col - nbase + grp;  // colw[a] = colind of nonzero a + grp (staged)
  const float* valw = s_val - nbase + grp;
  auto slot_ptr = [&](int worker, int ch) { return s_slot + worker * TW + (ch * G + gl) * VEC; };
  FVec<VEC> acc[NCH];
  auto reset = [&](FVec<VEC>& a) {
    if constexpr (SR == 0) a.zero(); else sr_reset<SR>(a);
  };
  // acc (+)= v (x) b for a slot that holds a nonzero of the current row (ok),
  // unchanged otherwise (ordinary SpMM: v is already 0 for such slots)
  auto apply = [&](FVec<VEC>& a, float v, bool ok, const FVec<VEC>& b) {
    if constexpr (SR == 0) a.fma(pair(ok ? v : 0.f), b); else sr_apply<SR>(a, v, b, ok);
  };
#pragma unroll
  for (int ch = 0; ch < NCH; ++ch) reset(acc[ch]);
  // Combine the S groups' partial rows: afterwards every group holds the sum.
  auto butterfly = [&] {
#pragma unroll
    for (int o = G; o < 32; o <<= 1)
#pragma unroll
      for (int ch = 0; ch < NCH; ++ch) {
        if constexpr (SR == 0) acc[ch].add_shfl_xor(o); else sr_combine_shfl_xor<SR>(acc[ch], o);
      }
  };
  auto store_row = [&](float* dst) {  // group 0 writes the row slice (streaming)
    if (grp == 0) {
#pragma unroll
      for (int ch = 0; ch < NCH; ++ch)
        if (coff[ch] < N) store_c<VEC>(dst + coff[ch], acc[ch]);
    }
  };
  auto park = [&](int r, int kind) {
    if (grp == 0) {
#pragma unroll
      for (int ch = 0; ch < NCH; ++ch) acc[ch].store_plain(slot_ptr(w, ch));
    }
    if (lane == 0) s_meta[w] = make_int2(r, kind);
  };

  // ---- 3. stream the sub-range --------------------------------------------
  int r = rw0;
  bool began_before = rp[r] < pw0;
  int next_end = r < rw1 ? rp[r + 1] : INT_MAX;
  float* const crow0 = C + size_t(i0) * N;
  // Row r ends: finish it (all warp-uniform).
  auto end_row = [&] {
    if (rp[r] != rp[r + 1]) {  // an empty row's accumulators are still zero
      butterfly();
      if (began_before) park(r, kSlotHead); else store_row(crow0 + size_t(r) * N);
#pragma unroll
      for (int ch = 0; ch < NCH; ++ch) reset(acc[ch]);
    } else {
      store_row(crow0 + size_t(r) * N);
    }
    ++r;
    began_before = false;
    next_end = r < rw1 ? rp[r + 1] : INT_MAX;
  };
  // One step: the S groups take nonzeros a .. a+S-1 (group grp: n = a + grp,
  // value v, B slice b); rows ending inside the step are completed in order.
  auto step = [&](int a, float v, bool ok, const BSlice<BT, VEC> (&bs)[NCH]) {
    FVec<VEC> b[NCH];
#pragma unroll
    for (int ch = 0; ch < NCH; ++ch) bs[ch].widen(b[ch]);
    const int n = a + grp;
    int lo = a;
    // (ordinary SpMM: slots without a nonzero of the row carry v = 0, so the
    // row test alone masks them; other semirings also need `ok`)
    while (next_end <= a + S) {  // a row ends inside (or right after) this step
      const bool in = (SR == 0 || ok) && n >= lo && n < next_end;
#pragma unroll
      for (int ch = 0; ch < NCH; ++ch) apply(acc[ch], v, in, b[ch]);
      lo = next_end;
      end_row();
    }
    const bool in = (SR == 0 || ok) && n >= lo;
#pragma unroll
    for (int ch = 0; ch < NCH; ++ch) apply(acc[ch], v, in, b[ch]);
  };
  int q = pw0;
  for (; q + U * S <= pw1; q += U * S) {  // full batches
    BSlice<BT, VEC> bs[U][NCH];
#pragma unroll
    for (int s = 0; s < U; ++s) {  // gathers first
      const size_t roff = size_t(uint32_t(colw[q + s * S])) * VEC;
#pragma unroll
      for (int ch = 0; ch < NCH; ++ch) bs[s][ch].load(bl[ch] + roff);
    }
    auto value = [&](int s) { return valw[q + s * S]; };
    if (next_end > q + U * S) {  // no row ends inside the batch
#pragma unroll
      for (int s = 0; s < U; ++s) {
        const float2 vv = pair(value(s));
#pragma unroll
        for (int ch = 0; ch < NCH; ++ch) {
          FVec<VEC> b;
          bs[s][ch].widen(b);
          if constexpr (SR == 0) acc[ch].fma(vv, b); else sr_apply<SR>(acc[ch], value(s), b, true);
        }
      }
    } else {
#pragma unroll
      for (int s = 0; s < U; ++s) step(q + s * S, value(s), true, bs[s]);
    }
  }
  if (q < pw1) {  // short last batch: slots past the sub-range re-read its last nonzero's row, value 0
    BSlice<BT, VEC> bs[U][NCH];
#pragma unroll
    for (int s = 0; s < U; ++s) {
      const int c = colw[min(q + s * S, pw1 - 1 - grp)];
      const size_t roff = size_t(uint32_t(c)) * VEC;
#pragma unroll
      for (int ch = 0; ch < NCH; ++ch) bs[s][ch].load(bl[ch] + roff);
    }
#pragma unroll
    for (int s = 0; s < U; ++s) {
      const int a = q + s * S;
      if (a >= pw1) break;
      const bool ok = a + grp < pw1;
      const float v = ok ? valw[a] : 0.f;
      step(a, v, ok, bs[s]);
    }
  }
  while (r < rw1) end_row();  // rows ending exactly at the sub-range end (empty rows too)
  bool has_tail = false;
  const int tail_row = r;
  if (i0 + r < M && rp[r] < pw1) {  // row r continues after this warp
    butterfly();
    if (began_before) park(r, kSlotMiddle); else has_tail = true;
  }
  __syncthreads();

  // ---- 4. complete rows split between warps ---------------------------------
  auto walk = [&](int row, int from) {  // add the parked pieces of `row` from warp `from` on
    for (int w2 = from; w2 < W; ++w2) {
      const int2 m = s_meta[w2];
      if (m.x != row) return false;  // the row continues past this CTA's nonzeros
#pragma unroll
      for (int ch = 0; ch < NCH; ++ch) {
        FVec<VEC> piece;
        piece.load_plain(slot_ptr(w2, ch));
        if constexpr (SR == 0) acc[ch].add(piece); else sr_combine<SR>(acc[ch], piece);
      }
      if (m.y == kSlotHead) return true;
    }
    return false;
  };
  if (w == 0 && s_meta[0].x >= 0) {  // the CTA's first row began before the CTA
    FVec<VEC> keep[NCH];             // warp 0 may also hold a register tail
#pragma unroll
    for (int ch = 0; ch < NCH; ++ch) {
      keep[ch] = acc[ch];
      reset(acc[ch]);
    }
    walk(s_meta[0].x, 0);
    store_row(carry + size_t(cta) * 2 * N);  // slot 0: completed by the fixup
#pragma unroll
    for (int ch = 0; ch < NCH; ++ch) acc[ch] = keep[ch];
  }
  if (has_tail) {
    if (walk(tail_row, w + 1)) store_row(crow0 + size_t(tail_row) * N);
    else store_row(carry + (size_t(cta) * 2 + 1) * N);  // slot 1: row continues after the CTA
  }
}

template <typename BT, int VEC, int G, int NCH, bool FUSED = false, int SR = 0>
cudaError_t launch_balanced_t(const Launch& L, const float* Cd = nullptr, const float* Bd = nullptr) {
  constexpr int W = kThreads / 32;
  constexpr int TW = G * VEC * NCH;
  const size_t smem = balanced_smem_layout_bytes(W, TW, L.items_per_cta);
  static bool attr_set[kMaxDevices] = {};  // per instantiation and device
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= kMaxDevices || !attr_set[dev]) {
    e = cudaFuncSetAttribute(spmm_balanced_kernel<BT, VEC, G, NCH, FUSED, SR>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             int(balanced_smem_layout_bytes(W, TW, kMaxItemsPerCta)));
    if (e != cudaSuccess) return e;
    if (dev < kMaxDevices) attr_set[dev] = true;
  }
  // B-row offsets are kept in 32 bits (VEC-element units): column c's row
  // starts c * N / VEC vectors into B (D for FusedMM).
  if (int64_t(L.K) * (L.N / VEC) > int64_t(UINT32_MAX)) return cudaErrorNotSupported;
  const dim3 grid(unsigned(L.num_ctas), unsigned((L.N + TW - 1) / TW));
  SPMM_DEBUG_RANGES(L.stream, L.err,
                    {{L.B, size_t(L.K) * L.N * sizeof(BT)}, {Cd, FUSED ? size_t(L.M) * L.N * 4 : 0},
                     {Bd, FUSED ? size_t(L.K) * L.N * 4 : 0}},
                    {{L.C, size_t(L.M) * L.N * 4}, {L.carry, size_t(L.num_ctas) * 2 * L.N * 4}});
  spmm_balanced_kernel<BT, VEC, G, NCH, FUSED, SR><<<grid, kThreads, smem, L.stream>>>(
      L.M, L.N, L.rowptr, L.colind, L.vals, static_cast<const BT*>(L.B), L.C, L.part,
      L.items_per_cta, L.carry, L.err, Cd, Bd);
  return cudaGetLastError();
}

}  // namespace spmm
