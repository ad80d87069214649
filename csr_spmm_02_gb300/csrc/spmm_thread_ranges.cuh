// SpMM for narrow B on merge-path ranges: one thread per slice of the range
// (balanced plans with N <= 2, N = 4 with 16-byte aligned fp32 B and N = 8
// with 16-byte aligned bf16 B).
//
// With N <= 8 a whole output row fits one thread's registers, so the
// merge-path split can go down to threads: each of the CTA's 256 threads
// takes IPT = T / 256 consecutive items (nonzeros and row ends) of its
// range.  This is the per-thread merge-path walk of the nnz-balanced SpMV
// that the Sgap page's related work credits to Yang et al. (the even split of
// nonzeros), with rows ending inside a thread summed in the thread.  The
// lane-group kernels pay a warp butterfly per row end; at N <= 8 a warp step
// covers up to 32 nonzeros and several row ends, and the butterflies dominate.
//
// Per CTA (range [(i0, p0), (i1, p1)) from the plan):
//  1. stage colind, vals and rowptr[i0..i1] in shared memory (bulk copies);
//  2. each thread finds its start (row r0, nonzero n0) and end (r1, n1) by a
//     merge-path search in the staged rowptr; its nonzeros are n0 .. n1-1 and
//     its row ends those of rows r0 .. r1-1, in merged order;
//  3. it gathers the B rows of U nonzeros at a time (all of a batch's loads
//     before any is used, across row ends) and walks its items: a row that
//     started in the thread and ends in it is stored to C; the first row, if
//     it started before the thread, is kept as the thread's head piece; the
//     nonzeros after its last row end form its trailing piece (key: the row);
//  4. a block-wide segmented inclusive scan over the trailing pieces (keyed
//     by row, in thread order) gives each thread the sum of the run of pieces
//     of its trailing row up to itself.  A thread with a head adds its
//     predecessor's scan value if that ends the same row and stores the row --
//     to C if the row started in this range (rowptr[r] >= p0), else to carry
//     slot 0.  The thread holding the range's last item passes a row that
//     continues past the range to carry slot 1 (slot 0 if the range lies
//     inside the row).  The fixup kernel adds the slots of rows split across
//     ranges, as for the balanced kernel.
//
// FusedMM mode (FusedMM section of the Intel Max page, Algorithm 3): the
// value of nonzero (i, j) is the dot product C_i . B_j of two dense fp32
// matrices, computed in the thread (a row of N <= 4 columns is local to it),
// and the gathered rows belong to D; the walk, scan, slots and fixup are the
// same.
//
// The summation order is fixed for a given plan (walk order in a thread, scan
// tree across threads, range order in the fixup): C is bitwise reproducible.
#pragma once

#include <climits>

#include "spmm_device.cuh"
#include "spmm_internal.h"

namespace spmm {

namespace tr {
constexpr int kWarps = kThreads / 32;

// An accumulator's VEC columns to and from plain floats (scan values, shuffles).
template <int VEC>
__device__ __forceinline__ void to_floats(const FVec<VEC>& a, float* out) {
  if constexpr (VEC == 1) {
    out[0] = a.x;
  } else {
#pragma unroll
    for (int j = 0; j < VEC / 2; ++j) {
      out[2 * j] = a.p[j].x;
      out[2 * j + 1] = a.p[j].y;
    }
  }
}
template <int VEC>
__device__ __forceinline__ void from_floats(FVec<VEC>& a, const float* in) {
  if constexpr (VEC == 1) {
    a.x = in[0];
  } else {
#pragma unroll
    for (int j = 0; j < VEC / 2; ++j) a.p[j] = make_float2(in[2 * j], in[2 * j + 1]);
  }
}
}  // namespace tr

__host__ __device__ constexpr size_t thread_ranges_smem_bytes(int T, int VW) {
  return size_t(3) * (T + 8) * 4           // colind, vals, rowptr slices
         + size_t(kThreads) * 4            // trailing-piece keys
         + size_t(kThreads) * VW * 4       // trailing-piece scan values
         + size_t(tr::kWarps) * (VW + 2) * 4  // per-warp run totals, keys, flags
         + 16;                             // mbarrier
}

// VEC columns per load (4: fp32 float4, 8: bf16 uint4, 1: scalar), NCH loads
// per row, so a thread's row holds VW = VEC * NCH >= N columns.
template <typename BT, int VEC, int NCH, bool FUSED = false>
__global__ void __launch_bounds__(kThreads)
    spmm_thread_ranges_kernel(int32_t M, int32_t N, const int32_t* __restrict__ rowptr,
                              const int32_t* __restrict__ colind, const float* __restrict__ vals,
                              const BT* __restrict__ B, float* __restrict__ C, const int2* __restrict__ part,
                              int32_t T, float* __restrict__ carry, int* __restrict__ err,
                              const float* __restrict__ Cd, const float* __restrict__ Bd) {
  // FUSED: B is D (gathered and accumulated), Cd and Bd the dot-product
  // operands, vals unused.
  static_assert(!FUSED || sizeof(BT) == 4, "FusedMM is fp32");
  constexpr int VW = VEC * NCH;
  // nonzeros whose gathered rows are in flight per thread (FusedMM: three
  // slices per nonzero, half as many)
  constexpr int U0 = 8 / NCH > 0 ? 8 / NCH : 1;
  constexpr int U = FUSED ? (U0 / 2 > 0 ? U0 / 2 : 1) : U0;
  constexpr int W = tr::kWarps;

  extern __shared__ __align__(16) unsigned char smem[];
  const int Tpad = T + 8;
  int* s_col = reinterpret_cast<int*>(smem);
  float* s_val = reinterpret_cast<float*>(s_col + Tpad);
  int* s_rp = s_col + 2 * Tpad;
  int* s_key = s_col + 3 * Tpad;                                   // [kThreads]
  float* s_scan = reinterpret_cast<float*>(s_key + kThreads);      // [kThreads][VW]
  float* s_wsum = s_scan + kThreads * VW;                           // [W][VW]
  int* s_wkey = reinterpret_cast<int*>(s_wsum + W * VW);           // [W]
  int* s_wflag = s_wkey + W;                                        // [W]
  uint64_t* s_bar = reinterpret_cast<uint64_t*>(s_wflag + W);

  const int tid = threadIdx.x;
  const int lane = tid & 31, w = tid >> 5;
  const int2 beg = __ldg(part + blockIdx.x);
  const int2 fin = __ldg(part + blockIdx.x + 1);
  const int i0 = beg.x, p0 = beg.y, i1 = fin.x, p1 = fin.y;
  const int nbase = p0 & ~3, rbase = i0 & ~3;
  const uint64_t stream_pol = policy_evict_first();

  // ---- 1. stage the range ----------------------------------------------------
  if (!stage_range<!FUSED>(colind, vals, rowptr, i0, p0, i1, p1, s_col, s_val, s_rp, s_bar, err, [] {})) return;

  // ---- 2. this thread's items -----------------------------------------------
  const int* rp = s_rp + (i0 - rbase);  // rp[r] = rowptr[i0 + r], 0 <= r <= R
  const int R = i1 - i0;                // local row i1 - i0 continues past the range
  const int items = R + (p1 - p0);
  const int ipt = T / kThreads;
  const int d0 = min(tid * ipt, items), d1 = min(d0 + ipt, items);
  auto locate = [&](int d, int& r, int& n) {  // first local row whose end item lies at or after d
    int lo = 0, hi = R;
    while (lo < hi) {
      const int mid = (lo + hi) >> 1;
      if (rp[mid + 1] - p0 + mid >= d) hi = mid; else lo = mid + 1;
    }
    r = lo;
    n = p0 + d - lo;
  };
  int r0, n0, r1, n1;
  locate(d0, r0, n0);
  locate(d1, r1, n1);

  int coff[NCH];  // the row's columns, VEC per load (stores keep those below N)
#pragma unroll
  for (int ch = 0; ch < NCH; ++ch) coff[ch] = ch * VEC;
  const BT* brow0[NCH];
  int cl[NCH];  // the same offsets clamped into the row, for every load
#pragma unroll
  for (int ch = 0; ch < NCH; ++ch) {
    cl[ch] = min(coff[ch], N - VEC);
    brow0[ch] = B + cl[ch];
  }
  float* const crow0 = C + size_t(i0) * N;
  auto store_row = [&](float* dst, const FVec<VEC> (&a)[NCH]) {
#pragma unroll
    for (int ch = 0; ch < NCH; ++ch)
      if (coff[ch] < N) store_c<VEC>(dst + coff[ch], a[ch]);
  };

  // ---- 3. walk: gathers of U nonzeros at a time ------------------------------
  FVec<VEC> acc[NCH], head[NCH];
#pragma unroll
  for (int ch = 0; ch < NCH; ++ch) {
    acc[ch].zero();
    head[ch].zero();
  }
  bool has_head = false;
  int r = r0;
  int next_end = r < R ? rp[r + 1] : INT_MAX;
  int n = n0;
  auto end_row = [&] {  // row r ends: store it, or keep it as the head piece
    if (rp[r] >= n0) {
      store_row(crow0 + size_t(r) * N, acc);
    } else {
#pragma unroll
      for (int ch = 0; ch < NCH; ++ch) head[ch] = acc[ch];
      has_head = true;
    }
#pragma unroll
    for (int ch = 0; ch < NCH; ++ch) acc[ch].zero();
    ++r;
    next_end = r < R ? rp[r + 1] : INT_MAX;
  };
  int rc = r0, rc_end = rc < R ? rp[rc + 1] : INT_MAX;  // FusedMM: the row of the next nonzero to gather
  for (int j0 = n0; j0 < n1; j0 += U) {
    BSlice<BT, VEC> bs[U][NCH];
    using DotSlice = BSlice<float, FUSED ? VEC : 1>;  // FusedMM's dot-product operands (fp32)
    DotSlice bd[FUSED ? U : 1][NCH], cd[FUSED ? U : 1][NCH];
    float v[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {  // gathers first (past n1: the batch's first nonzero again, unused)
      const int j = j0 + u < n1 ? j0 + u : j0;
      const int k = j - nbase;
      const size_t roff = size_t(s_col[k]) * N;
#pragma unroll
      for (int ch = 0; ch < NCH; ++ch) bs[u][ch].load(brow0[ch] + roff);
      if constexpr (FUSED) {
        while (j >= rc_end) {  // rows are non-decreasing along the nonzeros
          ++rc;
          rc_end = rc < R ? rp[rc + 1] : INT_MAX;
        }
        const size_t coffr = size_t(i0 + rc) * N;
#pragma unroll
        for (int ch = 0; ch < NCH; ++ch) {
          bd[u][ch].load(Bd + roff + cl[ch]);
          cd[u][ch].load(Cd + coffr + cl[ch]);
        }
      } else {
        v[u] = s_val[k];
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      if (j0 + u >= n1) break;
      while (n == next_end) end_row();  // rows ending before this nonzero (empty rows too)
      if constexpr (FUSED) {  // the value: C_row . B_col over the row's N columns
        float d = 0.f;
#pragma unroll
        for (int ch = 0; ch < NCH; ++ch) {
          FVec<VEC> x, y;
          bd[u][ch].widen(x);
          cd[u][ch].widen(y);
          float t[VEC], q[VEC];
          tr::to_floats<VEC>(x, t);
          tr::to_floats<VEC>(y, q);
#pragma unroll
          for (int e = 0; e < VEC; ++e)
            if (coff[ch] + e < N) d = fmaf(q[e], t[e], d);
        }
        v[u] = d;
      }
      FVec<VEC> b[NCH];
#pragma unroll
      for (int ch = 0; ch < NCH; ++ch) {
        bs[u][ch].widen(b[ch]);
        acc[ch].fma(pair(v[u]), b[ch]);
      }
      ++n;
    }
  }
  while (r < r1) end_row();  // rows ending after the thread's last nonzero
  // trailing piece: the nonzeros of row r1 in this thread (key -1: none)
  const bool trailing = n1 > max(n0, rp[r1]);
  const int key = trailing ? r1 : -1;

  // ---- 4. segmented scan of the trailing pieces, in thread order -------------
  s_key[tid] = key;
  __syncthreads();
  bool flag = tid == 0 || s_key[tid - 1] != key;  // a run of equal keys starts here
  float sv[VW];
#pragma unroll
  for (int ch = 0; ch < NCH; ++ch) tr::to_floats<VEC>(acc[ch], sv + ch * VEC);
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {  // warp: (f, v) = (f_left | f, f ? v : v_left + v)
    const bool f_up = __shfl_up_sync(0xffffffffu, flag, o);
    float up[VW];
#pragma unroll
    for (int e = 0; e < VW; ++e) up[e] = __shfl_up_sync(0xffffffffu, sv[e], o);
    if (lane >= o) {
      if (!flag) {
#pragma unroll
        for (int e = 0; e < VW; ++e) sv[e] = up[e] + sv[e];
      }
      flag = flag || f_up;
    }
  }
  if (lane == 31) {
    s_wkey[w] = key;
    s_wflag[w] = flag;
#pragma unroll
    for (int e = 0; e < VW; ++e) s_wsum[w * VW + e] = sv[e];
  }
  __syncthreads();
  if (tid == 0) {  // runs that cross warps: warp w's last run continues warp w-1's
    for (int w2 = 1; w2 < W; ++w2)
      if (!s_wflag[w2] && s_wkey[w2] == s_wkey[w2 - 1])
        for (int e = 0; e < VW; ++e) s_wsum[w2 * VW + e] = s_wsum[(w2 - 1) * VW + e] + s_wsum[w2 * VW + e];
  }
  __syncthreads();
  if (w > 0 && !flag && key == s_wkey[w - 1]) {  // this thread's run began in an earlier warp
#pragma unroll
    for (int e = 0; e < VW; ++e) sv[e] = s_wsum[(w - 1) * VW + e] + sv[e];
  }
#pragma unroll
  for (int e = 0; e < VW; ++e) s_scan[tid * VW + e] = sv[e];
  __syncthreads();

  // a head completes the row whose pieces end at the previous thread
  if (has_head) {
    FVec<VEC> total[NCH];
    if (tid > 0 && s_key[tid - 1] == r0) {
#pragma unroll
      for (int ch = 0; ch < NCH; ++ch) {
        tr::from_floats<VEC>(total[ch], s_scan + (tid - 1) * VW + ch * VEC);
        total[ch].add(head[ch]);
      }
    } else {
#pragma unroll
      for (int ch = 0; ch < NCH; ++ch) total[ch] = head[ch];
    }
    if (rp[r0] >= p0) {
      store_row(crow0 + size_t(r0) * N, total);
    } else {  // the range's first row began in an earlier range
#pragma unroll
      for (int ch = 0; ch < NCH; ++ch)
        if (coff[ch] < N) total[ch].store_plain(carry + size_t(blockIdx.x) * 2 * N + coff[ch]);
    }
  }
  // the thread holding the range's last item: a row that continues past the range
  if (items > 0 && d1 == items && d0 < d1 && key == R) {
    FVec<VEC> total[NCH];
#pragma unroll
    for (int ch = 0; ch < NCH; ++ch) tr::from_floats<VEC>(total[ch], sv + ch * VEC);
    const int slot = rp[R] >= p0 ? 1 : 0;  // 0: the whole range lies inside the row
#pragma unroll
    for (int ch = 0; ch < NCH; ++ch)
      if (coff[ch] < N) total[ch].store_plain(carry + (size_t(blockIdx.x) * 2 + slot) * N + coff[ch]);
  }
}

template <typename BT, int VEC, int NCH, bool FUSED = false>
cudaError_t launch_thread_ranges_t(const Launch& L, const float* Cd = nullptr, const float* Bd = nullptr) {
  constexpr int VW = VEC * NCH;
  const size_t smem = thread_ranges_smem_bytes(L.items_per_cta, VW);
  static bool attr_set[kMaxDevices] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= kMaxDevices || !attr_set[dev]) {
    e = cudaFuncSetAttribute(spmm_thread_ranges_kernel<BT, VEC, NCH, FUSED>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             int(thread_ranges_smem_bytes(kMaxItemsPerCta, VW)));
    if (e != cudaSuccess) return e;
    if (dev < kMaxDevices) attr_set[dev] = true;
  }
  SPMM_DEBUG_RANGES(L.stream, L.err,
                    {{L.B, size_t(L.K) * L.N * sizeof(BT)}, {Cd, FUSED ? size_t(L.M) * L.N * 4 : 0},
                     {Bd, FUSED ? size_t(L.K) * L.N * 4 : 0}},
                    {{L.C, size_t(L.M) * L.N * 4}, {L.carry, size_t(L.num_ctas) * 2 * L.N * 4}});
  spmm_thread_ranges_kernel<BT, VEC, NCH, FUSED><<<unsigned(L.num_ctas), kThreads, smem, L.stream>>>(
      L.M, L.N, L.rowptr, L.colind, L.vals, static_cast<const BT*>(L.B), L.C, L.part, L.items_per_cta, L.carry,
      L.err, Cd, Bd);
  return cudaGetLastError();
}

}  // namespace spmm
