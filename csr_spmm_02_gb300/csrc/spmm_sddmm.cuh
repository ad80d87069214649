// SDDMM on the CSR pattern of A: out[p] = C_i . B_j for every stored (i, j).
//
// The SDDMM section of "Performance Optimization of Deep Learning Sparse
// Matrix Kernels on Intel Max Series GPU" (Algorithm 1, Figs. 3-4, 7) assigns
// each row of the sparse output to one or more work-items (NT per row), keeps
// the row C_i in registers and produces every nonzero of the row as a dot
// product with the row B_j it selects.  Here the nonzeros of a CTA come from
// the same merge-path ranges as the SpMM kernels, and the work is laid out for
// a warp rather than for a row:
//
//  * the CTA stages its colind and rowptr slices in shared memory and writes
//    the (local) row of every staged nonzero next to its column, so a lane
//    finds both rows of a dot product with two shared loads, without a walk;
//  * a warp takes rounds of 32 consecutive nonzeros; its S = 32/G lane groups
//    take every S-th one, each lane holding VEC*NCH columns of both operands
//    (16-byte loads; the C row is re-read per nonzero and is an L1 hit while
//    the row lasts, so no load waits on a row change; a round that lies in
//    one row loads it once);
//  * a lane keeps the partial dot products of G nonzeros and the group sums
//    them with a transposed butterfly: G-1 shuffles for G results instead of
//    log2(G) per result, after which lane l of the group holds nonzero l's
//    value and the warp stores its 32 values with one coalesced store.
//
// Each output is written once; no reduction crosses lanes of different
// nonzeros or CTAs, and the summation order is fixed (deterministic).
#pragma once

#include <climits>

#include "spmm_device.cuh"
#include "spmm_internal.h"

#ifndef SPMM_SDDMM_LOADS
#define SPMM_SDDMM_LOADS 4  // nonzeros whose operand rows a lane has in flight (per chunk)
#endif
#ifndef SPMM_SDDMM_LOADS_WIDE
#define SPMM_SDDMM_LOADS_WIDE 2  // the same for 32-lane groups (each lane already keeps 32 partial sums)
#endif
#ifndef SPMM_SDDMM_MIN_BLOCKS
#define SPMM_SDDMM_MIN_BLOCKS 4  // resident CTAs asked of the compiler (64 registers; a few spill)
#endif

namespace spmm {

__host__ __device__ constexpr size_t sddmm_smem_layout_bytes(int T) {
  return size_t(3) * (T + 8) * 4 + 16;  // colind, row ids, rowptr slices; mbarrier
}

// Local row of every staged nonzero n in [p0, p1): the largest r <= last_row
// with rp[r] <= n (rows with no nonzeros are skipped by that rule).  Each
// thread takes one run of consecutive nonzeros (an odd run length, so the
// threads' runs start in distinct banks), finds the row of its first one by
// binary search and walks the row ends from there.  Ends with a CTA barrier.
__device__ __forceinline__ void fill_row_ids(const int* rp, int last_row, int p0, int p1, int nbase, int* s_row) {
  const int count = p1 - p0;
  int per = (count + kThreads - 1) / kThreads;
  if (per > 0 && (per & 1) == 0) ++per;
  const int k0 = min(int(threadIdx.x) * per, count), k1 = min(k0 + per, count);
  if (k0 < k1) {
    const int n0 = p0 + k0;
    int lo = 0, hi = last_row;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (rp[mid] <= n0) lo = mid; else hi = mid - 1;
    }
    int r = lo;
    int next = r < last_row ? rp[r + 1] : INT_MAX;  // first nonzero after row r
#pragma unroll 1
    for (int n = n0; n < p0 + k1; ++n) {
      while (n >= next) {  // row r ended (empty rows end at once)
        ++r;
        next = r < last_row ? rp[r + 1] : INT_MAX;
      }
      s_row[n - nbase] = r;
    }
  }
  __syncthreads();
}

// A lane's share of one dot product over its NCH chunks; chunks whose columns
// lie past N (their loads were clamped into the row) contribute nothing.
template <int VEC, int NCH>
__device__ __forceinline__ float dot_lane(const FVec<VEC> (&c)[NCH], const FVec<VEC> (&b)[NCH],
                                          const bool (&valid)[NCH]) {
  if constexpr (VEC == 1) {
    float d = 0.f;
#pragma unroll
    for (int ch = 0; ch < NCH; ++ch) d = valid[ch] ? fmaf(c[ch].x, b[ch].x, d) : d;
    return d;
  } else {
    float2 t = make_float2(0.f, 0.f);
#pragma unroll
    for (int ch = 0; ch < NCH; ++ch) {
      float2 u = __fmul2_rn(c[ch].p[0], b[ch].p[0]);
#pragma unroll
      for (int j = 1; j < VEC / 2; ++j) u = __ffma2_rn(c[ch].p[j], b[ch].p[j], u);
      t = valid[ch] ? __fadd2_rn(t, u) : t;
    }
    return t.x + t.y;
  }
}

// Dot-product share of a lane over the column tiles after the first (rows
// wider than one tile of G*VEC*NCH columns); loads are not batched.
template <int VEC, int G, int NCH>
__device__ __forceinline__ float dot_tail_tiles(const float* crow, const float* brow, int N, int gl) {
  constexpr int TW = G * VEC * NCH;
  float d = 0.f;
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
    d += dot_lane<VEC, NCH>(c, b, valid);
  }
  return d;
}

// Group sums of P partial values per lane (P <= G, both powers of two): on
// return every lane gl holds the sum over its G-lane group of v[gl % P].
// Offsets >= P are plain butterfly levels on all P values; the last log2(P)
// levels are transposed: a lane sends the half of its values that its partner
// keeps, so they cost P-1 shuffles in all.  Every lane of the warp takes part.
template <int G, int P>
__device__ __forceinline__ float group_reduce_transposed(float (&v)[P], int gl) {
  static_assert(P <= G && (P & (P - 1)) == 0 && (G & (G - 1)) == 0, "powers of two, P <= G");
#pragma unroll
  for (int o = G / 2; o >= P; o >>= 1)
#pragma unroll
    for (int i = 0; i < P; ++i) v[i] += __shfl_xor_sync(0xffffffffu, v[i], o);
#pragma unroll
  for (int o = P / 2; o >= 1; o >>= 1) {
    const bool upper = (gl & o) != 0;
#pragma unroll
    for (int i = 0; i < o; ++i) {
      const float send = upper ? v[i] : v[i + o];
      const float keep = upper ? v[i + o] : v[i];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
    }
  }
  return v[0];
}

// The dot products of one round of R steps (S = 32/G nonzeros each) starting
// at nonzero base.  ONE_ROW: all of the round's nonzeros lie in one row (long
// rows), so each lane loads its C slice once for the round instead of once per
// nonzero.
template <int VEC, int G, int NCH, int U, int R, bool ONE_ROW>
__device__ __forceinline__ void sddmm_round_dots(int base, int p1, int nbase, const int* s_col, const int* s_row, int N,
                                                 const float* __restrict__ B, const float* __restrict__ Crow0,
                                                 const int (&coffl)[NCH], const bool (&valid)[NCH], int grp, int gl,
                                                 float (&dots)[R]) {
  constexpr int S = 32 / G;
  FVec<VEC> crow[NCH];
  if constexpr (ONE_ROW) {
    const size_t coff = size_t(s_row[base - nbase]) * N;
#pragma unroll
    for (int ch = 0; ch < NCH; ++ch) {
      BSlice<float, VEC> x;
      x.load(Crow0 + coff + coffl[ch]);
      x.widen(crow[ch]);
    }
  }
#pragma unroll
  for (int s0 = 0; s0 < R; s0 += U) {
    BSlice<float, VEC> bs[U][NCH], cs[ONE_ROW ? 1 : U][NCH];
    int ks[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {  // gathers first: both operand rows of U nonzeros
      const int k = min(base + (s0 + u) * S + grp, p1 - 1) - nbase;
      ks[u] = k;
      const size_t boff = size_t(s_col[k]) * N;
#pragma unroll
      for (int ch = 0; ch < NCH; ++ch) bs[u][ch].load(B + boff + coffl[ch]);
      if constexpr (!ONE_ROW) {
        const size_t coff = size_t(s_row[k]) * N;
#pragma unroll
        for (int ch = 0; ch < NCH; ++ch) cs[u][ch].load(Crow0 + coff + coffl[ch]);
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      FVec<VEC> b[NCH], c[NCH];
#pragma unroll
      for (int ch = 0; ch < NCH; ++ch) {
        bs[u][ch].widen(b[ch]);
        if constexpr (ONE_ROW) c[ch] = crow[ch]; else cs[u][ch].widen(c[ch]);
      }
      float d = dot_lane<VEC, NCH>(c, b, valid);
      if (N > G * VEC * NCH)
        d += dot_tail_tiles<VEC, G, NCH>(Crow0 + size_t(s_row[ks[u]]) * N, B + size_t(s_col[ks[u]]) * N, N, gl);
      dots[s0 + u] = d;
    }
  }
}

// The dot products of the staged nonzeros [p0, p1): nonzero n (staged at
// n - nbase with column s_col and local row s_row) gets C_row . B_col, handed to
// store(n, value).  Warp w takes rounds of 32 consecutive nonzeros (R steps of
// S = 32/G, every S-th to each lane group), loads both operand rows of U steps
// at a time and sums each group's partial products by the transposed
// butterfly, after which lane l of a group holds nonzero l's value.  All of a
// round's s_col / s_row reads come before its first store, and a warp reads
// only its own rounds' entries, so store may overwrite them.
template <int VEC, int G, int NCH, typename Store>
__device__ __forceinline__ void sddmm_rounds(int N, const int* s_col, const int* s_row, int nbase, int p0, int p1,
                                             const float* __restrict__ Crow0, const float* __restrict__ B, int w,
                                             int lane, Store store) {
  constexpr int S = 32 / G;                     // nonzeros per warp step
  constexpr int W = kThreads / 32;
  constexpr int kLoads = G >= 32 ? SPMM_SDDMM_LOADS_WIDE : SPMM_SDDMM_LOADS;
  constexpr int U = kLoads / NCH > 0 ? kLoads / NCH : 1;  // steps per load batch
  constexpr int R = G > U ? G : U;              // steps per warp iteration
  constexpr int NPI = R * S;                    // nonzeros per warp iteration
  static_assert(R % U == 0 && R % G == 0, "powers of two");
  const int grp = lane / G, gl = lane & (G - 1);
  int coffl[NCH];
  bool valid[NCH];
#pragma unroll
  for (int ch = 0; ch < NCH; ++ch) {
    const int col = (ch * G + gl) * VEC;  // first column tile
    valid[ch] = col < N;
    coffl[ch] = min(col, N - VEC);
  }
  for (int base = p0 + w * NPI; base < p1; base += W * NPI) {
    float dots[R];
    // Rows are non-decreasing along the nonzeros: first == last means one row
    // (warp-uniform).  Groups of 8 and 16 lanes take the one-row form (rmat22
    // 1,029 -> 980 us at N = 32, rmat20 554 -> 525 us at N = 64); 32-lane
    // groups keep one form, as the second one's registers spilled (rmat20
    // 1,033 -> 1,402 us at N = 128), and 4-lane groups were slower with it
    // (rmat22 619 -> 670 us at N = 16).
    constexpr bool kOneRowForm = G >= 8 && G < 32;
    if (kOneRowForm && s_row[base - nbase] == s_row[min(base + NPI, p1) - 1 - nbase])
      sddmm_round_dots<VEC, G, NCH, U, R, kOneRowForm>(base, p1, nbase, s_col, s_row, N, B, Crow0, coffl, valid, grp,
                                                       gl, dots);
    else
      sddmm_round_dots<VEC, G, NCH, U, R, false>(base, p1, nbase, s_col, s_row, N, B, Crow0, coffl, valid, grp, gl,
                                                 dots);
#pragma unroll
    for (int r0 = 0; r0 < R; r0 += G) {  // one round: G steps, S*G = 32 nonzeros
      float v[G];
#pragma unroll
      for (int i = 0; i < G; ++i) v[i] = dots[r0 + i];
      const float x = group_reduce_transposed<G, G>(v, gl);
      const int n = base + (r0 + gl) * S + grp;  // the warp's 32 lanes cover 32 consecutive nonzeros
      if (n < p1) store(n, x);
    }
  }
}

template <int VEC, int G, int NCH>
__global__ void __launch_bounds__(kThreads, SPMM_SDDMM_MIN_BLOCKS)
    spmm_sddmm_kernel(int32_t M, int32_t N, const int32_t* __restrict__ rowptr, const int32_t* __restrict__ colind,
                      const float* __restrict__ Cd, const float* __restrict__ B, float* __restrict__ out,
                      const int2* __restrict__ part, int32_t T, int* __restrict__ err) {
  extern __shared__ __align__(16) unsigned char smem[];
  const int Tpad = T + 8;
  int* s_col = reinterpret_cast<int*>(smem);
  int* s_row = s_col + Tpad;
  int* s_rp = s_col + 2 * Tpad;
  uint64_t* s_bar = reinterpret_cast<uint64_t*>(s_col + 3 * Tpad);

  const int tid = threadIdx.x;
  const int2 beg = __ldg(part + blockIdx.x);
  const int2 fin = __ldg(part + blockIdx.x + 1);
  const int i0 = beg.x, p0 = beg.y, i1 = fin.x, p1 = fin.y;
  const int nbase = p0 & ~3, rbase = i0 & ~3;

  // ---- stage colind[p0, p1) and rowptr[i0, i1] ------------------------------
  if (!stage_range<false>(colind, nullptr, rowptr, i0, p0, i1, p1, s_col, nullptr, s_rp, s_bar, err, [] {})) return;
  fill_row_ids(s_rp + (i0 - rbase), i1 - i0, p0, p1, nbase, s_row);

  // ---- rounds of nonzeros ---------------------------------------------------
  sddmm_rounds<VEC, G, NCH>(N, s_col, s_row, nbase, p0, p1, Cd + size_t(i0) * N, B, tid >> 5, tid & 31,
                            [&](int n, float x) { st_stream1(out + n, x); });
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
  SPMM_DEBUG_RANGES(L.stream, L.err, {{L.B, size_t(L.K) * L.N * 4}, {Cd, size_t(L.M) * L.N * 4}},
                    {{out, size_t(L.nnz) * 4}});
  spmm_sddmm_kernel<VEC, G, NCH><<<unsigned(L.num_ctas), kThreads, smem, L.stream>>>(
      L.M, L.N, L.rowptr, L.colind, Cd, static_cast<const float*>(L.B), out, L.part, L.items_per_cta, L.err);
  return cudaGetLastError();
}

}  // namespace spmm
