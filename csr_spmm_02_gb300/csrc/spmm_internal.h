// Host-side internals shared by the library's translation units.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/spmm.h"

// 16-byte chunks of the output row each lane owns (fp32: 4 columns per chunk;
// bf16 B: 8 columns per chunk, so half as many chunks).  Wider lane slices
// spread each nonzero's bookkeeping over fewer lanes.
#ifndef SPMM_LANE_CHUNKS
#define SPMM_LANE_CHUNKS 1
#endif
#define SPMM_BF16_CHUNKS (SPMM_LANE_CHUNKS / 2 > 0 ? SPMM_LANE_CHUNKS / 2 : 1)
// The same for the balanced kernel (its warps split into 32/G groups that
// take consecutive nonzeros, so wider lane slices mean more nonzeros per step).
#ifndef SPMM_BAL_CHUNKS
#define SPMM_BAL_CHUNKS 1
#endif
#define SPMM_BAL_BF16_CHUNKS (SPMM_BAL_CHUNKS / 2 > 0 ? SPMM_BAL_CHUNKS / 2 : 1)

// (VEC, G, NCH) shapes compiled for each kernel: small rows use one lane with
// 1, 2 or 4 chunks; wider rows use G lanes with the standard chunk count.
#define SPMM_VECTOR_SHAPES(X, V, NC)                                                            \
  X(V, 1, 1) X(V, 1, 2) X(V, 1, 4) X(V, 2, NC) X(V, 4, NC) X(V, 8, NC) X(V, 16, NC) X(V, 32, NC)
#define SPMM_SCALAR_SHAPES(X) X(1, 8, 1) X(1, 32, 1)


struct spmm_plan_s {
  int32_t M = 0;
  int64_t nnz = 0;
  int32_t N = 0;
  const int32_t* rowptr = nullptr;  // device, borrowed from the caller
  int32_t kernel = SPMM_KERNEL_ROW;
  int32_t max_row_nnz = 0;
  int32_t empty_rows = 0;
  int32_t items_per_cta = 0;  // balanced only
  int32_t num_ctas = 0;       // balanced only
  int32_t group_lanes = 0;    // SMALLN only: lanes sharing a row
  int32_t column_tile = 0;    // N-slicing cap of the row and balanced kernels (0: none)
  int device = 0;
  // device workspace (one allocation, carved up)
  void* workspace = nullptr;
  int64_t workspace_bytes = 0;
  int2* part = nullptr;   // [num_ctas + 1] merge-path coordinates (row, nnz)
  float* carry = nullptr; // [num_ctas][2][N] partial rows split across CTAs
  int* err = nullptr;     // device error word (the plan's own, or the one-call forms' shared word)
  int* stats = nullptr;   // [3]: max row length, empty rows, rowptr[M]
  void* small = nullptr;  // one-call forms: the 16-byte allocation holding the error word and stats
                         // (a plan keeps them in the first 256 bytes of its workspace)
  cudaEvent_t split_event = nullptr;  // recorded between main kernel and fixup
};

namespace spmm {

// Everything one SpMM launch needs (device pointers).
struct Launch {
  int32_t M, N, K;
  int64_t nnz;
  const int32_t* rowptr;
  const int32_t* colind;
  const float* vals;
  const void* B;
  float* C;
  // balanced kernel
  const int2* part;
  int32_t num_ctas;
  int32_t items_per_cta;
  float* carry;
  int* err;
  cudaStream_t stream;
};

// Lane layout for one launch: VEC elements per 16-byte load, G lanes per row
// group (a power of two <= 32), NCH vector chunks per lane.  A group covers
// TW = G * VEC * NCH output columns; wider N is split into column tiles.
struct Shape {
  int vec, G, nch;
  int tile_width() const { return G * vec * nch; }
};

Shape choose_shape(int32_t N, bool bf16, bool vector_ok, int chunks_f32);
inline Shape choose_shape(int32_t N, bool bf16, bool vector_ok) {
  return choose_shape(N, bf16, vector_ok, SPMM_LANE_CHUNKS);
}
inline Shape choose_shape_balanced(int32_t N, bool bf16, bool vector_ok) {
  return choose_shape(N, bf16, vector_ok, SPMM_BAL_CHUNKS);
}

// N-slicing: narrow the column tile (fewer lanes per group) until it spans at
// most `cap` columns (0: no cap).  Column tiles run as grid.y, and CTAs of
// tile 0 are scheduled before those of tile 1, so each tile's slice of B is
// what the caches hold at a time.
inline Shape cap_tile(Shape s, int32_t cap) {
  while (cap > 0 && s.G > 1 && s.tile_width() > cap) s.G >>= 1;
  return s;
}

cudaError_t launch_row_f32(const Launch& L, Shape s);
cudaError_t launch_row_bf16(const Launch& L, Shape s);
cudaError_t launch_balanced_f32(const Launch& L, Shape s);
cudaError_t launch_balanced_bf16(const Launch& L, Shape s);
cudaError_t launch_rowgroup_f32(const Launch& L, int lanes);
// Balanced plans with N <= 2, N = 4 with aligned fp32 B or N = 8 with aligned
// bf16 B (thread_ranges_shape): one thread per slice of each merge-path range
// (spmm_thread_ranges.cuh); the fixup kernel completes rows split across ranges.
bool thread_ranges_shape(int32_t N, bool bf16, bool vector_ok);
cudaError_t launch_thread_ranges(const Launch& L, bool bf16, bool vector_ok);
// FusedMM on the same shapes (fp32; L.B is D, Cd and Bd the dot-product operands).
cudaError_t launch_thread_ranges_fused(const Launch& L, bool vector_ok, const float* Cd, const float* Bd);
cudaError_t launch_rowgroup_bf16(const Launch& L, int lanes);
cudaError_t launch_tc_window_bf16(const Launch& L);
cudaError_t launch_window_f32(const Launch& L);
cudaError_t launch_window_bf16(const Launch& L);
cudaError_t launch_fixup(const Launch& L, int sr = 0);  // sr: semiring code, 0 = sum
// The balanced SpMM kernels (ordinary and semiring) return
// cudaErrorNotSupported when K * N / VEC does not fit 32 bits.
// Balanced kernel with a semiring (fp32 B); sr = 2 * add + mul in 1..5
// (add 0 sum, 1 min, 2 max; mul 0 multiply, 1 add).
cudaError_t launch_semiring_f32(const Launch& L, Shape s, int sr);
cudaError_t launch_sddmm_f32(const Launch& L, Shape s, const float* Cd, float* out);
// SDDMM with one group of G lanes (4, 8, 16, 32) per row: 4 fp32 columns per lane, N <= 4G.
cudaError_t launch_sddmm_row_f32(const Launch& L, int G, const float* Cd, float* out);
cudaError_t launch_fusedmm_f32(const Launch& L, Shape s, const float* Cd, const float* Bd);
// SDDMM / FusedMM on window-class plans: the dense window of each 32-row block
// from shared memory (blocks whose columns span more than 96 gather instead).
// N a multiple of 4, at most 512, operands 16-byte aligned.  FusedMM: L.B is D.
cudaError_t launch_window_sddmm_f32(const Launch& L, const float* Cd, float* out);
cudaError_t launch_window_fusedmm_f32(const Launch& L, const float* Cd, const float* Bd);
// FusedMM with one group of G lanes (4, 8, 16, 32) per row: 4 fp32 columns per lane, N <= 4G; L.B is D.
cudaError_t launch_fusedmm_row_f32(const Launch& L, int G, const float* Cd, const float* Bd);
// Merge-path coordinates of the P+1 range starts (ranges of T items) into part.
// With err: rowptr[M] is compared with nnz on the device; on a mismatch every
// range is made empty (nothing is read past either array) and kErrInvalidCsr
// is set in *err.
cudaError_t launch_partition(const int32_t* rowptr, int32_t M, int64_t nnz, int32_t T, int32_t P, int2* part,
                             cudaStream_t stream, int* err = nullptr);

// Device address of the error word that the one-call forms share on the
// current device (looked up on every call, so it stays valid after the
// device's context is reset).
cudaError_t call_error_word(int** out);


constexpr int kDefaultItemsPerCta = 2048;
// The plan's merge-path range when the caller leaves it to the plan: rows of
// 9 to 32 columns put four to eight nonzeros in a warp step, so a range of a
// given size holds more row ends per step of work; 3072 items per CTA
// measured best there (R-MAT scale 22, N = 32: SpMM 848 -> 790 us, FusedMM
// 2.05 -> 1.96 ms).  N = 1 and 4 run the thread-range kernel, whose CTAs
// amortise their staging, searches and scan over more items at 3840 (15 per
// thread; the rmat20 pattern at N = 1 119 -> 113 us, N = 4 167 -> 138 us);
// N = 3 (lane groups) also gained there (165 -> 150 us), and so did N = 8 in
// both of its kernels (fp32 B, lane groups: 226 -> 195 us; bf16 B, thread
// ranges: 236 -> 185 us; rmat22 866 -> 783 and 941 -> 728 us).  2048
// elsewhere: N = 2, whose threads gather in batches of four (136 -> 206 us at
// 3840), and N = 5 .. 7, 64 and 128.
inline int default_items_per_cta(int32_t N) {
  if (N > 8 && N <= 32) return 3072;
  if (N == 1 || N == 3 || N == 4 || N == 8) return 3840;
  return kDefaultItemsPerCta;
}

constexpr int kMaxItemsPerCta = 8192;
constexpr int kMaxDevices = 64;

}  // namespace spmm
