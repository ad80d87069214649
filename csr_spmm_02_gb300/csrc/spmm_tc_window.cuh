// Tensor-core window kernel (bf16 B): the dense window of a row block
// multiplied by the 5th-generation tensor cores (tcgen05, accumulator in
// tensor memory).
//
// For rows whose columns are local (a band), the window kernel's work is a
// dense product per row block: A_w (rows x window columns, zero where A has no
// entry) times B_w (window columns x N).  On CUDA cores that product is bound
// by the FP32 pipe; here each 128-row tile hands it to tcgen05.mma:
//
//  * A's fp32 values are split exactly into three bf16 terms (hi + mid + lo
//    carries all 24 significand bits); each bf16 x bf16 product is exact in
//    fp32, so three MMAs per K-step reproduce the fp32 products and only the
//    accumulation order differs from a row loop;
//  * the tile's window (at most three chunks of 64 columns) is built once in
//    shared memory as three K-major bf16 tiles per chunk (128-byte swizzled
//    layout); B is streamed in 32-row pieces by the tensor memory accelerator
//    (boxes of 64 columns x 32 rows, 128-byte swizzled, landing directly in the
//    MN-major layout the MMA reads; rows past K zero-filled) through three
//    stages;
//  * per chunk, 4 K-steps x 3 terms of M=128, N, K=16 MMAs accumulate into one
//    of two tensor-memory accumulators.
//
// The kernel is persistent (one CTA per SM, tiles strided by the grid) and
// its warps have four roles, so that the steps of consecutive tiles overlap:
//
//  * warps 0-11 (builders) hold a tile's nonzeros in registers, check the
//    column span, publish the tile's description, then zero and fill the A
//    window once the previous tile's MMAs have read it; the hi terms go in
//    with shared-memory atomicOr, whose old value shows a (row, column) pair
//    met twice (a tile with such duplicates is discarded by the epilogue and
//    gathered by the builders instead);
//  * warp 12 (producer) loads the B pieces of each tensor-core tile with TMA
//    and prefetches the next tile's nonzeros into L2;
//  * warp 13 (MMA) issues the MMAs once the A window and a B stage are full;
//    tcgen05.commit frees the stage and the window and, per tile, marks the
//    accumulator full;
//  * warps 14-17 (epilogue) read a full accumulator with tcgen05.ld (warp w
//    reads lanes 32*(w%4)..), turn each 32 x 32 block around in shared memory
//    so that every store writes 4 rows x 128 contiguous bytes, then mark the
//    accumulator drained.
//
// Every wait on an mbarrier is bounded: on expiry the kernel records
// kErrStageTimeout in the plan's error word and stops instead of hanging.
//
// A tile whose column span exceeds three chunks, one holding more than 8448
// nonzeros, one with a duplicate (row, column) entry (both nonzero), or one
// holding a nonzero value below 2^-110 in magnitude (which the three-term
// split cannot carry exactly) is computed by the builders with per-row
// gathers (columns need not be sorted); a tile with
// no nonzeros stores zero rows.  The dense product multiplies absent entries
// as zeros, so a NaN/Inf in a B row inside the window reaches every row of
// the tile; IEEE special values are outside the accepted inputs.
#pragma once

#include <algorithm>
#include <climits>

#include <cuda.h>
#include <cuda_bf16.h>

#include "spmm_device.cuh"
#include "spmm_internal.h"

namespace spmm {

namespace tc {

constexpr int kRows = 128;       // rows per tile = MMA M
constexpr int kChunk = 64;       // window columns per chunk (4 K-steps of 16)
constexpr int kMaxChunks = 3;    // larger spans use the gather path
constexpr int kBRows = 32;       // B rows per stage (2 K-steps)
constexpr int kBCols = 64;                // B columns per TMA box (128 bytes: one swizzle span)
constexpr int kBBox = kBRows * kBCols * 2;  // one box: 32 rows x 128 bytes = 4 KB
constexpr int kStages = 3;
constexpr int kATile = kRows * kChunk * 2;         // one bf16 term of one chunk: 16 KB
constexpr int kAWindow = kMaxChunks * 3 * kATile;  // the whole window: 144 KB
constexpr int kBuilders = 384;                     // builder threads (warps 0-11)
constexpr int kProducerWarp = 12;
constexpr int kMmaWarp = 13;
constexpr int kEpiWarp0 = 14;  // warps 14-17
constexpr int kCtaThreads = 18 * 32;
constexpr int kPerThread = 22;  // nonzeros a builder holds: a tile of at most 8448 uses the tensor cores
constexpr int kTileNnz = kPerThread * kBuilders;
enum TileKind { kTensor = 0, kZero = 1, kGather = 2 };
constexpr int kTwFloats = 32 * 36;  // one epilogue warp's transpose buffer (rows of 36 floats)
// mbarriers: A full, A free, B full[3], B empty[3], accumulator full[2] and
// drained[2], tile description full[2] and consumed[2]
constexpr int kBars = 16;

__host__ __device__ constexpr size_t stage_bytes(int N) { return size_t((N + kBCols - 1) / kBCols) * kBBox; }

__host__ __device__ constexpr size_t smem_bytes(int N) {
  return size_t(kAWindow) + kStages * stage_bytes(N)  // A window, B stages
         + kTileNnz                                   // local row of every held nonzero (1 byte)
         + 4 * kTwFloats * 4                          // epilogue transposes
         + 2 * (kRows + 8) * 4                        // rowptr slices (this tile, the next)
         + kBars * 8 + 2 * 16 + 2 * 8 + 4 + 4 * 4 + 4;  // barriers, tile descriptions, ring, TMEM
                                                         // address, reductions, beat
}

// Shared-memory matrix descriptors (tcgen05): start address >> 4 in bits
// 0-13, leading-byte offset >> 4 in 16-29, stride-byte offset >> 4 in 32-45,
// version 1 in 46-47, layout type in 61-63.  Both operands use the 128-byte
// swizzle; the field assignments below were checked on exact integer inputs.
//
// A tiles use the K-major 128-byte swizzled layout: row r of a
// tile is the 128 bytes at r * 128 (its 64 K-elements), 8-row groups 1024
// bytes apart, and 16-byte piece c of a row sits at piece c ^ (r & 7).  A
// warp's consecutive nonzeros of one row then fall in distinct banks.  The
// tile base is 1024-byte aligned and a K-step of 16 advances the start
// address by 32 bytes (the swizzle acts on the address bits).
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr) {
  uint64_t d = uint64_t((saddr & 0x3FFFFu) >> 4);
  d |= uint64_t(1) << 16;             // leading-byte offset: unused for swizzled K-major
  d |= uint64_t(1024 >> 4) << 32;     // stride-byte offset: 8-row groups
  d |= uint64_t(1) << 46;             // descriptor version of this architecture
  d |= uint64_t(2) << 61;             // layout type: 128-byte swizzle
  return d;
}
// B pieces are MN-major with the same 128-byte swizzle, as the TMA unit lays
// them out: K-row k of a 64-column block is the 128 bytes at k * 128 (16-byte
// piece c at c ^ (k & 7)), 8-row groups 1024 bytes apart along K, 64-column
// blocks 4 KB apart along N.  A K-step of 16 rows advances the start by 2 KB.
__device__ __forceinline__ uint64_t sdesc_b_sw128(uint32_t saddr) {
  uint64_t d = uint64_t((saddr & 0x3FFFFu) >> 4);
  d |= uint64_t(kBBox >> 4) << 16;    // leading-byte offset: next 64-column block (N)
  d |= uint64_t(1024 >> 4) << 32;     // stride-byte offset: next 8 rows (K)
  d |= uint64_t(1) << 46;             // descriptor version of this architecture
  d |= uint64_t(2) << 61;             // layout type: 128-byte swizzle
  return d;
}
__device__ __forceinline__ uint32_t a_offset(int r, int kk) {  // byte of element (r, kk) in a tile
  return uint32_t(r) * 128u + (uint32_t((kk >> 3) ^ (r & 7)) << 4) + uint32_t(kk & 7) * 2u;
}

// kind::f16 instruction descriptor: D fp32, A and B bf16, A K-major, B
// MN-major, M = 128, N = n.
__device__ __forceinline__ uint32_t idesc(int n) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (0u << 15) | (1u << 16) | (uint32_t(n >> 3) << 17) |
         (uint32_t(kRows >> 4) << 24);
}

__device__ __forceinline__ void mma(uint32_t tmem_d, uint64_t a, uint64_t b, uint32_t id, bool accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
      "l"(a), "l"(b), "r"(id), "r"(uint32_t(accumulate)));
}
__device__ __forceinline__ void commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
               : "memory");
}
__device__ __forceinline__ void fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// 16 consecutive fp32 accumulator columns of this thread's lane.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ uint16_t bf16_rn_bits(float x) { return __bfloat16_as_ushort(__float2bfloat16_rn(x)); }
__device__ __forceinline__ float bf16_bits_to_float(uint16_t b) { return __uint_as_float(uint32_t(b) << 16); }

// Plain arrive (release semantics at CTA scope).
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// One 2-D TMA box of B (64 columns x 32 rows, 4 KB, 128-byte swizzled) into
// shared memory, completing its bytes on `bar`.  x (the column) is a
// multiple of 64.
__device__ __forceinline__ void tma_load_b(uint32_t dst, const CUtensorMap* map, int x, int y, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], "
      "[%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}

// Barrier 1 joins the builder warps only.
__device__ __forceinline__ void builders_sync() { asm volatile("bar.sync 1, %0;" ::"n"(kBuilders) : "memory"); }
// The same barrier, returning whether `p` holds in every builder thread.
__device__ __forceinline__ bool builders_and(bool p) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred a, b;\n\tsetp.ne.u32 a, %1, 0;\n\t"
      "bar.red.and.pred b, 1, %2, a;\n\tselp.u32 %0, 1, 0, b;\n\t}"
      : "=r"(r)
      : "r"(uint32_t(p)), "n"(kBuilders)
      : "memory");
  return r != 0;
}

// The same barrier, returning whether `p` holds in some builder thread.
__device__ __forceinline__ bool builders_or(bool p) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred a, b;\n\tsetp.ne.u32 a, %1, 0;\n\t"
      "bar.red.or.pred b, 1, %2, a;\n\tselp.u32 %0, 1, 0, b;\n\t}"
      : "=r"(r)
      : "r"(uint32_t(p)), "n"(kBuilders)
      : "memory");
  return r != 0;
}

// Bounded wait that tolerates slow builders: the poll budget restarts while
// `beat` (advanced by the builders per tile and per gathered row) moves, so it
// expires only when the builders make no progress.
__device__ __forceinline__ bool mbar_wait_progress(uint32_t bar, uint32_t parity, const volatile int* beat) {
  int seen = *beat;
  for (;;) {
    if (mbar_wait_bounded(bar, parity, kSpinLimit)) return true;
    const int now = *beat;
    if (now == seen) return false;
    seen = now;
  }
}

// Hint: bring [lo, hi) into L2, shrunk to 16-byte boundaries inside the range.
__device__ __forceinline__ void l2_prefetch(const void* lo, const void* hi) {
  const uintptr_t a = (reinterpret_cast<uintptr_t>(lo) + 15) & ~uintptr_t(15);
  const uintptr_t e = reinterpret_cast<uintptr_t>(hi) & ~uintptr_t(15);
  if (e > a)
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(a), "r"(uint32_t(e - a)) : "memory");
}

}  // namespace tc

__global__ void __launch_bounds__(tc::kCtaThreads, 1)
    spmm_tc_window_kernel(int32_t M, int32_t N, int32_t K, const int32_t* __restrict__ rowptr,
                          const int32_t* __restrict__ colind, const float* __restrict__ vals,
                          const uint16_t* __restrict__ B, float* __restrict__ C, int* __restrict__ err,
                          uint32_t acc_cols, const __grid_constant__ CUtensorMap bmap) {
  using namespace tc;
  extern __shared__ __align__(1024) unsigned char smem[];
  const size_t sb = stage_bytes(N);
  unsigned char* s_A = smem;                                  // chunk c, term t at (3c + t) * kATile
  unsigned char* s_B = smem + kAWindow;                       // stage s at s * sb
  uint8_t* s_rowid = s_B + kStages * sb;                      // [kTileNnz] local row of each held nonzero
  float* s_tw = reinterpret_cast<float*>(s_rowid + kTileNnz);  // [4 warps][kTwFloats]
  int* s_rp_buf = reinterpret_cast<int*>(s_tw + 4 * kTwFloats);  // [2][kRows + 8] rowptr slices
  uint64_t* s_bar = reinterpret_cast<uint64_t*>(s_rp_buf + 2 * (kRows + 8));
  int4* s_info = reinterpret_cast<int4*>(s_bar + kBars);      // [2] (first row, rows, cmin, kind | chunks << 8)
  int* s_ring = reinterpret_cast<int*>(s_info + 2);           // [2][2] first row and rows per accumulator
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(s_ring + 4);
  int* s_red = reinterpret_cast<int*>(s_tmem + 1);  // [0] min col, [1] max col, [2] flags, [3] discard
  volatile int* s_beat = s_red + 4;                           // builders' progress counter

  const int tid = threadIdx.x, w = tid >> 5, lane = tid & 31;
  const int ntiles = int((int64_t(M) + kRows - 1) / kRows);
  const uint32_t bar0 = smem_addr(s_bar);
  auto bar = [bar0](int i) { return bar0 + 8u * uint32_t(i); };
  constexpr int kAFull = 0, kAFree = 1, kBFull = 2, kBEmpty = 5, kAccFull = 8, kAccDrained = 10, kInfoFull = 12,
                kInfoUsed = 14;

  // ---- set-up: two accumulators of acc_cols columns, the barriers ----------
  if (w == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(s_tmem)),
                 "r"(2 * acc_cols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  if (tid == 0) {
    *s_beat = 0;
    mbar_init(bar(kAFull), 1);   // the builders, once the window is written
    mbar_init(bar(kAFree), 1);   // commit after a tile's last MMAs
    for (int s = 0; s < kStages; ++s) {
      mbar_init(bar(kBFull + s), 1);   // the producer's expect-tx arrive + the TMA bytes
      mbar_init(bar(kBEmpty + s), 1);  // commit after the stage's MMAs
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(kAccFull + s), 2);        // the tile's last commit + the ring entry's arrive
      mbar_init(bar(kAccDrained + s), 4);     // one arrive per epilogue warp
      mbar_init(bar(kInfoFull + s), 1);       // the builders publish a tile description
      mbar_init(bar(kInfoUsed + s), 2);       // the producer and the MMA warp have read it
    }
  }
  fence_before();
  __syncthreads();
  fence_after();
  const uint32_t tmem = *s_tmem;

  if (w < kBuilders / 32) {
    // =================== builders ===================
    constexpr uint32_t kNone = 0xFFFFFFFFu;
    const uint64_t stream_pol = policy_evict_first();
    uint32_t tt = 0;  // tensor-core tiles built
    bool ok = true;
    int j = 0;
    if (int(blockIdx.x) < ntiles) {  // the first tile's rowptr slice; each tile loads the next one's
      const int i0 = blockIdx.x * kRows, nr = min(kRows, M - i0);
      for (int t = tid; t <= nr; t += kBuilders) s_rp_buf[t] = ld_stream(rowptr + i0 + t, stream_pol);
    }
    for (int tile = blockIdx.x; tile < ntiles && ok; tile += gridDim.x, ++j) {
      const int i0 = tile * kRows;
      const int nrows = min(kRows, M - i0);
      int* s_rp = s_rp_buf + (j & 1) * (kRows + 8);
      int* s_rp_next = s_rp_buf + ((j + 1) & 1) * (kRows + 8);
      builders_sync();  // this tile's rowptr slice is in; the previous tile is done with s_red and s_rowid
      if (tid == 0) {
        s_red[0] = INT_MAX;
        s_red[1] = -1;
        s_red[2] = 0;
        *s_beat = *s_beat + 1;
      }
      // the next tile's rowptr slice, stored at the end of this tile
      const int next = tile + int(gridDim.x);
      const int next_rows = next < ntiles ? min(kRows, M - next * kRows) : -1;
      static_assert(kBuilders > kRows, "one rowptr entry per builder thread");
      int rp_next = 0;
      if (tid <= next_rows) rp_next = ld_stream(rowptr + int64_t(next) * kRows + tid, stream_pol);
      builders_sync();

      // ---- the tile's nonzeros into registers (one load round) ----------
      // Thread t holds nonzeros p0 + t + 384 i (i < kPerThread): its value and
      // its column (later a packed word (row << 16) | local column), or kNone.
      const int p0 = s_rp[0], p1 = s_rp[nrows];
      const bool fits = p1 - p0 <= kTileNnz;
      uint32_t pk[kPerThread];
      float val[kPerThread];
      if (fits) {
#pragma unroll
        for (int i = 0; i < kPerThread; ++i) {
          const int g = p0 + tid + kBuilders * i;
          pk[i] = g < p1 ? uint32_t(ld_stream(colind + g, stream_pol)) : kNone;
          val[i] = g < p1 ? ld_stream(vals + g, stream_pol) : 0.f;
        }
      }
      if (fits) {
        // the local row of every tile nonzero, one byte each: thread r fills
        // row r, 4-byte stores for the aligned middle (no word is shared
        // between rows there), bytes at the ends
        for (int r = tid; r < nrows; r += kBuilders) {
          const int e = s_rp[r + 1] - p0;
          int g = s_rp[r] - p0;
          for (; g < e && (g & 3); ++g) s_rowid[g] = uint8_t(r);
          const uint32_t rep4 = uint32_t(r) * 0x01010101u;
          for (; g + 4 <= e; g += 4) *reinterpret_cast<uint32_t*>(s_rowid + g) = rep4;
          for (; g < e; ++g) s_rowid[g] = uint8_t(r);
        }
      }
      builders_sync();
      if (fits) {
        // column span, and the row of every held nonzero
        int lo = INT_MAX, hi = -1;
#pragma unroll
        for (int i = 0; i < kPerThread; ++i) {
          const int g = p0 + tid + kBuilders * i;
          const bool valid = g < p1;
          const int c = int(pk[i]);
          if (valid) {
            lo = min(lo, c);
            hi = max(hi, c);
          }
          const int r = valid ? int(s_rowid[g - p0]) : 0;
          pk[i] = valid ? (uint32_t(r) << 16) | (uint32_t(c) & 0xFFFFu) : kNone;
        }
        lo = __reduce_min_sync(0xffffffffu, lo);
        hi = __reduce_max_sync(0xffffffffu, hi);
        if (lane == 0) {
          atomicMin(s_red + 0, lo);
          atomicMax(s_red + 1, hi);
        }
      } else if (tid == 0) {
        s_red[2] = 1;  // too many nonzeros to hold: gather path
      }
      builders_sync();
      const int cmin = s_red[0], cmax = s_red[1];
      const int nch = cmax < 0 ? 0 : (cmax - cmin) / kChunk + 1;
      const int kind = (s_red[2] != 0 || nch > kMaxChunks) ? kGather : (nch == 0 ? kZero : kTensor);

      // ---- publish the tile's description to the producer and MMA warps ---
      const uint32_t slot = uint32_t(j) & 1u;
      bool got = true;
      if (tid == 0) {
        if (j >= 2) got = mbar_wait_bounded(bar(kInfoUsed + slot), (uint32_t(j >> 1) - 1) & 1u, kSpinLimit);
        s_info[slot] = make_int4(i0, nrows, cmin, kind | (nch << 8));
        mbar_arrive(bar(kInfoFull + slot));
        if (kind == kTensor) l2_prefetch(B + size_t(cmin) * N, B + size_t(min(cmax + 1, K)) * N);  // for the TMA
      }
      if (!builders_and(got)) {
        ok = false;
        break;
      }

      bool discard = false;  // a tensor-core tile with duplicate entries
      if (kind == kTensor) {
        // local column of each held nonzero: its low 16 bits minus cmin's,
        // modulo 2^16 (exact, since the span is below 2^16)
#pragma unroll
        for (int i = 0; i < kPerThread; ++i)
          if (pk[i] != kNone) pk[i] = (pk[i] & 0xFFFF0000u) | ((pk[i] - uint32_t(cmin)) & 0xFFFFu);
        if (tt >= 1) {  // the previous tile's MMAs have read the window
          ok = builders_and(mbar_wait_bounded(bar(kAFree), (tt - 1) & 1u, kSpinLimit));
          fence_after();
          if (!ok) break;
        }
        for (int t = tid; t < nch * 3 * kATile / 16; t += kBuilders)
          reinterpret_cast<uint4*>(s_A)[t] = make_uint4(0u, 0u, 0u, 0u);
        builders_sync();
        // every held nonzero into its chunk: value -> three bf16 terms.  A
        // zero value adds nothing and is left out; the hi term of any other
        // value is nonzero, so an atomicOr that finds its half-word already
        // set has met a second nonzero for the same (row, column).  The split
        // is exact only for |v| >= 2^-110 (below that the lo term is subnormal
        // in bf16 and keeps fewer bits; under about 2^-134 even the hi term
        // rounds to zero): a tile holding a nonzero value of smaller
        // magnitude is gathered instead, like one with a duplicate.
        bool dup = false;
#pragma unroll
        for (int i = 0; i < kPerThread; ++i) {
          if (pk[i] != kNone) {
            const int k = int(pk[i] & 0xFFFFu), r = int(pk[i] >> 16);
            const int ch = k >> 6, kk = k & (kChunk - 1);
            const float v = val[i];
            dup |= v != 0.f && fabsf(v) < 0x1p-110f;
            const uint16_t h = bf16_rn_bits(v);
            if (h != 0) {
              const float r1 = v - bf16_bits_to_float(h);
              const uint16_t m = bf16_rn_bits(r1);
              const uint16_t l = bf16_rn_bits(r1 - bf16_bits_to_float(m));
              const uint32_t off = uint32_t(3 * ch) * kATile + a_offset(r, kk);
              const uint32_t shift = (off & 2u) * 8u;
              const uint32_t old = atomicOr(reinterpret_cast<uint32_t*>(s_A + (off & ~3u)), uint32_t(h) << shift);
              dup |= ((old >> shift) & 0xFFFFu) != 0;
              *reinterpret_cast<uint16_t*>(s_A + kATile + off) = m;
              *reinterpret_cast<uint16_t*>(s_A + 2 * kATile + off) = l;
            }
          }
        }
        fence_proxy_async();  // generic-proxy writes become visible to the tensor cores
        discard = builders_or(dup);
        if (tid == 0) {
          s_red[3] = discard;  // read by the MMA warp once the window is full
          mbar_arrive(bar(kAFull));
        }
        ++tt;
      }
      if (kind == kZero) {  // no nonzeros in the tile: zero rows
        for (int t = tid; t < nrows * (N / 4); t += kBuilders) {
          const int r = t / (N / 4), c4 = t - r * (N / 4);
          st_stream4(C + size_t(i0 + r) * N + 4 * c4, 0.f, 0.f, 0.f, 0.f);
        }
      } else if (kind == kGather || discard) {  // gather path: warp w computes rows w, w + 12, ...
        for (int r = w; r < nrows; r += kBuilders / 32) {
          const int start = s_rp[r], end = s_rp[r + 1];
          if (tid == 0) *s_beat = *s_beat + 1;
          for (int c0 = lane * 8; c0 < N; c0 += 32 * 8) {
            FVec<8> acc;
            acc.zero();
            for (int g = start; g < end; ++g) {
              const int c = __ldg(colind + g);
              BSlice<uint16_t, 8> bs;
              bs.load(B + size_t(c) * N + c0);
              FVec<8> bv;
              bs.widen(bv);
              acc.fma(pair(__ldg(vals + g)), bv);
            }
            store_c<8>(C + size_t(i0 + r) * N + c0, acc);
          }
        }
      }
      if (tid <= next_rows) s_rp_next[tid] = rp_next;
    }
    if (!ok && tid == 0) atomicOr(err, kErrStageTimeout);
  } else if (w == kProducerWarp) {
    // =================== producer: B chunks by TMA ===================
    if (lane == 0) {
      uint32_t gc = 0;  // B pieces loaded (stage gc % kStages)
      bool ok = true;
      int j = 0;
      for (int tile = blockIdx.x; tile < ntiles && ok; tile += gridDim.x, ++j) {
        const uint32_t slot = uint32_t(j) & 1u;
        if (!mbar_wait_progress(bar(kInfoFull + slot), uint32_t(j >> 1) & 1u, s_beat)) {
          ok = false;
          break;
        }
        const int4 info = s_info[slot];
        mbar_arrive(bar(kInfoUsed + slot));
        // the next tile's nonzeros into L2 while the builders finish this one
        const int next = tile + int(gridDim.x);
        if (next < ntiles) {
          const int q0 = __ldg(rowptr + int64_t(next) * kRows);
          const int q1 = __ldg(rowptr + min(int64_t(M), int64_t(next) * kRows + kRows));
          if (q1 > q0 && q1 - q0 <= kTileNnz) {
            l2_prefetch(colind + q0, colind + q1);
            l2_prefetch(vals + q0, vals + q1);
          }
        }
        if ((info.w & 0xFF) != kTensor) continue;
        const int pieces = (info.w >> 8) * (kChunk / kBRows);
        for (int c = 0; c < pieces; ++c) {
          const uint32_t s = gc % kStages, use = gc / kStages;
          if (use >= 1 && !mbar_wait_bounded(bar(kBEmpty + s), (use - 1) & 1u, kSpinLimit)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(bar(kBFull + s), uint32_t(sb));
          const uint32_t dst = smem_addr(s_B + s * sb);
          for (int q = 0; q < (N + kBCols - 1) / kBCols; ++q)
            tma_load_b(dst + uint32_t(q) * kBBox, &bmap, kBCols * q, info.z + c * kBRows, bar(kBFull + s));
          ++gc;
        }
      }
      if (!ok) atomicOr(err, kErrStageTimeout);
    }
  } else if (w == kMmaWarp) {
    // =================== MMA issue ===================
    if (lane == 0) {
      const uint32_t id = idesc(N);
      const uint32_t a_base = smem_addr(s_A), b_base = smem_addr(s_B);
      uint32_t gc = 0, tt = 0;  // B pieces and tensor-core tiles issued
      bool ok = true;
      int j = 0;
      for (int tile = blockIdx.x; tile < ntiles && ok; tile += gridDim.x, ++j) {
        const uint32_t slot = uint32_t(j) & 1u;
        if (!mbar_wait_progress(bar(kInfoFull + slot), uint32_t(j >> 1) & 1u, s_beat)) {
          ok = false;
          break;
        }
        const int4 info = s_info[slot];
        mbar_arrive(bar(kInfoUsed + slot));
        if ((info.w & 0xFF) != kTensor) continue;
        const int nch = info.w >> 8;
        const uint32_t b = tt & 1u, ub = tt >> 1;
        // the window is built, and the epilogue has read this accumulator's previous tile
        if (!mbar_wait_progress(bar(kAFull), tt & 1u, s_beat) ||
            (ub >= 1 && !mbar_wait_bounded(bar(kAccDrained + b), (ub - 1) & 1u, kSpinLimit))) {
          ok = false;
          break;
        }
        fence_after();
        const bool discard = s_red[3] != 0;  // written by the builders before the window-full arrive
        const uint32_t acc = tmem + b * acc_cols;
        // piece c holds B rows cmin + 32c ..: K-steps 2c, 2c+1 of the window
        for (int c = 0; c < nch * (kChunk / kBRows) && ok; ++c) {
          const uint32_t s = gc % kStages, use = gc / kStages;
          if (!mbar_wait_bounded(bar(kBFull + s), use & 1u, kSpinLimit)) {
            ok = false;
            break;
          }
          fence_after();
          const int ch = c / (kChunk / kBRows), kp = c % (kChunk / kBRows);
#pragma unroll
          for (int ks = 0; ks < kBRows / 16; ++ks) {
#pragma unroll
            for (int term = 0; term < 3; ++term) {
              const uint64_t a = sdesc_sw128(a_base + uint32_t(3 * ch + term) * kATile +
                                             uint32_t(kp * (kBRows / 16) + ks) * 32u);
              const uint64_t bd = sdesc_b_sw128(b_base + s * uint32_t(sb) + uint32_t(ks) * 2048u);
              mma(acc, a, bd, id, c > 0 || ks > 0 || term > 0);
            }
          }
          commit(bar(kBEmpty + s));  // the stage is free once these MMAs have read it
          ++gc;
        }
        if (!ok) break;
        commit(bar(kAFree));  // the window too
        s_ring[2 * b] = info.x;
        s_ring[2 * b + 1] = discard ? 0 : info.y;  // a discarded tile is gathered by the builders
        commit(bar(kAccFull + b));  // the accumulator is complete once the MMAs are
        mbar_arrive(bar(kAccFull + b));
        ++tt;
      }
      // end marker in the next accumulator's ring entry
      const uint32_t b = tt & 1u, ub = tt >> 1;
      if (ub >= 1 && !mbar_wait_bounded(bar(kAccDrained + b), (ub - 1) & 1u, kSpinLimit)) ok = false;
      s_ring[2 * b] = -1;
      s_ring[2 * b + 1] = 0;
      mbar_arrive(bar(kAccFull + b));
      mbar_arrive(bar(kAccFull + b));
      // the last tile's commits have arrived before the CTA's shared memory goes away
      if (tt >= 1 && !mbar_wait_bounded(bar(kAFree), (tt - 1) & 1u, kSpinLimit)) ok = false;
      if (!ok) atomicOr(err, kErrStageTimeout);
    }
  } else {
    // =================== epilogue ===================
    // Warp w reads accumulator lanes 32*(w%4).. (rows 32*(w%4).. of the
    // tile) 32 columns at a time; a per-warp shared-memory transpose (rows of
    // 36 floats) turns them into 4-row x 128-byte coalesced stores.
    const int q = w & 3;
    float* tw = s_tw + (w - kEpiWarp0) * kTwFloats;
    const int rr = lane >> 3, cc = (lane & 7) * 4;  // store phase: row (of 4) and column of this lane
    for (uint32_t k = 0;; ++k) {
      const uint32_t b = k & 1u, use = k >> 1;
      if (!mbar_wait_progress(bar(kAccFull + b), use & 1u, s_beat)) {
        if (lane == 0) atomicOr(err, kErrStageTimeout);
        break;
      }
      fence_after();
      const int i0 = s_ring[2 * b], nrows = s_ring[2 * b + 1];
      if (i0 < 0) break;
      const uint32_t acc = tmem + b * acc_cols + (uint32_t(32 * q) << 16);
      for (int c0 = 0; c0 < N; c0 += 32) {
        uint32_t v0[16], v1[16];
        const bool two = c0 + 16 < N;  // N is a multiple of 16
        tmem_ld16(acc + uint32_t(c0), v0);
        if (two) tmem_ld16(acc + uint32_t(c0 + 16), v1);
        tmem_wait_ld();
        __syncwarp();  // every lane is done reading the previous block
#pragma unroll
        for (int e = 0; e < 16; e += 4)
          *reinterpret_cast<uint4*>(tw + lane * 36 + e) = make_uint4(v0[e], v0[e + 1], v0[e + 2], v0[e + 3]);
        if (two)
#pragma unroll
          for (int e = 0; e < 16; e += 4)
            *reinterpret_cast<uint4*>(tw + lane * 36 + 16 + e) = make_uint4(v1[e], v1[e + 1], v1[e + 2], v1[e + 3]);
        __syncwarp();
        const int ncols = two ? 32 : 16;
#pragma unroll
        for (int k8 = 0; k8 < 8; ++k8) {  // rows 4k8 .. 4k8+3 of the warp's 32
          const int lr = 4 * k8 + rr;
          if (32 * q + lr < nrows && cc < ncols) {
            const float4 x = *reinterpret_cast<const float4*>(tw + lr * 36 + cc);
            st_stream4(C + (size_t(i0) + size_t(32 * q + lr)) * N + c0 + cc, x.x, x.y, x.z, x.w);
          }
        }
      }
      fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(kAccDrained + b));
    }
  }

  // ---- release the tensor memory -------------------------------------------
  fence_before();
  __syncthreads();
  if (w == 0) {
    fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(2 * acc_cols) : "memory");
  }
}

// The driver's tensor-map encoder, looked up once through the runtime.
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

inline EncodeTiledFn encode_tiled() {
  static EncodeTiledFn fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      p = nullptr;
    return reinterpret_cast<EncodeTiledFn>(p);
  }();
  return fn;
}

// B (K x N bf16, row-major) as a 2-D tensor for TMA: boxes of 64 columns x 32 rows, 128-byte swizzle.
inline cudaError_t make_b_map(const uint16_t* B, int32_t K, int32_t N, CUtensorMap* map) {
  const EncodeTiledFn enc = encode_tiled();
  if (!enc) return cudaErrorNotSupported;
  const cuuint64_t dims[2] = {cuuint64_t(N), cuuint64_t(K)};
  const cuuint64_t strides[1] = {cuuint64_t(N) * 2};
  const cuuint32_t box[2] = {uint32_t(tc::kBCols), uint32_t(tc::kBRows)};
  const cuuint32_t elem[2] = {1, 1};
  const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t*>(B), dims, strides, box, elem,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorNotSupported;
}

// N a multiple of 16 up to 256, B and C 16-byte aligned (checked by exec).
inline cudaError_t launch_tc_window(const Launch& L) {
  if (L.nnz == 0) return cudaMemsetAsync(L.C, 0, size_t(L.M) * size_t(L.N) * sizeof(float), L.stream);
  static bool attr_set[kMaxDevices] = {};
  static int sm_count[kMaxDevices] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  if (!attr_set[dev]) {
    e = cudaFuncSetAttribute(spmm_tc_window_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             int(tc::smem_bytes(256)));
    if (e != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&sm_count[dev], cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  CUtensorMap map;
  if ((e = make_b_map(static_cast<const uint16_t*>(L.B), L.K, L.N, &map)) != cudaSuccess) return e;
  uint32_t cols = 32;  // one accumulator: a power of two >= N
  while (cols < uint32_t(L.N)) cols <<= 1;
  const int64_t tiles = (int64_t(L.M) + tc::kRows - 1) / tc::kRows;
  const unsigned grid = unsigned(std::min<int64_t>(tiles, sm_count[dev]));
  SPMM_DEBUG_RANGES(L.stream, L.err, {{L.B, size_t(L.K) * L.N * 2}}, {{L.C, size_t(L.M) * L.N * 4}});
  spmm_tc_window_kernel<<<grid, tc::kCtaThreads, tc::smem_bytes(L.N), L.stream>>>(
      L.M, L.N, L.K, L.rowptr, L.colind, L.vals, static_cast<const uint16_t*>(L.B), L.C, L.err, cols, map);
  return cudaGetLastError();
}

}  // namespace spmm
