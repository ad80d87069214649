// Tensor-core window kernel (bf16 B): the dense window of a row block
// multiplied by the 5th-generation tensor cores (tcgen05, accumulator in
// tensor memory).
//
// For rows whose columns are local (a band), the window kernel's work is a
// dense product per row block: A_w (rows x window columns, zero where A has no
// entry) times B_w (window columns x N).  On CUDA cores that product is bound
// by the FP32 pipe; here a CTA of 128 rows hands it to tcgen05.mma:
//
//  * A's fp32 values are split exactly into three bf16 terms (hi + mid + lo
//    carries all 24 significand bits); each bf16 x bf16 product is exact in
//    fp32, so three MMAs per K-step reproduce the fp32 products and only the
//    accumulation order differs from a row loop;
//  * the window is walked in chunks of 64 columns: per chunk the CTA zeroes the
//    three A tiles, scatters its rows' values into them (K-major core
//    matrices), copies the chunk's 64 B rows straight into MN-major core
//    matrices with 16-byte cp.async (rows past K are zero-filled), and one
//    thread issues 4 K-steps x 3 terms of M=128, N, K=16 MMAs into the tensor
//    memory accumulator, committing to an mbarrier that the CTA waits on
//    (bounded) before it reuses the tiles;
//  * the epilogue reads the accumulator with tcgen05.ld (warp w reads lanes
//    32*(w%4).. and half (w/4) of the columns) and stores the rows.
//
// A tile whose column span exceeds four chunks, or one with a row whose
// columns do not strictly increase (duplicates), is computed by per-row
// gathers in the same launch.  The dense product multiplies absent entries
// as zeros, so a NaN/Inf in a B row inside the window reaches every row of
// the tile; IEEE special values are outside the accepted inputs.
#pragma once

#include <climits>

#include <cuda_bf16.h>

#include "spmm_device.cuh"
#include "spmm_internal.h"

namespace spmm {

namespace tc {

constexpr int kRows = 128;       // rows per CTA = MMA M
constexpr int kChunk = 64;       // window columns per chunk (4 K-steps of 16)
constexpr int kMaxChunks = 4;    // larger spans use the gather path
constexpr int kKStride = 128;    // bytes between K-adjacent core matrices (8 rows x 16 bytes)
constexpr int kMNStride = 1024;  // bytes between M/N-adjacent core matrices (8 along K per chunk)
constexpr int kATile = kRows * kChunk * 2;  // one bf16 term: 16 KB
constexpr int kPerThread = 32;   // nonzeros a thread holds: a tile of at most 8192 uses the tensor cores
// the column exchange (4 bytes per held nonzero) and the row ids (1 byte) use the A tiles' space
static_assert(kPerThread * 256 * 5 <= 3 * kATile, "exchange area");

__host__ __device__ constexpr size_t smem_bytes(int N) {
  return size_t(3) * kATile          // A terms hi, mid, lo
         + size_t(kChunk) * N * 2    // B chunk
         + (kRows + 8) * 4           // rowptr slice
         + 64;                       // mbarrier, TMEM address, reductions
}

// Shared-memory matrix descriptor: no swizzle, canonical core-matrix layout
// (8 rows x 16 bytes per core matrix).  For the K-major A and the MN-major B
// alike, the leading-byte-offset field holds the stride between K-adjacent core
// matrices and the stride-byte-offset field the stride between M/N-adjacent
// ones (the other assignments give wrong products on exact integer inputs).
__device__ __forceinline__ uint64_t sdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = uint64_t((saddr & 0x3FFFFu) >> 4);
  d |= uint64_t((lbo >> 4) & 0x3FFFu) << 16;
  d |= uint64_t((sbo >> 4) & 0x3FFFu) << 32;
  d |= uint64_t(1) << 46;  // descriptor version of this architecture
  return d;                // base offset 0, layout type 0 (no swizzle)
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

__device__ __forceinline__ void cp_async16_zfill(uint32_t dst, const void* src, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(valid ? 16 : 0)
               : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// 8 consecutive fp32 accumulator columns of this thread's lane.
__device__ __forceinline__ void tmem_ld8(uint32_t taddr, uint32_t (&r)[8]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
               : "r"(taddr));
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ uint16_t bf16_rn_bits(float x) { return __bfloat16_as_ushort(__float2bfloat16_rn(x)); }
__device__ __forceinline__ float bf16_bits_to_float(uint16_t b) { return __uint_as_float(uint32_t(b) << 16); }

}  // namespace tc

__global__ void __launch_bounds__(kThreads, 2)
    spmm_tc_window_kernel(int32_t M, int32_t N, int32_t K, const int32_t* __restrict__ rowptr,
                          const int32_t* __restrict__ colind, const float* __restrict__ vals,
                          const uint16_t* __restrict__ B, float* __restrict__ C, int* __restrict__ err,
                          uint32_t tmem_cols) {
  using namespace tc;
  extern __shared__ __align__(1024) unsigned char smem[];
  unsigned char* s_A = smem;                                // 3 x [16 row groups][8 k groups][8][8] bf16
  unsigned char* s_B = smem + 3 * kATile;                   // [N/8 n groups][8 k groups][8][8] bf16
  int* s_rp = reinterpret_cast<int*>(s_B + size_t(kChunk) * N * 2);
  uint64_t* s_bar = reinterpret_cast<uint64_t*>(s_rp + kRows + 8);
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(s_bar + 1);
  int* s_red = reinterpret_cast<int*>(s_tmem + 1);  // [0] min col, [1] max col, [2] flags

  const int tid = threadIdx.x, w = tid >> 5, lane = tid & 31;
  const int i0 = blockIdx.x * kRows;
  const int nrows = min(kRows, M - i0);
  const uint64_t stream_pol = policy_evict_first();

  // ---- set-up: tensor memory, barrier, rowptr slice ----------------------
  if (w == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(s_tmem)),
                 "r"(tmem_cols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  if (tid == 0) {
    mbar_init(smem_addr(s_bar), 1);
    s_red[0] = INT_MAX;
    s_red[1] = -1;
    s_red[2] = 0;
  }
  for (int t = tid; t <= nrows; t += kThreads) s_rp[t] = ld_stream(rowptr + i0 + t, stream_pol);
  fence_before();
  __syncthreads();
  fence_after();
  const uint32_t tmem = *s_tmem;
  const uint32_t bar = smem_addr(s_bar);

  // ---- the tile's nonzeros into registers (one load round) ---------------
  // Thread t holds nonzeros p0 + t + 256 i (i < kPerThread): its value and a
  // packed word, (row << 16) | (column & 0xFFFF), or kNone past the tile.
  constexpr uint32_t kNone = 0xFFFFFFFFu;
  const int p0 = s_rp[0], p1 = s_rp[nrows];
  const bool fits = p1 - p0 <= kThreads * kPerThread;
  uint32_t pk[kPerThread];
  float val[kPerThread];
  if (fits) {
    // all loads first (one latency), then the columns go through shared
    // memory (the A tiles are still free) so each thread can see the column
    // of the nonzero before each of its own
    int* s_cols = reinterpret_cast<int*>(s_A);  // [kPerThread][kThreads]
#pragma unroll
    for (int i = 0; i < kPerThread; ++i) {
      const int g = p0 + tid + kThreads * i;
      pk[i] = g < p1 ? uint32_t(ld_stream(colind + g, stream_pol)) : kNone;
      val[i] = g < p1 ? ld_stream(vals + g, stream_pol) : 0.f;
    }
#pragma unroll
    for (int i = 0; i < kPerThread; ++i) s_cols[i * kThreads + tid] = int(pk[i]);
    // the local row of every tile nonzero, one byte each (warp w fills rows w, w+8, ...)
    uint8_t* s_rowid = reinterpret_cast<uint8_t*>(s_cols + kPerThread * kThreads);
    for (int r = w; r < nrows; r += kThreads / 32)
      for (int g = s_rp[r] + lane; g < s_rp[r + 1]; g += 32) s_rowid[g - p0] = uint8_t(r);
  }
  __syncthreads();
  if (fits) {
    const int* s_cols = reinterpret_cast<const int*>(s_A);
    const uint8_t* s_rowid = reinterpret_cast<const uint8_t*>(s_cols + kPerThread * kThreads);
    int lo = INT_MAX, hi = -1;
    bool inc = true;
#pragma unroll
    for (int i = 0; i < kPerThread; ++i) {
      const int g = p0 + tid + kThreads * i;
      if (g < p1) {
        const int c = int(pk[i]);
        lo = min(lo, c);
        hi = max(hi, c);
        const int r = s_rowid[g - p0];
        if (g > s_rp[r])  // the previous nonzero is in the same row
          inc &= c > s_cols[tid > 0 ? i * kThreads + tid - 1 : (i - 1) * kThreads + kThreads - 1];
        pk[i] = (uint32_t(r) << 16) | (uint32_t(c) & 0xFFFFu);
      }
    }
    lo = __reduce_min_sync(0xffffffffu, lo);
    hi = __reduce_max_sync(0xffffffffu, hi);
    const bool all_inc = __all_sync(0xffffffffu, inc);
    if (lane == 0) {
      atomicMin(s_red + 0, lo);
      atomicMax(s_red + 1, hi);
      if (!all_inc) atomicOr(s_red + 2, 1);
    }
  } else if (tid == 0) {
    s_red[2] = 1;  // too many nonzeros to hold: gather path
  }
  __syncthreads();
  const int cmin = s_red[0], cmax = s_red[1];
  const int nchunks = cmax < 0 ? 0 : (cmax - cmin) / kChunk + 1;
  const bool use_tc = s_red[2] == 0 && nchunks <= kMaxChunks;

  if (use_tc && nchunks > 0) {
    // local column of each held nonzero: its low 16 bits minus cmin's, modulo
    // 2^16 (exact, since the span is below 2^16)
#pragma unroll
    for (int i = 0; i < kPerThread; ++i)
      if (pk[i] != kNone) pk[i] = (pk[i] & 0xFFFF0000u) | ((pk[i] - uint32_t(cmin)) & 0xFFFFu);
    const uint32_t id = idesc(N);
    const uint32_t a_base = smem_addr(s_A), b_base = smem_addr(s_B);
    // B rows c0 .. c0+63 of chunk ch (16-byte chunks: row k, column group q)
    const int qn = N / 8;
    auto issue_b = [&](int ch) {
      const int c0 = cmin + ch * kChunk;
      const uint32_t base = b_base;
      for (int t = tid; t < kChunk * qn; t += kThreads) {
        const int k = t / qn, q = t - k * qn;
        const int j = c0 + k;
        const uint32_t dst = base + uint32_t(q) * kMNStride + uint32_t(k >> 3) * kKStride + uint32_t(k & 7) * 16;
        cp_async16_zfill(dst, j < K ? static_cast<const void*>(B + size_t(j) * N + q * 8) : B, j < K);
      }
      asm volatile("cp.async.commit_group;" ::: "memory");
    };
    bool ok = true;
    for (int ch = 0; ch < nchunks; ++ch) {
      if (ch > 0) {  // the previous chunk's MMAs have read the tiles (decided by the whole CTA)
        if (!__syncthreads_and(mbar_wait_bounded(bar, uint32_t(ch - 1) & 1u, kSpinLimit))) {
          ok = false;
          break;
        }
        fence_after();
      }
      issue_b(ch);  // in flight while the A tiles are built
      // zero the three A tiles
      for (int t = tid; t < 3 * kATile / 16; t += kThreads)
        reinterpret_cast<uint4*>(s_A)[t] = make_uint4(0u, 0u, 0u, 0u);
      __syncthreads();
      // scatter the held nonzeros of this chunk: value -> three bf16 terms
#pragma unroll
      for (int i = 0; i < kPerThread; ++i) {
        const int k = int(pk[i] & 0xFFFFu) - ch * kChunk;
        if (pk[i] != kNone && k >= 0 && k < kChunk) {
          const int r = int(pk[i] >> 16);
          const float v = val[i];
          const uint16_t h = bf16_rn_bits(v);
          const float r1 = v - bf16_bits_to_float(h);
          const uint16_t m = bf16_rn_bits(r1);
          const uint16_t l = bf16_rn_bits(r1 - bf16_bits_to_float(m));
          const uint32_t off = uint32_t(r >> 3) * kMNStride + uint32_t(k >> 3) * kKStride + uint32_t(r & 7) * 16 +
                               uint32_t(k & 7) * 2;
          *reinterpret_cast<uint16_t*>(s_A + off) = h;
          *reinterpret_cast<uint16_t*>(s_A + kATile + off) = m;
          *reinterpret_cast<uint16_t*>(s_A + 2 * kATile + off) = l;
        }
      }
      asm volatile("cp.async.wait_group 0;" ::: "memory");  // this chunk's B rows
      fence_proxy_async();  // generic-proxy writes become visible to the tensor cores
      fence_before();
      __syncthreads();
      if (tid == 0) {
        fence_after();
        const uint32_t bbuf = b_base;
#pragma unroll
        for (int ks = 0; ks < kChunk / 16; ++ks) {
#pragma unroll
          for (int term = 0; term < 3; ++term) {
            const uint64_t a = sdesc(a_base + uint32_t(term) * kATile + uint32_t(2 * ks) * kKStride, kKStride, kMNStride);
            const uint64_t b = sdesc(bbuf + uint32_t(2 * ks) * kKStride, kKStride, kMNStride);
            mma(tmem, a, b, id, ch > 0 || ks > 0 || term > 0);
          }
        }
        commit(bar);
      }
    }
    if (ok) ok = __syncthreads_and(mbar_wait_bounded(bar, uint32_t(nchunks - 1) & 1u, kSpinLimit));
    if (!ok) {  // the tensor cores did not finish: report, write nothing
      if (tid == 0) atomicOr(err, kErrStageTimeout);
    } else {
      fence_after();
      // epilogue: warp w reads lanes 32*(w%4).. (its 32 rows) and half w/4 of
      // the columns, 32 at a time; a per-warp shared-memory transpose (rows of
      // 36 floats) turns them into 4-row x 128-byte coalesced stores
      const int q = w & 3, half = w >> 2;
      const int cols = N / 2;
      float* tw = reinterpret_cast<float*>(s_A) + w * (32 * 36);
      const int rr = lane >> 3, cc = (lane & 7) * 4;  // store phase: row (of 4) and column of this lane
      for (int c = half * cols; c < (half + 1) * cols; c += 32) {  // N/2 is a multiple of 8
        const int n8 = min(32, (half + 1) * cols - c) / 8;
        uint32_t v[4][8];
#pragma unroll
        for (int j = 0; j < 4; ++j)
          if (j < n8) tc::tmem_ld8(tmem + (uint32_t(32 * q) << 16) + uint32_t(c + 8 * j), v[j]);
        tmem_wait_ld();
        __syncwarp();
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          *reinterpret_cast<uint4*>(tw + lane * 36 + 8 * j) = make_uint4(v[j][0], v[j][1], v[j][2], v[j][3]);
          *reinterpret_cast<uint4*>(tw + lane * 36 + 8 * j + 4) = make_uint4(v[j][4], v[j][5], v[j][6], v[j][7]);
        }
        __syncwarp();
#pragma unroll
        for (int k = 0; k < 8; ++k) {  // rows 4k .. 4k+3 of the warp's 32
          const int lr = 4 * k + rr;
          const int row = i0 + 32 * q + lr;
          if (row < M && cc < 8 * n8) {
            const float4 x = *reinterpret_cast<const float4*>(tw + lr * 36 + cc);
            st_stream4(C + size_t(row) * N + c + cc, x.x, x.y, x.z, x.w);
          }
        }
      }
    }
  } else if (use_tc) {  // no nonzeros in the tile: zero rows
    for (int t = tid; t < nrows * (N / 4); t += kThreads) {
      const int r = t / (N / 4), c4 = t - r * (N / 4);
      st_stream4(C + size_t(i0 + r) * N + 4 * c4, 0.f, 0.f, 0.f, 0.f);
    }
  } else {  // gather path: warp w computes rows w, w + 8, ... (8 columns per lane per pass)
    for (int r = w; r < nrows; r += kThreads / 32) {
      const int start = s_rp[r], end = s_rp[r + 1];
      for (int c0 = lane * 8; c0 < N; c0 += 32 * 8) {
        FVec<8> acc;
        acc.zero();
        for (int g = start; g < end; ++g) {
          const int c = __ldg(colind + g);
          BSlice<uint16_t, 8> bs;
          bs.load(B + size_t(c) * N + c0);
          FVec<8> b;
          bs.widen(b);
          acc.fma(pair(__ldg(vals + g)), b);
        }
        store_c<8>(C + size_t(i0 + r) * N + c0, acc);
      }
    }
  }

  // ---- release the tensor memory -----------------------------------------
  fence_before();
  __syncthreads();
  if (w == 0) {
    fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(tmem_cols) : "memory");
  }
}

inline cudaError_t launch_tc_window(const Launch& L) {
  const size_t smem = tc::smem_bytes(L.N);
  static bool attr_set[kMaxDevices] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= kMaxDevices || !attr_set[dev]) {
    e = cudaFuncSetAttribute(spmm_tc_window_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             int(tc::smem_bytes(256)));
    if (e != cudaSuccess) return e;
    if (dev < kMaxDevices) attr_set[dev] = true;
  }
  uint32_t cols = 32;
  while (cols < uint32_t(L.N)) cols <<= 1;
  const unsigned grid = unsigned((int64_t(L.M) + tc::kRows - 1) / tc::kRows);
  spmm_tc_window_kernel<<<grid, kThreads, smem, L.stream>>>(L.M, L.N, L.K, L.rowptr, L.colind, L.vals,
                                                            static_cast<const uint16_t*>(L.B), L.C, L.err, cols);
  return cudaGetLastError();
}

}  // namespace spmm
