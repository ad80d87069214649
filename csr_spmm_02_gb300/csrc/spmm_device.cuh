// Device building blocks shared by the SpMM kernels (sm_103a).
//
//  * FVec<VEC>: a lane's VEC fp32 accumulators, as float2 pairs for packed
//    FMAs (fma.rn.f32x2: two IEEE fp32 FMAs per instruction, bitwise equal
//    to two scalar fmaf).
//  * BSlice<BT, VEC>: one lane's VEC consecutive elements of a B row, loaded
//    raw in one 16-byte (or scalar) load and widened to fp32 at use.  bf16 is
//    the top half of an IEEE binary32, so widening is an exact 16-bit shift.
//  * streaming (evict-first) stores of C rows, which are written once.
//  * 1-D bulk copies (cp.async.bulk, the TMA engine's non-tensor form) into
//    shared memory completed on an mbarrier, with a bounded wait.
#pragma once

#include <cstdint>
#include <initializer_list>

#include <cuda_runtime.h>

namespace spmm {

constexpr int kThreads = 256;           // threads per CTA for every SpMM kernel
constexpr uint32_t kSpinLimit = 1u << 22;  // bound on mbarrier polls before giving up

// Device error word bits.
constexpr int kErrStageTimeout = 1;  // a bounded wait gave up
constexpr int kErrInvalidCsr = 2;    // rowptr[M] differs from the nnz the caller passed
constexpr int kErrBounds = 4;        // (bounds-checked build) an access outside its buffers was skipped

// The first wait of a kernel for its staged copies.  A test build lowers it
// (SPMM_STAGE_SPIN_LIMIT=1: one non-blocking look) to make that wait give up
// while the copies are still in flight; the kernel then still waits
// (kSpinLimit) for them to land before it leaves.
#ifndef SPMM_STAGE_SPIN_LIMIT
#define SPMM_STAGE_SPIN_LIMIT kSpinLimit
#endif
constexpr uint32_t kStageSpinLimit = SPMM_STAGE_SPIN_LIMIT;

#ifndef SPMM_L2_HINTS
#define SPMM_L2_HINTS 1  // stream A and C with evict-first so B's reused rows stay in L2
#endif
#ifndef SPMM_B_EVICT_LAST
#define SPMM_B_EVICT_LAST 0  // give B gathers evict-last priority in L2
#endif

// ---------------------------------------------------------------------------
// Bounds-checked build (-DSPMM_DEBUG_BOUNDS): every B-row gather
// (BSlice::load, the row kernel's policy loads, the window kernel's cp.async
// staging of B rows) and every C / output store (st_stream4, st_stream1,
// st_plain1) checks its address against the buffers the launch registered;
// an access outside them is skipped and kErrBounds is set in the launch's
// error word.  Nothing traps: the kernel runs to its end and the host reads
// the word.  The ranges live in a per-translation-unit __device__ variable
// that each launch wrapper fills on the launch stream before its launch.
// ---------------------------------------------------------------------------
#ifdef SPMM_DEBUG_BOUNDS
struct DebugRanges {
  uint64_t load_lo[3], load_hi[3];    // buffers gathered from
  uint64_t store_lo[2], store_hi[2];  // buffers stored to
  int* err;
};
static __device__ DebugRanges g_debug_ranges;

__device__ __forceinline__ bool debug_access_ok(const void* p, int bytes, const uint64_t* lo, const uint64_t* hi,
                                                int n) {
  const uint64_t a = reinterpret_cast<uint64_t>(p);
  for (int k = 0; k < n; ++k)
    if (a >= lo[k] && a + uint64_t(bytes) <= hi[k]) return true;
  if (g_debug_ranges.err) atomicOr(g_debug_ranges.err, kErrBounds);
  return false;
}
__device__ __forceinline__ bool debug_load_ok(const void* p, int bytes) {
  return debug_access_ok(p, bytes, g_debug_ranges.load_lo, g_debug_ranges.load_hi, 3);
}
__device__ __forceinline__ bool debug_store_ok(const void* p, int bytes) {
  return debug_access_ok(p, bytes, g_debug_ranges.store_lo, g_debug_ranges.store_hi, 2);
}

struct DebugBuffer {
  const void* p;
  size_t bytes;
};
// Register the buffers of the next launch on `s` (up to three gathered, two stored).
static inline cudaError_t debug_ranges(cudaStream_t s, int* err, std::initializer_list<DebugBuffer> loads,
                                       std::initializer_list<DebugBuffer> stores) {
  DebugRanges h{};
  int k = 0;
  for (const DebugBuffer& b : loads) {
    h.load_lo[k] = reinterpret_cast<uint64_t>(b.p);
    h.load_hi[k] = h.load_lo[k] + (b.p ? b.bytes : 0);
    ++k;
  }
  k = 0;
  for (const DebugBuffer& b : stores) {
    h.store_lo[k] = reinterpret_cast<uint64_t>(b.p);
    h.store_hi[k] = h.store_lo[k] + (b.p ? b.bytes : 0);
    ++k;
  }
  h.err = err;
  return cudaMemcpyToSymbolAsync(g_debug_ranges, &h, sizeof h, 0, cudaMemcpyHostToDevice, s);
}
#define SPMM_DEBUG_LOAD_GUARD(p, bytes, on_fail) \
  if (!debug_load_ok(p, bytes)) { on_fail; return; }
#define SPMM_DEBUG_STORE_GUARD(p, bytes) \
  if (!debug_store_ok(p, bytes)) return;
#define SPMM_DEBUG_RANGES(...) \
  do { const cudaError_t de_ = debug_ranges(__VA_ARGS__); if (de_ != cudaSuccess) return de_; } while (0)
#else
#define SPMM_DEBUG_LOAD_GUARD(p, bytes, on_fail)
#define SPMM_DEBUG_STORE_GUARD(p, bytes)
#define SPMM_DEBUG_RANGES(...) \
  do { } while (0)
#endif

// ---------------------------------------------------------------------------
// L2 cache policies.  A (colind, vals, rowptr) is read once and C is written
// once: both are marked evict-first, so the L2 keeps the rows of B that many
// nonzeros reuse (the temporal locality the kkmem page attributes to B).
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// Read-once loads of A's arrays.
__device__ __forceinline__ int ld_stream(const int* p, uint64_t pol) {
#if SPMM_L2_HINTS
  int v;
  asm volatile("ld.global.nc.L2::cache_hint.b32 %0, [%1], %2;" : "=r"(v) : "l"(p), "l"(pol));
  return v;
#else
  return __ldg(p);
#endif
}
__device__ __forceinline__ float ld_stream(const float* p, uint64_t pol) {
  return __int_as_float(ld_stream(reinterpret_cast<const int*>(p), pol));
}

// ---------------------------------------------------------------------------
// FVec<VEC>: VEC fp32 values of one lane.  Even widths are kept as float2
// pairs so packed FMAs (fma.rn.f32x2 through __ffma2_rn: two IEEE fp32 FMAs,
// bitwise equal to two fmaf) need no register moves.
// ---------------------------------------------------------------------------
template <int VEC>
struct FVec {
  static_assert(VEC % 2 == 0, "even widths only");
  float2 p[VEC / 2];
  __device__ __forceinline__ void zero() {
#pragma unroll
    for (int j = 0; j < VEC / 2; ++j) p[j] = make_float2(0.f, 0.f);
  }
  __device__ __forceinline__ void fma(float2 vv, const FVec& b) {  // this += (v, v) * b
#pragma unroll
    for (int j = 0; j < VEC / 2; ++j) p[j] = __ffma2_rn(vv, b.p[j], p[j]);
  }
  __device__ __forceinline__ void add(const FVec& o) {
#pragma unroll
    for (int j = 0; j < VEC / 2; ++j) p[j] = make_float2(p[j].x + o.p[j].x, p[j].y + o.p[j].y);
  }
  __device__ __forceinline__ void add_shfl_xor(int mask) {
#pragma unroll
    for (int j = 0; j < VEC / 2; ++j) {
      p[j].x += __shfl_xor_sync(0xffffffffu, p[j].x, mask);
      p[j].y += __shfl_xor_sync(0xffffffffu, p[j].y, mask);
    }
  }
  __device__ __forceinline__ void load_plain(const float* src) {  // 16-byte aligned
#pragma unroll
    for (int j = 0; j < VEC / 2; j += 2) {
      const float4 t = *reinterpret_cast<const float4*>(src + 2 * j);
      p[j] = make_float2(t.x, t.y);
      p[j + 1] = make_float2(t.z, t.w);
    }
  }
  __device__ __forceinline__ void store_plain(float* dst) const {
#pragma unroll
    for (int j = 0; j < VEC / 2; j += 2)
      *reinterpret_cast<float4*>(dst + 2 * j) = make_float4(p[j].x, p[j].y, p[j + 1].x, p[j + 1].y);
  }
};

template <>
struct FVec<1> {
  float x;
  __device__ __forceinline__ void zero() { x = 0.f; }
  __device__ __forceinline__ void fma(float2 vv, const FVec& b) { x = fmaf(vv.x, b.x, x); }
  __device__ __forceinline__ void add(const FVec& o) { x += o.x; }
  __device__ __forceinline__ void add_shfl_xor(int mask) { x += __shfl_xor_sync(0xffffffffu, x, mask); }
  __device__ __forceinline__ void load_plain(const float* src) { x = *src; }
  __device__ __forceinline__ void store_plain(float* dst) const { *dst = x; }
};

// ---------------------------------------------------------------------------
// B slices: one 16-byte (or scalar) load of a lane's VEC elements of a B row,
// widened to fp32 at use.  bf16 is the top half of an IEEE binary32, so
// widening is an exact 16-bit shift.
// ---------------------------------------------------------------------------
template <typename BT, int VEC>
struct BSlice;

template <>
struct BSlice<float, 4> {
  float4 r;
  __device__ __forceinline__ void load(const float* p) {
    SPMM_DEBUG_LOAD_GUARD(p, 16, r = make_float4(0.f, 0.f, 0.f, 0.f))
    r = __ldg(reinterpret_cast<const float4*>(p));
  }
  __device__ __forceinline__ void load_shared(const float* p) { r = *reinterpret_cast<const float4*>(p); }
  __device__ __forceinline__ void widen(FVec<4>& o) const {
    o.p[0] = make_float2(r.x, r.y);
    o.p[1] = make_float2(r.z, r.w);
  }
};

template <>
struct BSlice<float, 1> {
  float r;
  __device__ __forceinline__ void load(const float* p) {
    SPMM_DEBUG_LOAD_GUARD(p, 4, r = 0.f)
    r = __ldg(p);
  }
  __device__ __forceinline__ void widen(FVec<1>& o) const { o.x = r; }
};

__device__ __forceinline__ float2 bf16x2_widen(uint32_t w) {
  return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}

template <>
struct BSlice<uint16_t, 8> {
  uint4 r;
  __device__ __forceinline__ void load(const uint16_t* p) {
    SPMM_DEBUG_LOAD_GUARD(p, 16, r = make_uint4(0u, 0u, 0u, 0u))
    r = __ldg(reinterpret_cast<const uint4*>(p));
  }
  __device__ __forceinline__ void load_shared(const uint16_t* p) { r = *reinterpret_cast<const uint4*>(p); }
  __device__ __forceinline__ void widen(FVec<8>& o) const {
    o.p[0] = bf16x2_widen(r.x);
    o.p[1] = bf16x2_widen(r.y);
    o.p[2] = bf16x2_widen(r.z);
    o.p[3] = bf16x2_widen(r.w);
  }
};

template <>
struct BSlice<uint16_t, 1> {
  unsigned short r;
  __device__ __forceinline__ void load(const uint16_t* p) {
    SPMM_DEBUG_LOAD_GUARD(p, 2, r = 0)
    r = __ldg(reinterpret_cast<const unsigned short*>(p));
  }
  __device__ __forceinline__ void widen(FVec<1>& o) const { o.x = __uint_as_float(uint32_t(r) << 16); }
};

__device__ __forceinline__ float2 pair(float v) { return make_float2(v, v); }

// ---------------------------------------------------------------------------
// Semirings: C[i][n] = (+) over row i of vals (x) B (the Sgap page's
// generalised reduction, sparse-dense hybrid algebra, Eq. 3).  Code SR =
// 2 * add + mul with add 0 sum, 1 min, 2 max and mul 0 multiply, 1 add;
// SR = 0 is the ordinary SpMM, which keeps its packed-FMA path.
// ---------------------------------------------------------------------------
template <int SR>
__device__ __forceinline__ float sr_identity() {
  return SR / 2 == 0 ? 0.f : __int_as_float(SR / 2 == 1 ? 0x7f800000 : 0xff800000);  // 0, +inf, -inf
}
template <int SR>
__device__ __forceinline__ float sr_plus(float a, float b) {
  if constexpr (SR / 2 == 0) return a + b;
  else if constexpr (SR / 2 == 1) return fminf(a, b);
  else return fmaxf(a, b);
}
template <int SR>
__device__ __forceinline__ float sr_times(float v, float b) {
  if constexpr (SR % 2 == 0) return v * b;
  else return v + b;
}
// Every element of `a` set to the identity of (+).
template <int SR, int VEC>
__device__ __forceinline__ void sr_reset(FVec<VEC>& a) {
  if constexpr (VEC == 1) {
    a.x = sr_identity<SR>();
  } else {
#pragma unroll
    for (int j = 0; j < VEC / 2; ++j) a.p[j] = make_float2(sr_identity<SR>(), sr_identity<SR>());
  }
}
// a (+)= v (x) b where `valid`, else unchanged.
template <int SR, int VEC>
__device__ __forceinline__ void sr_apply(FVec<VEC>& a, float v, const FVec<VEC>& b, bool valid) {
  if constexpr (VEC == 1) {
    a.x = valid ? sr_plus<SR>(a.x, sr_times<SR>(v, b.x)) : a.x;
  } else {
#pragma unroll
    for (int j = 0; j < VEC / 2; ++j) {
      const float x = sr_plus<SR>(a.p[j].x, sr_times<SR>(v, b.p[j].x));
      const float y = sr_plus<SR>(a.p[j].y, sr_times<SR>(v, b.p[j].y));
      a.p[j] = valid ? make_float2(x, y) : a.p[j];
    }
  }
}
// a (+)= o
template <int SR, int VEC>
__device__ __forceinline__ void sr_combine(FVec<VEC>& a, const FVec<VEC>& o) {
  if constexpr (VEC == 1) {
    a.x = sr_plus<SR>(a.x, o.x);
  } else {
#pragma unroll
    for (int j = 0; j < VEC / 2; ++j) a.p[j] = make_float2(sr_plus<SR>(a.p[j].x, o.p[j].x), sr_plus<SR>(a.p[j].y, o.p[j].y));
  }
}
// a (+)= the lane (lane ^ mask)'s a
template <int SR, int VEC>
__device__ __forceinline__ void sr_combine_shfl_xor(FVec<VEC>& a, int mask) {
  if constexpr (VEC == 1) {
    a.x = sr_plus<SR>(a.x, __shfl_xor_sync(0xffffffffu, a.x, mask));
  } else {
#pragma unroll
    for (int j = 0; j < VEC / 2; ++j) {
      a.p[j].x = sr_plus<SR>(a.p[j].x, __shfl_xor_sync(0xffffffffu, a.p[j].x, mask));
      a.p[j].y = sr_plus<SR>(a.p[j].y, __shfl_xor_sync(0xffffffffu, a.p[j].y, mask));
    }
  }
}

// ---------------------------------------------------------------------------
// C stores (each C element is written once: streaming / evict-first)
// ---------------------------------------------------------------------------
__device__ __forceinline__ void st_stream4(float* p, float x, float y, float z, float w) {
  SPMM_DEBUG_STORE_GUARD(p, 16)
#if SPMM_L2_HINTS
  asm volatile("st.global.L2::cache_hint.v4.f32 [%0], {%1,%2,%3,%4}, %5;" ::"l"(p), "f"(x), "f"(y), "f"(z), "f"(w),
               "l"(policy_evict_first())
               : "memory");
#else
  __stcs(reinterpret_cast<float4*>(p), make_float4(x, y, z, w));
#endif
}
__device__ __forceinline__ void st_stream1(float* p, float x) {
  SPMM_DEBUG_STORE_GUARD(p, 4)
#if SPMM_L2_HINTS
  asm volatile("st.global.L2::cache_hint.f32 [%0], %1, %2;" ::"l"(p), "f"(x), "l"(policy_evict_first()) : "memory");
#else
  __stcs(p, x);
#endif
}

// A plain (write-back) store of one output value.
__device__ __forceinline__ void st_plain1(float* p, float x) {
  SPMM_DEBUG_STORE_GUARD(p, 4)
  *p = x;
}

template <int VEC>
__device__ __forceinline__ void store_c(float* p, const FVec<VEC>& a) {
  if constexpr (VEC == 1) {
    st_stream1(p, a.x);
  } else {
#pragma unroll
    for (int j = 0; j < VEC / 2; j += 2) st_stream4(p + 2 * j, a.p[j].x, a.p[j].y, a.p[j + 1].x, a.p[j + 1].y);
  }
}

// ---------------------------------------------------------------------------
// mbarrier + 1-D bulk copy (global -> shared)
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

// dst (shared) and src (global) 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
#if SPMM_L2_HINTS
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
          dst),
      "l"(src), "r"(bytes), "r"(bar), "l"(policy_evict_first())
      : "memory");
#else
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
#endif
}

// One non-blocking look at the barrier's phase `parity` (test_wait never
// suspends the thread, unlike try_wait); true when it has completed.
__device__ __forceinline__ bool mbar_test(uint32_t bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(bar), "r"(parity)
      : "memory");
  return done != 0;
}

// Poll the barrier's phase `parity` at most `limit` times; true when it completed.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity, uint32_t limit) {
  for (uint32_t it = 0; it < limit; ++it) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(bar), "r"(parity)
        : "memory");
    if (done) return true;
  }
  return false;
}



// Stage one merge-path range of a CTA in shared memory: colind[p0, p1) at
// s_col[g - (p0 & ~3)] and, with VALS, vals[p0, p1) at s_val[g - (p0 & ~3)];
// rowptr[i0 .. i1] at s_rp[g - (i0 & ~3)].  The 16-byte aligned interiors go
// by 1-D bulk copies (the TMA engine) that complete on the mbarrier s_bar,
// initialised here for one arrival; the at most three unaligned entries at
// each end, or everything when a pointer is misaligned, by plain loads (A is
// read once: evict-first).  pre_barrier() runs before the first CTA barrier
// (per-CTA shared state to set).  Returns false on every thread when the wait
// for the copies gave up (kErrStageTimeout set in *err, after waiting again
// for the copies in flight): the caller returns.  kThreads threads.
template <bool VALS, typename Pre>
__device__ __forceinline__ bool stage_range(const int32_t* __restrict__ colind, const float* __restrict__ vals,
                                            const int32_t* __restrict__ rowptr, int i0, int p0, int i1, int p1,
                                            int* s_col, float* s_val, int* s_rp, uint64_t* s_bar, int* err,
                                            Pre pre_barrier) {
  const int tid = threadIdx.x;
  const int nbase = p0 & ~3, rbase = i0 & ~3;
  const uint64_t stream_pol = policy_evict_first();
  const uint32_t bar = smem_addr(s_bar);
  const bool bulk_ok = ((reinterpret_cast<uintptr_t>(colind) | (VALS ? reinterpret_cast<uintptr_t>(vals) : 0) |
                         reinterpret_cast<uintptr_t>(rowptr)) & 15) == 0;
  const int ca = (p0 + 3) & ~3, cb = p1 & ~3;        // 16-byte aligned interior of [p0, p1)
  const int ra = (i0 + 3) & ~3, rb = (i1 + 1) & ~3;  // ... of [i0, i1 + 1)
  const bool c_bulk = bulk_ok && cb > ca;
  const bool r_bulk = bulk_ok && rb > ra;
  if (tid == 0) mbar_init(bar, 1);
  pre_barrier();
  __syncthreads();
  if (tid == 0) {
    mbar_arrive_expect_tx(bar, (c_bulk ? (VALS ? 8u : 4u) * uint32_t(cb - ca) : 0u) +
                                   (r_bulk ? 4u * uint32_t(rb - ra) : 0u));
    if (c_bulk) {
      bulk_g2s(smem_addr(s_col + (ca - nbase)), colind + ca, 4u * uint32_t(cb - ca), bar);
      if (VALS) bulk_g2s(smem_addr(s_val + (ca - nbase)), vals + ca, 4u * uint32_t(cb - ca), bar);
    }
    if (r_bulk) bulk_g2s(smem_addr(s_rp + (ra - rbase)), rowptr + ra, 4u * uint32_t(rb - ra), bar);
  }
  if (c_bulk) {  // at most 3 leading and 3 trailing nonzeros
    const int g = tid < 4 ? p0 + tid : cb + (tid - 4);
    if (tid < 8 && ((tid < 4 && g < ca) || (tid >= 4 && g < p1))) {
      s_col[g - nbase] = ld_stream(colind + g, stream_pol);
      if (VALS) s_val[g - nbase] = ld_stream(vals + g, stream_pol);
    }
  } else {
    for (int g = p0 + tid; g < p1; g += kThreads) {
      s_col[g - nbase] = ld_stream(colind + g, stream_pol);
      if (VALS) s_val[g - nbase] = ld_stream(vals + g, stream_pol);
    }
  }
  if (r_bulk) {
    const int g = tid < 4 ? i0 + tid : rb + (tid - 4);
    if (tid < 8 && ((tid < 4 && g < ra) || (tid >= 4 && g <= i1))) s_rp[g - rbase] = ld_stream(rowptr + g, stream_pol);
  } else {
    for (int g = i0 + tid; g <= i1; g += kThreads) s_rp[g - rbase] = ld_stream(rowptr + g, stream_pol);
  }
  // (the test build's limit of one poll takes a single non-blocking look)
  const bool staged = kStageSpinLimit <= 1 ? mbar_test(bar, 0) : mbar_wait_bounded(bar, 0, kStageSpinLimit);
  if (__syncthreads_or(!staged)) {
    if (tid == 0) atomicOr(err, kErrStageTimeout);
    mbar_wait_bounded(bar, 0, kSpinLimit);  // let copies in flight land before leaving
    return false;
  }
  return true;
}

}  // namespace spmm
