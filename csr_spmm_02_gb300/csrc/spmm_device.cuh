// Device building blocks shared by the SpMM kernels (sm_103a).
//
//  * BSlice<BT, VEC>: one lane's VEC consecutive elements of a B row, loaded
//    raw in one 16-byte (or scalar) load and widened to fp32 at use.  bf16 is
//    the top half of an IEEE binary32, so widening is an exact 16-bit shift.
//  * axpy: acc += v * b with packed fma.rn.f32x2 (two IEEE fp32 FMAs per
//    instruction; bitwise equal to two scalar fmaf).
//  * streaming (evict-first) stores of C rows, which are written once.
//  * 1-D bulk copies (cp.async.bulk, the TMA engine's non-tensor form) into
//    shared memory completed on an mbarrier, with a bounded wait.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace spmm {

constexpr int kThreads = 256;           // threads per CTA for every SpMM kernel
constexpr uint32_t kSpinLimit = 1u << 22;  // bound on mbarrier polls before giving up

#ifndef SPMM_L2_HINTS
#define SPMM_L2_HINTS 1  // stream A and C with evict-first so B's reused rows stay in L2
#endif
#ifndef SPMM_B_EVICT_LAST
#define SPMM_B_EVICT_LAST 0  // give B gathers evict-last priority in L2
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
// B slices
// ---------------------------------------------------------------------------
template <typename BT, int VEC>
struct BSlice;

template <>
struct BSlice<float, 4> {
  float4 r;
  __device__ __forceinline__ void load(const float* p) { r = __ldg(reinterpret_cast<const float4*>(p)); }
  __device__ __forceinline__ void load_if(const float* p, bool pred) {
#if SPMM_B_EVICT_LAST
    r = make_float4(0.f, 0.f, 0.f, 0.f);
    if (pred)
      asm volatile("ld.global.nc.L2::cache_hint.v4.f32 {%0,%1,%2,%3}, [%4], %5;"
                   : "=f"(r.x), "=f"(r.y), "=f"(r.z), "=f"(r.w) : "l"(p), "l"(policy_evict_last()));
#else
    r = pred ? __ldg(reinterpret_cast<const float4*>(p)) : make_float4(0.f, 0.f, 0.f, 0.f);
#endif
  }
  __device__ __forceinline__ void widen(float (&o)[4]) const {
    o[0] = r.x; o[1] = r.y; o[2] = r.z; o[3] = r.w;
  }
};

template <>
struct BSlice<float, 1> {
  float r;
  __device__ __forceinline__ void load(const float* p) { r = __ldg(p); }
  __device__ __forceinline__ void load_if(const float* p, bool pred) { r = pred ? __ldg(p) : 0.f; }
  __device__ __forceinline__ void widen(float (&o)[1]) const { o[0] = r; }
};

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

template <>
struct BSlice<uint16_t, 8> {
  uint4 r;
  __device__ __forceinline__ void load(const uint16_t* p) { r = __ldg(reinterpret_cast<const uint4*>(p)); }
  __device__ __forceinline__ void load_if(const uint16_t* p, bool pred) {
#if SPMM_B_EVICT_LAST
    r = make_uint4(0u, 0u, 0u, 0u);
    if (pred)
      asm volatile("ld.global.nc.L2::cache_hint.v4.u32 {%0,%1,%2,%3}, [%4], %5;"
                   : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p), "l"(policy_evict_last()));
#else
    r = pred ? __ldg(reinterpret_cast<const uint4*>(p)) : make_uint4(0u, 0u, 0u, 0u);
#endif
  }
  __device__ __forceinline__ void widen(float (&o)[8]) const {
    o[0] = bf16_lo(r.x); o[1] = bf16_hi(r.x);
    o[2] = bf16_lo(r.y); o[3] = bf16_hi(r.y);
    o[4] = bf16_lo(r.z); o[5] = bf16_hi(r.z);
    o[6] = bf16_lo(r.w); o[7] = bf16_hi(r.w);
  }
};

template <>
struct BSlice<uint16_t, 1> {
  unsigned short r;
  __device__ __forceinline__ void load(const uint16_t* p) {
    r = __ldg(reinterpret_cast<const unsigned short*>(p));
  }
  __device__ __forceinline__ void load_if(const uint16_t* p, bool pred) {
    r = pred ? __ldg(reinterpret_cast<const unsigned short*>(p)) : (unsigned short)0;
  }
  __device__ __forceinline__ void widen(float (&o)[1]) const { o[0] = __uint_as_float(uint32_t(r) << 16); }
};

// ---------------------------------------------------------------------------
// acc += v * b.  The scalar v is packed once per nonzero into a (v, v) pair
// that every packed FMA of that nonzero reuses.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint64_t pack_pair(float v) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %1};" : "=l"(r) : "f"(v));
  return r;
}

__device__ __forceinline__ void fma2(float& a0, float& a1, uint64_t vv, float b0, float b1) {
  asm("{\n\t.reg .b64 rb, rc;\n\t"
      "mov.b64 rb, {%3, %4};\n\t"
      "mov.b64 rc, {%0, %1};\n\t"
      "fma.rn.f32x2 rc, %2, rb, rc;\n\t"
      "mov.b64 {%0, %1}, rc;\n\t}"
      : "+f"(a0), "+f"(a1)
      : "l"(vv), "f"(b0), "f"(b1));
}

template <int VEC>
__device__ __forceinline__ void axpy(float (&acc)[VEC], float v, uint64_t vv, const float (&b)[VEC]) {
  if constexpr (VEC % 2 == 0) {
#pragma unroll
    for (int j = 0; j < VEC; j += 2) fma2(acc[j], acc[j + 1], vv, b[j], b[j + 1]);
  } else {
#pragma unroll
    for (int j = 0; j < VEC; ++j) acc[j] = fmaf(v, b[j], acc[j]);
  }
}

// ---------------------------------------------------------------------------
// C stores (each C element is written once: streaming / evict-first)
// ---------------------------------------------------------------------------
__device__ __forceinline__ void st_stream4(float* p, float x, float y, float z, float w) {
#if SPMM_L2_HINTS
  asm volatile("st.global.L2::cache_hint.v4.f32 [%0], {%1,%2,%3,%4}, %5;" ::"l"(p), "f"(x), "f"(y), "f"(z), "f"(w),
               "l"(policy_evict_first())
               : "memory");
#else
  __stcs(reinterpret_cast<float4*>(p), make_float4(x, y, z, w));
#endif
}
__device__ __forceinline__ void st_stream1(float* p, float x) {
#if SPMM_L2_HINTS
  asm volatile("st.global.L2::cache_hint.f32 [%0], %1, %2;" ::"l"(p), "f"(x), "l"(policy_evict_first()) : "memory");
#else
  __stcs(p, x);
#endif
}

template <int VEC>
__device__ __forceinline__ void store_c(float* p, const float (&a)[VEC]) {
  if constexpr (VEC % 4 == 0) {
#pragma unroll
    for (int j = 0; j < VEC; j += 4) st_stream4(p + j, a[j], a[j + 1], a[j + 2], a[j + 3]);
  } else {
#pragma unroll
    for (int j = 0; j < VEC; ++j) st_stream1(p + j, a[j]);
  }
}

template <int VEC>
__device__ __forceinline__ void store_f4(float* p, const float (&a)[VEC]) {  // plain store
  if constexpr (VEC % 4 == 0) {
#pragma unroll
    for (int j = 0; j < VEC; j += 4)
      *reinterpret_cast<float4*>(p + j) = make_float4(a[j], a[j + 1], a[j + 2], a[j + 3]);
  } else {
#pragma unroll
    for (int j = 0; j < VEC; ++j) p[j] = a[j];
  }
}

template <int VEC>
__device__ __forceinline__ void load_f4(const float* p, float (&a)[VEC]) {  // plain load
  if constexpr (VEC % 4 == 0) {
#pragma unroll
    for (int j = 0; j < VEC; j += 4) {
      float4 t = *reinterpret_cast<const float4*>(p + j);
      a[j] = t.x; a[j + 1] = t.y; a[j + 2] = t.z; a[j + 3] = t.w;
    }
  } else {
#pragma unroll
    for (int j = 0; j < VEC; ++j) a[j] = p[j];
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

// Device error word bits.
constexpr int kErrStageTimeout = 1;

}  // namespace spmm
