// Plan construction (row statistics, kernel choice, merge-path partition),
// CSR validation and the deterministic fixup of rows split across CTAs.
#include <algorithm>
#include <cstdint>
#include <mutex>
#include <new>

#include "spmm_device.cuh"
#include "spmm_internal.h"

namespace spmm {

// One pass over rowptr.  stats[0] = longest row, stats[1] = number of empty
// rows, stats[2] = rowptr[M] (block-reduced, one atomic per block).  With
// part: the merge-path coordinates of the P+1 range starts, found without a
// search: row i's end item sits at e(i) = rowptr[i+1] + i, so the diagonals
// c*T with e(i-1) < c*T <= e(i) start inside row i, at nonzero c*T - i;
// part[P] = (M, nnz) closes the sequence.  nnz and P are the caller's (a
// rowptr[M] that differs is caught from stats[2] on the host; no index past
// part[P] is written either way).
__global__ void __launch_bounds__(kThreads) plan_rows_kernel(const int32_t* __restrict__ rowptr, int32_t M,
                                                             int64_t nnz, int64_t T, int32_t P,
                                                             int* __restrict__ stats, int2* __restrict__ part) {
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    stats[2] = __ldg(rowptr + M);
    if (part) part[P] = make_int2(M, int(nnz));
  }
  int longest = 0, empty = 0;
  for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < M; i += int64_t(gridDim.x) * blockDim.x) {
    const int a = __ldg(rowptr + i), b = __ldg(rowptr + i + 1);
    const int len = b - a;
    longest = max(longest, len);
    empty += len == 0;
    if (part) {
      // Row i's items end at e(i) = b + i, below 2^32 since nnz and M are
      // each below 2^31: 32-bit arithmetic.  The diagonals that start inside
      // row i are the multiples of T in (e(i-1), e(i)] = (e - len - 1, e];
      // with q = e / T and r = e - q*T there are none unless r <= len.
      const uint32_t e = uint32_t(b) + uint32_t(i), ut = uint32_t(T);
      const uint32_t q = e / ut, r = e - q * ut;
      if (r <= uint32_t(len)) {
        const uint32_t s = uint32_t(a) + uint32_t(i);  // e(i-1) + 1
        const uint32_t first = s == 0 ? 0u : (s - 1u) / ut + 1u;
        const uint32_t last = min(q, uint32_t(P) - 1u);
        for (uint32_t c = first; c <= last; ++c) part[c] = make_int2(int(i), int(c * ut - uint32_t(i)));
      }
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    longest = max(longest, __shfl_xor_sync(0xffffffffu, longest, o));
    empty += __shfl_xor_sync(0xffffffffu, empty, o);
  }
  __shared__ int s_long[kThreads / 32], s_empty[kThreads / 32];
  const int w = threadIdx.x >> 5;
  if ((threadIdx.x & 31) == 0) {
    s_long[w] = longest;
    s_empty[w] = empty;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int k = 1; k < kThreads / 32; ++k) {
      longest = max(longest, s_long[k]);
      empty += s_empty[k];
    }
    atomicMax(stats, longest);
    atomicAdd(stats + 1, empty);
  }
}

// part[c] = (row, nonzero) where the merged sequence of nonzeros and row ends
// is cut at diagonal d = min(c * T, M + nnz): the row is the number of rows
// whose end position rowptr[r+1] + r lies before d.  With err, a caller's nnz
// that differs from rowptr[M] empties every range (part[c] = (0, 0)) and sets
// kErrInvalidCsr, so no kernel reads past the nonzeros that exist.
__global__ void __launch_bounds__(kThreads) merge_path_partition_kernel(const int32_t* __restrict__ rowptr,
                                                                        int32_t M, int64_t nnz, int64_t T,
                                                                        int32_t P, int2* __restrict__ part,
                                                                        int* __restrict__ err) {
  const int c = blockIdx.x * blockDim.x + threadIdx.x;
  if (c > P) return;
  if (err != nullptr && int64_t(__ldg(rowptr + M)) != nnz) {
    part[c] = make_int2(0, 0);
    if (c == 0) atomicOr(err, kErrInvalidCsr);
    return;
  }
  const int64_t d = min(int64_t(c) * T, int64_t(M) + nnz);
  int lo = 0, hi = M;
  while (lo < hi) {
    const int mid = lo + ((hi - lo) >> 1);
    if (int64_t(__ldg(rowptr + mid + 1)) + mid >= d) hi = mid; else lo = mid + 1;
  }
  part[c] = make_int2(lo, int(d - lo));
}

// flag |= 1: rowptr[0] != 0, rowptr[M] != nnz or a decreasing step; |= 2: colind out of range.
__global__ void __launch_bounds__(kThreads) validate_kernel(const int32_t* __restrict__ rowptr,
                                                            const int32_t* __restrict__ colind, int32_t M,
                                                            int32_t K, int64_t nnz, int* __restrict__ flag) {
  const int64_t stride = int64_t(gridDim.x) * blockDim.x;
  int bad = 0;
  for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i <= M; i += stride) {
    const int v = rowptr[i];
    if (i == 0 && v != 0) bad |= 1;
    if (i == M && int64_t(v) != nnz) bad |= 1;
    if (i < M && rowptr[i + 1] < v) bad |= 1;
  }
  for (int64_t p = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; p < nnz; p += stride) {
    const int c = colind[p];
    if (c < 0 || c >= K) bad |= 2;
  }
  if (bad) atomicOr(flag, bad);
}

// One warp per CTA range c.  If a row starts inside range c and its end item
// lies in a later range (carry slot 1 of c), add slot 1 of c and slot 0 of
// every following range up to the one holding the row's end, in range order,
// and write the C row.  The ranges are T items each, so the range holding the
// row's end item (position rowptr[row+1] + row) follows from rowptr alone and
// every carry load of the row can be in flight at once.  SR: the semiring
// whose (+) combines the pieces.
template <int SR>
__global__ void __launch_bounds__(kThreads) spmm_fixup_kernel(int32_t M, int32_t N,
                                                              const int32_t* __restrict__ rowptr,
                                                              const int2* __restrict__ part, int32_t P, int32_t T,
                                                              const float* __restrict__ carry,
                                                              float* __restrict__ C) {
  const int c = blockIdx.x * (kThreads / 32) + threadIdx.x / 32;
  const int lane = threadIdx.x & 31;
  if (c >= P) return;
  const int2 beg = __ldg(part + c);
  const int2 fin = __ldg(part + c + 1);
  const int row = fin.x;  // the row whose end item is the first one after range c
  if (row >= M) return;
  const int rs = __ldg(rowptr + row);
  if (rs < beg.y || rs >= fin.y) return;  // the row does not start inside range c
  const int last = int((int64_t(__ldg(rowptr + row + 1)) + row) / T);  // range holding the row's end item
  for (int n = lane; n < N; n += 32) {
    float s = __ldcg(carry + (size_t(c) * 2 + 1) * N + n);
    constexpr int kAhead = 8;  // slot loads in flight per lane
    for (int c0 = c + 1; c0 <= last; c0 += kAhead) {
      float v[kAhead];
#pragma unroll
      for (int k = 0; k < kAhead; ++k) v[k] = c0 + k <= last ? __ldcg(carry + (size_t(c0 + k) * 2) * N + n) : 0.f;
#pragma unroll
      for (int k = 0; k < kAhead; ++k)
        if (c0 + k <= last) s = sr_plus<SR>(s, v[k]);
    }
    st_stream1(C + size_t(row) * N + n, s);
  }
}

cudaError_t launch_fixup(const Launch& L, int sr) {
  constexpr int kWarps = kThreads / 32;
  const unsigned grid = unsigned((L.num_ctas + kWarps - 1) / kWarps);
  SPMM_DEBUG_RANGES(L.stream, L.err, {}, {{L.C, size_t(L.M) * L.N * 4}});
  switch (sr) {
#define SPMM_FIXUP_CASE(X) \
  case X: spmm_fixup_kernel<X><<<grid, kThreads, 0, L.stream>>>(L.M, L.N, L.rowptr, L.part, L.num_ctas, L.items_per_cta, L.carry, L.C); break;
    SPMM_FIXUP_CASE(0) SPMM_FIXUP_CASE(1) SPMM_FIXUP_CASE(2) SPMM_FIXUP_CASE(3) SPMM_FIXUP_CASE(4) SPMM_FIXUP_CASE(5)
#undef SPMM_FIXUP_CASE
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

cudaError_t launch_partition(const int32_t* rowptr, int32_t M, int64_t nnz, int32_t T, int32_t P, int2* part,
                             cudaStream_t stream, int* err) {
  const unsigned grid = unsigned((int64_t(P) + 1 + kThreads - 1) / kThreads);
  merge_path_partition_kernel<<<grid, kThreads, 0, stream>>>(rowptr, M, nnz, T, P, part, err);
  return cudaGetLastError();
}

}  // namespace spmm

using namespace spmm;

namespace {

// Plans (and so the one-call forms) allocate from a pool of the library's
// own on each device, with the release threshold raised so that freed blocks
// stay reserved for the next plan.  (The device's default pool returns its memory to the system at
// every synchronisation, and mapping it again costs about 0.1 ms per call.)
std::mutex g_pool_mutex;
cudaMemPool_t g_pool[kMaxDevices] = {};

cudaError_t library_pool(cudaMemPool_t* out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_pool_mutex);
  if (!g_pool[dev]) {
    cudaMemPoolProps props = {};
    props.allocType = cudaMemAllocationTypePinned;
    props.location.type = cudaMemLocationTypeDevice;
    props.location.id = dev;
    cudaMemPool_t pool = nullptr;
    if ((e = cudaMemPoolCreate(&pool, &props)) != cudaSuccess) return e;
    uint64_t keep = UINT64_MAX;
    if ((e = cudaMemPoolSetAttribute(pool, cudaMemPoolAttrReleaseThreshold, &keep)) != cudaSuccess) {
      cudaMemPoolDestroy(pool);
      return e;
    }
    g_pool[dev] = pool;
  }
  *out = g_pool[dev];
  return cudaSuccess;
}

// Stream-ordered allocation on `s` from the library's pool (cheap once the
// pool holds enough; no device-wide synchronisation).
cudaError_t dev_alloc(void** p, size_t bytes, cudaStream_t s) {
  cudaMemPool_t pool = nullptr;
  const cudaError_t e = library_pool(&pool);
  return e == cudaSuccess ? cudaMallocFromPoolAsync(p, bytes, pool, s) : e;
}
void dev_free(void* p, cudaStream_t s) {
  if (p) cudaFreeAsync(p, s);
}

// A pinned host buffer per host thread for the plan's one read-back of its
// statistics (an asynchronous copy into it needs no staging through a driver
// buffer, unlike one into pageable memory).  Allocated on the thread's first
// plan and kept for the life of the process.
int* pinned_stats_buffer() {
  thread_local int* buf = nullptr;
  if (!buf) {
    void* p = nullptr;
    if (cudaHostAlloc(&p, 16, cudaHostAllocPortable) == cudaSuccess) buf = static_cast<int*>(p);
  }
  return buf;
}

unsigned stats_grid(int32_t M) {
  const int64_t blocks = (int64_t(M) + kThreads - 1) / kThreads;
  return unsigned(std::max<int64_t>(1, std::min<int64_t>(blocks, 152 * 8)));
}

}  // namespace

// Plan construction shared by spmm_csr_plan(_ex) and the one-call forms.
// one_call: nnz is read from rowptr[M] along with the row statistics (the
// caller passes -1), the workspace comes from the one-call pool, and the
// merge-path partition is built only when the chosen kernel uses it.
spmm_status spmm_make_plan(const int32_t* rowptr, int32_t M, int64_t nnz, int32_t N, int32_t kernel,
                           int32_t items_per_cta, cudaStream_t stream, bool one_call, spmm_plan_t* plan_out) {
  if (!plan_out) return SPMM_ERR_INVALID_ARG;
  *plan_out = nullptr;
  if (M < 0 || N < 0 || (nnz < 0 && !one_call)) return SPMM_ERR_INVALID_ARG;
  if (M > SPMM_MAX_EXTENT || nnz > SPMM_MAX_EXTENT) return SPMM_ERR_UNSUPPORTED;
  if (M > 0 && !rowptr) return SPMM_ERR_INVALID_ARG;
  if (kernel < SPMM_KERNEL_AUTO || kernel > SPMM_KERNEL_WINDOW_TC) return SPMM_ERR_INVALID_ARG;
  if (items_per_cta != 0 && (items_per_cta < 256 || items_per_cta > kMaxItemsPerCta || items_per_cta % 256 != 0))
    return SPMM_ERR_INVALID_ARG;

  spmm_plan_s* plan = new (std::nothrow) spmm_plan_s();
  if (!plan) return SPMM_ERR_CUDA;
  plan->M = M;
  plan->nnz = std::max<int64_t>(nnz, 0);
  plan->N = N;
  plan->rowptr = rowptr;
  plan->kernel = kernel == SPMM_KERNEL_AUTO ? SPMM_KERNEL_ROW : kernel;
  if (cudaGetDevice(&plan->device) != cudaSuccess) {
    delete plan;
    return SPMM_ERR_CUDA;
  }
  if (M == 0 || N == 0) {  // nothing to compute; exec is a no-op
    *plan_out = plan;
    return SPMM_OK;
  }

  auto fail = [&](spmm_status st) {
    dev_free(plan->workspace, stream);
    dev_free(plan->small, stream);
    delete plan;
    return st;
  };

  // The plan form knows nnz up front: the workspace is allocated first and
  // one pass over rowptr computes the statistics and the merge-path
  // partition together (one launch, one synchronisation).  The one-call
  // forms learn nnz from that pass and build the partition afterwards, only
  // when the balanced kernel is chosen.
  const int T = items_per_cta ? items_per_cta : default_items_per_cta(N);
  auto carve = [&](int64_t P, size_t head) -> spmm_status {  // [head] + partition + carry rows for P ranges
    if (P > INT32_MAX - 1) return SPMM_ERR_UNSUPPORTED;
    plan->items_per_cta = T;
    plan->num_ctas = int32_t(P);
    const size_t part_bytes = (size_t(P) + 1) * sizeof(int2);
    const size_t part_padded = (part_bytes + 255) & ~size_t(255);
    const size_t carry_bytes = size_t(P) * 2 * size_t(N) * sizeof(float);
    plan->workspace_bytes += int64_t(head + part_padded + carry_bytes);
    if (dev_alloc(&plan->workspace, head + part_padded + carry_bytes, stream) != cudaSuccess) return SPMM_ERR_CUDA;
    char* w = static_cast<char*>(plan->workspace);
    plan->part = reinterpret_cast<int2*>(w + head);
    plan->carry = reinterpret_cast<float*>(w + head + part_padded);
    return SPMM_OK;
  };
  const int64_t P_known = one_call ? 0 : (int64_t(M) + nnz + T - 1) / T;
  // The error word and statistics (16 bytes): the head of the workspace in
  // the plan form (one allocation), an allocation of their own in the
  // one-call forms, whose workspace size is known only after the statistics.
  if (!one_call) {
    const spmm_status st = carve(P_known, 256);
    if (st != SPMM_OK) return fail(st);
    plan->err = static_cast<int*>(plan->workspace);
  } else {
    if (dev_alloc(&plan->small, 16, stream) != cudaSuccess) return fail(SPMM_ERR_CUDA);
    plan->workspace_bytes += 16;
    plan->err = static_cast<int*>(plan->small);
  }
  plan->stats = plan->err + 1;
  cudaError_t e = cudaMemsetAsync(plan->err, 0, 16, stream);
  if (e != cudaSuccess) return fail(SPMM_ERR_CUDA);
  plan_rows_kernel<<<stats_grid(M), kThreads, 0, stream>>>(rowptr, M, std::max<int64_t>(nnz, 0), T, int32_t(P_known),
                                                           plan->stats, plan->part);
  if ((e = cudaGetLastError()) != cudaSuccess) return fail(SPMM_ERR_CUDA);
  int host_stats[3] = {0, 0, 0};
  int* pinned = pinned_stats_buffer();
  if ((e = cudaMemcpyAsync(pinned ? pinned : host_stats, plan->stats, sizeof host_stats, cudaMemcpyDeviceToHost,
                           stream)) != cudaSuccess)
    return fail(SPMM_ERR_CUDA);
  if ((e = cudaStreamSynchronize(stream)) != cudaSuccess) return fail(SPMM_ERR_CUDA);
  if (pinned) std::copy(pinned, pinned + 3, host_stats);
  plan->max_row_nnz = host_stats[0];
  plan->empty_rows = host_stats[1];
  if (host_stats[2] < 0 || (nnz >= 0 && host_stats[2] != nnz)) return fail(SPMM_ERR_INVALID_CSR);
  if (host_stats[2] > SPMM_MAX_EXTENT) return fail(SPMM_ERR_UNSUPPORTED);  // one-call forms: nnz from rowptr[M]
  nnz = plan->nnz = host_stats[2];

  if (kernel == SPMM_KERNEL_AUTO) {
    // Short, even rows: one group per row keeps all lanes busy with no
    // partition or fixup.  Skewed rows (a row far longer than the mean): the
    // merge-path split bounds every CTA's work.
    const double mean = double(nnz) / double(M);
    plan->kernel = double(plan->max_row_nnz) <= 4.0 * mean + 32.0 ? SPMM_KERNEL_ROW : SPMM_KERNEL_BALANCED;
    // Rows wide enough for a warp per column tile: the window kernels (they
    // fall back to per-row gathers where the columns are scattered); the
    // tensor-core form where B is bf16 and N fits one MMA, else CUDA cores.
    if (plan->kernel == SPMM_KERNEL_ROW && N >= 128) plan->kernel = SPMM_KERNEL_WINDOW_TC;
    // Narrow B: a whole output row fits a lane; several lanes share a row.
    if (plan->kernel == SPMM_KERNEL_ROW && N <= 8) plan->kernel = SPMM_KERNEL_SMALLN;
  }
  if (plan->kernel == SPMM_KERNEL_SMALLN) {
    // r lanes per row so that each lane takes about 4 nonzeros of a mean row
    // (4 gathers in flight per lane), between 2 and 32.
    const double mean = M > 0 ? double(nnz) / double(M) : 0.0;
    int r = 2;
    while (r < 32 && 4.0 * r < mean) r <<= 1;
    plan->group_lanes = r;
  }

  // one-call forms: the merge-path partition and carry rows, only for the
  // balanced kernel (a one-call SpMM on another kernel needs neither)
  if (one_call && plan->kernel == SPMM_KERNEL_BALANCED) {
    const int64_t P = (int64_t(M) + nnz + T - 1) / T;
    const spmm_status st = carve(P, 0);
    if (st != SPMM_OK) return fail(st);
    plan_rows_kernel<<<stats_grid(M), kThreads, 0, stream>>>(rowptr, M, nnz, T, int32_t(P), plan->stats, plan->part);
    if ((e = cudaGetLastError()) != cudaSuccess) return fail(SPMM_ERR_CUDA);
  }
  *plan_out = plan;
  return SPMM_OK;
}

void spmm_free_plan(spmm_plan_t plan, cudaStream_t stream) {
  if (!plan) return;
  dev_free(plan->workspace, stream);
  dev_free(plan->small, stream);
  delete plan;
}

extern "C" {

spmm_status spmm_csr_plan_ex(const int32_t* rowptr, int32_t M, int64_t nnz, int32_t N, int32_t kernel,
                             int32_t items_per_cta, void* stream, spmm_plan_t* plan_out) {
  return spmm_make_plan(rowptr, M, nnz, N, kernel, items_per_cta, static_cast<cudaStream_t>(stream), false,
                        plan_out);
}

spmm_status spmm_csr_plan(const int32_t* rowptr, int32_t M, int64_t nnz, int32_t N, void* stream,
                          spmm_plan_t* plan_out) {
  return spmm_csr_plan_ex(rowptr, M, nnz, N, SPMM_KERNEL_AUTO, 0, stream, plan_out);
}

spmm_status spmm_plan_get_info(spmm_plan_t plan, spmm_plan_info* info) {
  if (!plan || !info) return SPMM_ERR_INVALID_ARG;
  info->kernel = plan->kernel;
  info->M = plan->M;
  info->nnz = plan->nnz;
  info->N = plan->N;
  info->max_row_nnz = plan->max_row_nnz;
  info->empty_rows = plan->empty_rows;
  info->items_per_cta = plan->items_per_cta;
  info->num_ctas = plan->num_ctas;
  info->workspace_bytes = plan->workspace_bytes;
  info->group_lanes = plan->group_lanes;
  info->column_tile = plan->column_tile;
  return SPMM_OK;
}

spmm_status spmm_plan_set_column_tile(spmm_plan_t plan, int32_t columns) {
  if (!plan) return SPMM_ERR_PLAN_MISMATCH;
  if (columns < 0) return SPMM_ERR_INVALID_ARG;
  plan->column_tile = columns;
  return SPMM_OK;
}

spmm_status spmm_plan_set_group_lanes(spmm_plan_t plan, int32_t lanes) {
  if (!plan) return SPMM_ERR_PLAN_MISMATCH;
  if (plan->kernel != SPMM_KERNEL_SMALLN) return SPMM_ERR_INVALID_ARG;
  if (lanes != 2 && lanes != 4 && lanes != 8 && lanes != 16 && lanes != 32) return SPMM_ERR_INVALID_ARG;
  plan->group_lanes = lanes;
  return SPMM_OK;
}

spmm_status spmm_plan_destroy(spmm_plan_t plan) {
  if (!plan) return SPMM_OK;
  cudaDeviceSynchronize();  // the plan may be in use on any stream
  spmm_free_plan(plan, nullptr);
  return SPMM_OK;
}

spmm_status spmm_plan_check_device(spmm_plan_t plan, void* stream) {
  if (!plan) return SPMM_ERR_INVALID_ARG;
  if (!plan->err) return SPMM_OK;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int word = 0;
  if (cudaMemcpyAsync(&word, plan->err, sizeof word, cudaMemcpyDeviceToHost, s) != cudaSuccess) return SPMM_ERR_CUDA;
  if (cudaMemsetAsync(plan->err, 0, sizeof word, s) != cudaSuccess) return SPMM_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return SPMM_ERR_CUDA;
  if (word & kErrBounds) return SPMM_ERR_OUT_OF_BOUNDS;
  return word ? SPMM_ERR_DEVICE_TIMEOUT : SPMM_OK;
}

spmm_status spmm_csr_validate(const int32_t* rowptr, const int32_t* colind, int32_t M, int32_t K, int64_t nnz,
                              void* stream) {
  if (M < 0 || K < 0 || nnz < 0) return SPMM_ERR_INVALID_ARG;
  if (M > SPMM_MAX_EXTENT || nnz > SPMM_MAX_EXTENT) return SPMM_ERR_UNSUPPORTED;
  if (!rowptr || (nnz > 0 && !colind)) return SPMM_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int* flag = nullptr;
  if (dev_alloc(reinterpret_cast<void**>(&flag), sizeof(int), s) != cudaSuccess) return SPMM_ERR_CUDA;
  int host = 0;
  cudaError_t e = cudaMemsetAsync(flag, 0, sizeof(int), s);
  if (e == cudaSuccess) {
    const int64_t work = std::max<int64_t>(int64_t(M) + 1, nnz);
    const unsigned grid = unsigned(std::max<int64_t>(1, std::min<int64_t>((work + kThreads - 1) / kThreads, 152 * 16)));
    validate_kernel<<<grid, kThreads, 0, s>>>(rowptr, colind, M, K, nnz, flag);
    e = cudaGetLastError();
  }
  if (e == cudaSuccess) e = cudaMemcpyAsync(&host, flag, sizeof(int), cudaMemcpyDeviceToHost, s);
  dev_free(flag, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return SPMM_ERR_CUDA;
  return host ? SPMM_ERR_INVALID_CSR : SPMM_OK;
}

spmm_status spmm_pool_release(void) {
  std::lock_guard<std::mutex> lock(g_pool_mutex);
  for (int d = 0; d < kMaxDevices; ++d)
    if (g_pool[d] && cudaMemPoolTrimTo(g_pool[d], 0) != cudaSuccess) return SPMM_ERR_CUDA;
  return SPMM_OK;
}

}  // extern "C"
