// token_table.cu -- this ABI's request metadata (cu_seqlens_q, cu_seqlens_k,
// a per-page block table) from a per-token slot table: the req / req_table
// arguments of SGLang PR 42861's fp4_index_logits_paged, where req[t] is the
// request of query row t and req_table[b][s] the cache slot (page * page_size
// + offset) of logical position s of request b.
//
// Three launches, no workspace (cu_seqlens_k carries the per-request key
// counts between the first two):
//   1. per request: its key count = 1 + the last position with a slot >= 0;
//   2. one CTA: the prefix sums of the key counts, and each request's first
//      row (binary search in req, which must be non-decreasing);
//   3. per (request, logical page): the page's slots below the key count
//      must be one cache page's offsets in order; then the block-table entry
//      is that page, else -1 (FP4IDX_ERR_TOKEN_TABLE).
#include "internal.h"
#include "ptx.cuh"

namespace fp4idx {
namespace {

constexpr int kThreads = 256;

// cu_seqlens_k[b + 1] = key count of request b (the prefix sum comes next).
__global__ void __launch_bounds__(kThreads) token_counts_kernel(const TokenTableParams p) {
  const int b = blockIdx.x;
  const int32_t* row = p.req_table + static_cast<int64_t>(b) * p.req_stride;
  int32_t last = -1;
  for (int64_t s = threadIdx.x; s < p.req_stride; s += kThreads)
    if (__ldg(row + s) >= 0) last = static_cast<int32_t>(s);
  last = __reduce_max_sync(0xffffffffu, last);
  __shared__ int32_t wmax[kThreads / 32];
  if ((threadIdx.x & 31) == 0) wmax[threadIdx.x >> 5] = last;
  __syncthreads();
  if (threadIdx.x == 0) {
    int32_t m = -1;
    for (int w = 0; w < kThreads / 32; ++w) m = max(m, wmax[w]);
    p.cu_seqlens_k[b + 1] = m + 1;
  }
}

// One CTA: prefix sums of the key counts; the first row of every request.
__global__ void __launch_bounds__(kThreads) token_offsets_kernel(const TokenTableParams p) {
  __shared__ int32_t carry;
  if (threadIdx.x == 0) {
    carry = 0;
    p.cu_seqlens_k[0] = 0;
  }
  __syncthreads();
  for (int base = 0; base < p.num_reqs; base += kThreads) {
    const int b = base + static_cast<int>(threadIdx.x);
    const int32_t v = b < p.num_reqs ? p.cu_seqlens_k[b + 1] : 0;
    // block-wide inclusive scan of v
    int32_t incl = v;
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int32_t y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    __shared__ int32_t wsum[kThreads / 32];
    if (lane == 31) wsum[wid] = incl;
    __syncthreads();
    int32_t before = 0, all = 0;
    for (int w = 0; w < kThreads / 32; ++w) {
      before += w < wid ? wsum[w] : 0;
      all += wsum[w];
    }
    if (b < p.num_reqs) p.cu_seqlens_k[b + 1] = carry + before + incl;
    __syncthreads();
    if (threadIdx.x == 0) carry += all;
    __syncthreads();
  }
  // first row of request b: the number of rows whose request is below b
  for (int b = threadIdx.x; b <= p.num_reqs; b += kThreads) {
    int lo = 0, hi = p.num_rows;
    while (lo < hi) {
      const int mid = (lo + hi) >> 1;
      if (__ldg(p.req + mid) < b) lo = mid + 1; else hi = mid;
    }
    p.cu_seqlens_q[b] = b == p.num_reqs ? p.num_rows : lo;
  }
  // the rows' requests must be valid and non-decreasing
  for (int t = threadIdx.x; t < p.num_rows; t += kThreads) {
    const int32_t r = __ldg(p.req + t);
    if (r < 0 || r >= p.num_reqs || (t + 1 < p.num_rows && __ldg(p.req + t + 1) < r)) atomicOr(p.err, kErrTokenTable);
  }
}

// Block-table entry of logical page blockIdx.x of request blockIdx.y.
__global__ void __launch_bounds__(128) token_pages_kernel(const TokenTableParams p) {
  const int j = blockIdx.x, b = blockIdx.y;
  const int32_t klen = p.cu_seqlens_k[b + 1] - p.cu_seqlens_k[b];
  const int64_t s0 = static_cast<int64_t>(j) * p.page_size;
  const int32_t* row = p.req_table + static_cast<int64_t>(b) * p.req_stride;
  const int32_t first = s0 < klen ? __ldg(row + s0) : -1;
  bool good = first >= 0 && first % p.page_size == 0 && first / p.page_size < p.num_pages;
  for (int i = threadIdx.x; i < p.page_size; i += 128) {
    const int64_t s = s0 + i;
    if (s < klen && __ldg(row + s) != first + i) good = false;
  }
  good = __syncthreads_and(good);
  if (threadIdx.x == 0) {
    const bool any = s0 < klen;
    p.block_table[static_cast<int64_t>(b) * p.table_pages + j] = any && good ? first / p.page_size : -1;
    if (any && !good) atomicOr(p.err, kErrTokenTable);
  }
}

}  // namespace

cudaError_t launch_token_table(const TokenTableParams& p, cudaStream_t stream) {
  token_counts_kernel<<<p.num_reqs, kThreads, 0, stream>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  token_offsets_kernel<<<1, kThreads, 0, stream>>>(p);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  token_pages_kernel<<<dim3(p.table_pages, p.num_reqs), 128, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace fp4idx
