// token_table.cu -- this ABI's request metadata (cu_seqlens_q, cu_seqlens_k,
// a per-page block table) from a per-token slot table: the req / req_table
// arguments of SGLang PR 42861's fp4_index_logits_paged, where req[t] is the
// request of query row t and req_table[b][s] the cache slot (page * page_size
// + offset) of logical position s of request b.
//
// Two launches, no workspace, chained by programmatic dependent launch:
//   1. one warp per (request, logical page): the page's slots must be one
//      cache page's offsets in order, followed only by empty entries (< 0);
//      its block-table entry is that page, -1 for a page with no slot, and
//      -1 with FP4IDX_ERR_TOKEN_TABLE otherwise.  An empty entry followed by
//      a filled one is reported too.  The page holding the request's last
//      filled position (found locally: the next page starts empty) writes
//      the request's key count, 1 + that position, to cu_seqlens_k[b + 1].
//   2. one CTA: the prefix sums of the key counts, and each request's first
//      row (binary search in req, which must be non-decreasing).
#include <cstring>

#include "internal.h"
#include "ptx.cuh"

namespace fp4idx {
namespace {

constexpr int kThreads = 256;
constexpr int kPagesPerCta = kThreads / 32;

__global__ void __launch_bounds__(kThreads) token_pages_kernel(const TokenTableParams p) {
  pdl_wait();  // the table may come from the kernel before this one
  pdl_launch_dependents();
  const int b = blockIdx.x;
  const int lane = threadIdx.x & 31;
  const int j = blockIdx.y * kPagesPerCta + static_cast<int>(threadIdx.x >> 5);
  if (j >= p.table_pages) return;
  const int32_t* row = p.req_table + static_cast<int64_t>(b) * p.req_stride;
  const int64_t s0 = static_cast<int64_t>(j) * p.page_size;
  const int per = p.page_size / 32;  // 2 or 4 entries per lane
  int32_t v[4];
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const int64_t s = s0 + u * 32 + lane;  // coalesced: one 128-byte line per u
    v[u] = (u < per && s < p.req_stride) ? __ldg(row + s) : -1;  // past the table: empty
  }
  const int32_t first = __shfl_sync(0xffffffffu, v[0], 0);
  int last_filled = -1, first_empty = p.page_size;
  bool ordered = true;
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    if (u >= per) break;
    const int i = u * 32 + lane;
    if (v[u] >= 0) {
      last_filled = max(last_filled, i);
      ordered &= v[u] == first + i;
    } else {
      first_empty = min(first_empty, i);
    }
  }
  last_filled = __reduce_max_sync(0xffffffffu, last_filled);
  first_empty = __reduce_min_sync(0xffffffffu, first_empty);
  ordered = __all_sync(0xffffffffu, ordered);
  if (lane != 0) return;
  const int64_t next_s = s0 + p.page_size;
  const int32_t next_first = next_s < p.req_stride ? __ldg(row + next_s) : -1;
  const bool any = last_filled >= 0;
  const bool good = any && ordered && last_filled < first_empty && first % p.page_size == 0 &&
                    first / p.page_size < p.num_pages;
  p.block_table[static_cast<int64_t>(b) * p.table_pages + j] = good ? first / p.page_size : -1;
  const bool hole = first_empty < p.page_size && next_first >= 0;  // an empty entry before a filled one
  if ((any && !good) || hole) atomicOr(p.err, kErrTokenTable);
  if ((any || j == 0) && next_first < 0) p.cu_seqlens_k[b + 1] = static_cast<int32_t>(s0 + last_filled + 1);
}

// One CTA: prefix sums of the key counts; the first row of every request.
__global__ void __launch_bounds__(kThreads) token_offsets_kernel(const TokenTableParams p) {
  pdl_wait();  // the key counts come from token_pages_kernel
  pdl_launch_dependents();
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

template <class K>
cudaError_t launch_pdl(K kern, dim3 grid, cudaStream_t stream, const TokenTableParams& p) {
  cudaLaunchConfig_t cfg;
  std::memset(&cfg, 0, sizeof(cfg));
  cfg.gridDim = grid;
  cfg.blockDim = dim3(kThreads);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, p);
}

}  // namespace

cudaError_t launch_token_table(const TokenTableParams& p, cudaStream_t stream) {
  const dim3 grid(static_cast<unsigned>(p.num_reqs), static_cast<unsigned>((p.table_pages + kPagesPerCta - 1) / kPagesPerCta));
  cudaError_t e = launch_pdl(token_pages_kernel, grid, stream, p);
  if (e != cudaSuccess) return e;
  return launch_pdl(token_offsets_kernel, dim3(1), stream, p);
}

}  // namespace fp4idx
