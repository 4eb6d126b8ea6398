// topk_slots.cu -- physical cache slots of selected logical positions (vLLM
// QSA page, _qsa_physical_slots_kernel): page << offset_bits | page offset,
// -1 for masked entries and the padding past the selection.
//
// One thread per output slot, one CTA row of threads per query row: the
// row's request comes from cu_seqlens_q (binary search, once per thread, the
// few words stay in L1), the indices are read and the slots written
// coalesced, the page table is gathered.  Memory-bound and small.
#include "internal.h"

namespace fp4idx {
namespace {

constexpr int kSlotThreads = 256;

__global__ void __launch_bounds__(kSlotThreads) topk_slots_kernel(const SlotParams p) {
  const int32_t t = blockIdx.y;
  const int32_t c = blockIdx.x * kSlotThreads + threadIdx.x;
  if (c >= p.ncols) return;
  int32_t slot = -1;
  if (c < p.k) {
    const int32_t s = __ldg(p.indices + static_cast<int64_t>(t) * p.k + c);
    int lo = 0, hi = p.num_seqs - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (__ldg(p.cu_seqlens_q + mid) <= t) lo = mid; else hi = mid - 1;
    }
    const int32_t k_len = __ldg(p.cu_seqlens_k + lo + 1) - __ldg(p.cu_seqlens_k + lo);
    if (s >= 0 && s < k_len) {
      const int64_t base = p.page_offsets ? static_cast<int64_t>(__ldg(p.page_offsets + lo))
                                          : static_cast<int64_t>(lo) * p.table_stride;
      const int32_t page = __ldg(p.block_table + base + (s >> p.page_shift));
      if (page >= 0 && page < p.num_pages)
        slot = (page << p.offset_bits) | (s & (p.page_size - 1));
    }
  }
  p.slots[static_cast<int64_t>(t) * p.ncols + c] = slot;
}

}  // namespace

cudaError_t launch_topk_slots(const SlotParams& p, int32_t rows, cudaStream_t stream) {
  if (rows <= 0) return cudaSuccess;
  const dim3 grid((p.ncols + kSlotThreads - 1) / kSlotThreads, rows);
  topk_slots_kernel<<<grid, kSlotThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace fp4idx
