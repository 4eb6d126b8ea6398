// block_topk.cu -- top-k blocks of every (head, row) column of a block-score
// tensor [Hq][Ktiles][T] (M3-indexer README, "输出 shape 和类型": a caller that
// needs a top-k of the block scores takes it along Ktiles).
//
// One thread per (h, t) column.  The column's scores are streamed in block
// order (for a fixed block, the threads of a warp read 32 consecutive t: one
// coalesced 128-byte line) and kept as a list of at most k (score, block)
// keys in registers, ordered by (score desc, block asc); a candidate is
// bubbled through the list only when it beats the current k-th entry.
// HBM-bound: 4 bytes read per score, 8 (+4) bytes written per selected block.
#include <math.h>
#include <stdint.h>

#include "internal.h"

namespace fp4idx {
namespace {

constexpr int kTopkThreads = 256;

template <int KM>
__global__ void __launch_bounds__(kTopkThreads, 2) block_topk_kernel(const float* __restrict__ scores, int32_t H,
                                                                  int32_t Kt, int32_t T, int32_t k,
                                                                  int32_t* __restrict__ indices,
                                                                  float* __restrict__ values,
                                                                  int32_t* __restrict__ valid_count) {
  const int64_t col = static_cast<int64_t>(blockIdx.x) * kTopkThreads + threadIdx.x;
  if (col >= static_cast<int64_t>(H) * T) return;
  const int64_t h = col / T, t = col - h * T;
  const float* src = scores + h * Kt * T + t;
  // Each candidate is one 64-bit key: the order-preserving bits of its score
  // over ~block, so (score desc, block asc) is plain key order.  The list is
  // the last k of KM slots in descending key order (0 = empty); the first
  // KM - k slots hold a sentinel no key exceeds, so the k-th entry is always
  // slot KM - 1.
  uint64_t lk[KM];
#pragma unroll
  for (int i = 0; i < KM; ++i) lk[i] = i < KM - k ? ~0ull : 0ull;
  int32_t n = 0;
  // the column is read eight blocks at a time, all eight loads in flight
  constexpr int kBatch = 8;
  for (int32_t b0 = 0; b0 < Kt; b0 += kBatch) {
    float vb[kBatch];
#pragma unroll
    for (int j = 0; j < kBatch; ++j)
      vb[j] = b0 + j < Kt ? __ldg(src + static_cast<int64_t>(b0 + j) * T) : -INFINITY;
#pragma unroll
    for (int j = 0; j < kBatch; ++j) {
      const float v = vb[j];
      if (!(v > -INFINITY)) continue;  // -inf (no visible key) and NaN are not candidates
      ++n;
      const uint32_t u = __float_as_uint(v + 0.0f);
      uint64_t cand = (static_cast<uint64_t>((u & 0x80000000u) ? ~u : (u | 0x80000000u)) << 32) |
                      static_cast<uint32_t>(~static_cast<uint32_t>(b0 + j));
      if (cand <= lk[KM - 1]) continue;  // does not beat the k-th entry
      // bubble down: each slot keeps the larger key and passes on the smaller
#pragma unroll
      for (int i = 0; i < KM; ++i) {
        const uint64_t t = lk[i];
        const bool move = cand > t;
        lk[i] = move ? cand : t;
        cand = move ? t : cand;
      }
    }
  }
  int32_t* oi = indices + col * k;
  float* ov = values ? values + col * k : nullptr;
#pragma unroll
  for (int i = 0; i < KM; ++i) {
    if (i >= KM - k) {
      const uint64_t key = lk[i];
      oi[i - (KM - k)] = key ? static_cast<int32_t>(~static_cast<uint32_t>(key)) : -1;
      if (ov) {
        const uint32_t o = static_cast<uint32_t>(key >> 32);
        ov[i - (KM - k)] = key ? __uint_as_float((o & 0x80000000u) ? (o & 0x7FFFFFFFu) : ~o) : -INFINITY;
      }
    }
  }
  if (valid_count) valid_count[col] = n < k ? n : k;
}

template <int KM>
cudaError_t launch_km(const float* scores, int32_t H, int32_t Kt, int32_t T, int32_t k, int32_t* indices,
                      float* values, int32_t* valid_count, cudaStream_t stream) {
  const int64_t cols = static_cast<int64_t>(H) * T;
  const unsigned grid = static_cast<unsigned>((cols + kTopkThreads - 1) / kTopkThreads);
  block_topk_kernel<KM><<<grid, kTopkThreads, 0, stream>>>(scores, H, Kt, T, k, indices, values, valid_count);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_block_topk(const float* scores, int32_t H, int32_t Kt, int32_t T, int32_t k, int32_t* indices,
                              float* values, int32_t* valid_count, cudaStream_t stream) {
  if (k <= 8) return launch_km<8>(scores, H, Kt, T, k, indices, values, valid_count, stream);
  if (k <= 16) return launch_km<16>(scores, H, Kt, T, k, indices, values, valid_count, stream);
  return launch_km<32>(scores, H, Kt, T, k, indices, values, valid_count, stream);
}

}  // namespace fp4idx
