// block_topk.cu -- top-k blocks of every (head, row) column of a block-score
// tensor [Hq][Ktiles][T] (M3-indexer README, "输出 shape 和类型": a caller that
// needs a top-k of the block scores takes it along Ktiles).
//
// Order (score desc, block asc); -inf (no visible key) and NaN are not
// candidates.  Each candidate is one 64-bit key: the order-preserving bits of
// its score over ~block, so the order is plain key order and every key of a
// column is distinct.
//
// k <= 32: one thread per column with the column's KM best keys so far in
// registers (KM = 8, 16 or 32 >= k), in descending order.  Each warp owns
// groups of 32 consecutive rows of one head and streams their scores through
// shared memory in chunks of 32 blocks, double buffered with cp.async
// (16-byte copies when T is a multiple of 4 and the scores are 16-byte
// aligned), so the reads are coalesced lines kept in flight while the
// previous chunk is selected.  The scores are taken KM at a time: the batch
// is sorted by a bitonic network, and the best KM of list and batch are the
// element-wise maxima of the list and the reversed batch (a bitonic
// sequence) put in order by a bitonic merge -- the same instructions for
// every thread, so no thread waits on another's data-dependent inserts.
// 32 < k <= 128: one warp per column.  Each lane holds Ktiles / 32 keys and
// counts, for each of them, the keys of the column that are larger (shuffled
// from every lane): that count is the key's place in the order, so a
// candidate whose count is below k is written straight to its output slot.
#include <math.h>
#include <stdint.h>

#include "internal.h"
#include "ptx.cuh"

namespace fp4idx {
namespace {

constexpr int kWarpsPerCta = 8;
constexpr int kChunk = 32;  // blocks per staged chunk
constexpr uint32_t kStageBytes = kChunk * 32 * 4;  // one chunk of a 32-row group
constexpr uint32_t kListSmem = kWarpsPerCta * 2 * kStageBytes;

__device__ __forceinline__ uint64_t block_key(float v, int32_t b) {
  const uint32_t u = __float_as_uint(v + 0.0f);  // -0 folded into +0
  return (static_cast<uint64_t>((u & 0x80000000u) ? ~u : (u | 0x80000000u)) << 32) |
         static_cast<uint32_t>(~static_cast<uint32_t>(b));
}
__device__ __forceinline__ float key_value(uint64_t key) {
  const uint32_t o = static_cast<uint32_t>(key >> 32);
  return __uint_as_float((o & 0x80000000u) ? (o & 0x7FFFFFFFu) : ~o);
}

// Compare-exchange keeping a >= b.
__device__ __forceinline__ void cx_desc(uint64_t& a, uint64_t& b) {
  const uint64_t x = a, y = b;
  const bool sw = x < y;
  a = sw ? y : x;
  b = sw ? x : y;
}
// A bitonic sequence of N keys into descending order.
template <int N>
__device__ __forceinline__ void bitonic_merge_desc(uint64_t (&v)[N]) {
#pragma unroll
  for (int stride = N / 2; stride >= 1; stride /= 2)
#pragma unroll
    for (int i = 0; i < N; ++i)
      if ((i & stride) == 0) cx_desc(v[i], v[i + stride]);
}
// N keys (a power of two) into descending order.
template <int N>
__device__ __forceinline__ void bitonic_sort_desc(uint64_t (&v)[N]) {
#pragma unroll
  for (int size = 2; size <= N; size *= 2)
#pragma unroll
    for (int stride = size / 2; stride >= 1; stride /= 2)
#pragma unroll
      for (int i = 0; i < N; ++i)
        if ((i & stride) == 0) {
          // blocks of `size` alternate direction; the last stage is all descending
          if ((i & size) == 0 || size == N) cx_desc(v[i], v[i + stride]);
          else cx_desc(v[i + stride], v[i]);
        }
}

template <int KM>
__global__ void __launch_bounds__(kWarpsPerCta * 32) block_topk_list_kernel(
    const float* __restrict__ scores, int32_t H, int32_t Kt, int32_t T, int32_t k, int32_t* __restrict__ indices,
    float* __restrict__ values, int32_t* __restrict__ valid_count) {
  extern __shared__ __align__(16) uint8_t smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float* stage0 = reinterpret_cast<float*>(smem + warp * 2 * kStageBytes);
  const int64_t row_groups = (T + 31) / 32;
  const int64_t groups = static_cast<int64_t>(H) * row_groups;
  const int chunks = (Kt + kChunk - 1) / kChunk;
  const bool vec4 = (T & 3) == 0 && (reinterpret_cast<uintptr_t>(scores) & 15) == 0;
  const int64_t gstride = static_cast<int64_t>(gridDim.x) * kWarpsPerCta;
  const int64_t g0 = static_cast<int64_t>(blockIdx.x) * kWarpsPerCta + warp;
  // this warp's work: chunk c of group g, for g = g0, g0 + gstride, ...
  const int64_t items = g0 < groups ? ((groups - 1 - g0) / gstride + 1) * chunks : 0;

  auto load = [&](int64_t item, int buf) {
    const int64_t g = g0 + (item / chunks) * gstride;
    const int c = static_cast<int>(item % chunks);
    const int64_t h = g / row_groups;
    const int32_t t0 = static_cast<int32_t>((g - h * row_groups) * 32);
    const int kb0 = c * kChunk;
    const int nb = min(kChunk, Kt - kb0);
    const float* src = scores + (h * Kt + kb0) * static_cast<int64_t>(T) + t0;
    const uint32_t dst = smem_u32(stage0) + buf * kStageBytes;
    if (vec4) {  // 8 lanes per block row, four rows per warp copy
      for (int e = lane; e < nb * 8; e += 32) {
        const int kb = e >> 3, q = e & 7;
        if (t0 + 4 * q < T) cp_async_16(dst + (kb * 32 + 4 * q) * 4, src + static_cast<int64_t>(kb) * T + 4 * q);
      }
    } else {
      for (int e = lane; e < nb * 32; e += 32) {
        const int kb = e >> 5, q = e & 31;
        if (t0 + q < T) cp_async_4(dst + (kb * 32 + q) * 4, src + static_cast<int64_t>(kb) * T + q);
      }
    }
    cp_async_commit();
  };

  uint64_t lk[KM];  // the column's best KM keys so far, descending (0 = none)
  int32_t n = 0;
  if (items > 0) load(0, 0);
  for (int64_t item = 0; item < items; ++item) {
    const int buf = static_cast<int>(item & 1);
    if (item + 1 < items) {
      load(item + 1, buf ^ 1);
      cp_async_wait_group<1>();  // this item's copies landed
    } else {
      cp_async_wait_group<0>();
    }
    __syncwarp();  // every lane's copies visible to every lane
    const int64_t g = g0 + (item / chunks) * gstride;
    const int c = static_cast<int>(item % chunks);
    const int64_t h = g / row_groups;
    const int32_t t = static_cast<int32_t>((g - h * row_groups) * 32) + lane;
    if (c == 0) {
#pragma unroll
      for (int i = 0; i < KM; ++i) lk[i] = 0ull;
      n = 0;
    }
    const int kb0 = c * kChunk;
    const int nb = min(kChunk, Kt - kb0);
    const float* col = stage0 + buf * (kStageBytes / 4) + lane;
    if (t < T) {
      for (int b0 = 0; b0 < nb; b0 += KM) {
        uint64_t bk[KM];  // the batch's keys; -inf, NaN and padding are 0
#pragma unroll
        for (int i = 0; i < KM; ++i) {
          const int kb = b0 + i;
          const float v = kb < nb ? col[kb * 32] : -INFINITY;
          const bool cand = v > -INFINITY;
          n += cand ? 1 : 0;
          bk[i] = cand ? block_key(v, kb0 + kb) : 0ull;
        }
        bitonic_sort_desc<KM>(bk);
        // best KM of both: max(list[i], batch[KM-1-i]) is bitonic
#pragma unroll
        for (int i = 0; i < KM; ++i) lk[i] = bk[KM - 1 - i] > lk[i] ? bk[KM - 1 - i] : lk[i];
        bitonic_merge_desc<KM>(lk);
      }
      if (c == chunks - 1) {
        const int64_t colid = h * T + t;
        int32_t* oi = indices + colid * k;
        float* ov = values ? values + colid * k : nullptr;
#pragma unroll
        for (int i = 0; i < KM; ++i) {
          if (i < k) {
            const uint64_t key = lk[i];
            oi[i] = key ? static_cast<int32_t>(~static_cast<uint32_t>(key)) : -1;
            if (ov) ov[i] = key ? key_value(key) : -INFINITY;
          }
        }
        if (valid_count) valid_count[colid] = n < k ? n : k;
      }
    }
    __syncwarp();  // the buffer is read before the next load reuses it
  }
}

// One warp per column; Kt <= 32 * kMaxPerLane.
constexpr int kMaxPerLane = 32;

template <int E>
__global__ void __launch_bounds__(256) block_topk_rank_kernel(const float* __restrict__ scores, int32_t H, int32_t Kt,
                                                             int32_t T, int32_t k, int32_t* __restrict__ indices,
                                                             float* __restrict__ values,
                                                             int32_t* __restrict__ valid_count) {
  const int lane = threadIdx.x & 31;
  const int64_t colid = static_cast<int64_t>(blockIdx.x) * 8 + (threadIdx.x >> 5);
  if (colid >= static_cast<int64_t>(H) * T) return;  // warp-uniform
  const int64_t h = colid / T, t = colid - h * T;
  const float* src = scores + h * Kt * static_cast<int64_t>(T) + t;
  uint64_t key[E];  // block lane + 32 e; 0 when not a candidate (below every candidate)
  int cnt = 0;
#pragma unroll
  for (int e = 0; e < E; ++e) {
    const int b = lane + 32 * e;
    const float v = b < Kt ? __ldg(src + static_cast<int64_t>(b) * T) : -INFINITY;
    const bool cand = v > -INFINITY;  // false for -inf and NaN
    key[e] = cand ? block_key(v, b) : 0ull;
    cnt += cand ? 1 : 0;
  }
  const int n = __reduce_add_sync(0xffffffffu, cnt);
  // place of each key: the number of larger keys of the column
  int rank[E];
#pragma unroll
  for (int e = 0; e < E; ++e) rank[e] = 0;
#pragma unroll
  for (int e2 = 0; e2 < E; ++e2) {
    for (int src_lane = 0; src_lane < 32; ++src_lane) {
      const uint64_t y = __shfl_sync(0xffffffffu, key[e2], src_lane);
#pragma unroll
      for (int e = 0; e < E; ++e) rank[e] += y > key[e] ? 1 : 0;
    }
  }
  int32_t* oi = indices + colid * k;
  float* ov = values ? values + colid * k : nullptr;
#pragma unroll
  for (int e = 0; e < E; ++e) {
    if (key[e] != 0ull && rank[e] < k) {
      oi[rank[e]] = static_cast<int32_t>(~static_cast<uint32_t>(key[e]));
      if (ov) ov[rank[e]] = key_value(key[e]);
    }
  }
  const int m = n < k ? n : k;
  for (int i = m + lane; i < k; i += 32) {
    oi[i] = -1;
    if (ov) ov[i] = -INFINITY;
  }
  if (valid_count && lane == 0) valid_count[colid] = m;
}

template <int KM>
cudaError_t launch_list(const float* scores, int32_t H, int32_t Kt, int32_t T, int32_t k, int32_t* indices,
                        float* values, int32_t* valid_count, int sms, cudaStream_t stream) {
  auto kern = block_topk_list_kernel<KM>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(kListSmem));
  if (e != cudaSuccess) return e;
  const int64_t groups = static_cast<int64_t>(H) * ((T + 31) / 32);
  const int64_t want = (groups + kWarpsPerCta - 1) / kWarpsPerCta;
  const unsigned grid = static_cast<unsigned>(want < sms ? want : sms);
  kern<<<grid, kWarpsPerCta * 32, kListSmem, stream>>>(scores, H, Kt, T, k, indices, values, valid_count);
  return cudaGetLastError();
}

template <int E>
cudaError_t launch_rank(const float* scores, int32_t H, int32_t Kt, int32_t T, int32_t k, int32_t* indices,
                        float* values, int32_t* valid_count, cudaStream_t stream) {
  const int64_t cols = static_cast<int64_t>(H) * T;
  const unsigned grid = static_cast<unsigned>((cols + 7) / 8);
  block_topk_rank_kernel<E><<<grid, 256, 0, stream>>>(scores, H, Kt, T, k, indices, values, valid_count);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_block_topk(const float* scores, int32_t H, int32_t Kt, int32_t T, int32_t k, int32_t* indices,
                              float* values, int32_t* valid_count, int sms, cudaStream_t stream) {
  if (k <= 8) return launch_list<8>(scores, H, Kt, T, k, indices, values, valid_count, sms, stream);
  if (k <= 16) return launch_list<16>(scores, H, Kt, T, k, indices, values, valid_count, sms, stream);
  if (k <= 32) return launch_list<32>(scores, H, Kt, T, k, indices, values, valid_count, sms, stream);
  if (Kt <= 64) return launch_rank<2>(scores, H, Kt, T, k, indices, values, valid_count, stream);
  if (Kt <= 256) return launch_rank<8>(scores, H, Kt, T, k, indices, values, valid_count, stream);
  return launch_rank<kMaxPerLane>(scores, H, Kt, T, k, indices, values, valid_count, stream);
}

}  // namespace fp4idx
