// topk_smem.cuh -- exact k-largest selection over 64-bit keys held in shared
// memory, cooperatively by a fixed group of threads.
//
// Keys are built by topk_key(): larger key = larger logit, then lower
// position; all keys of one row are distinct.  A selection returns the
// threshold T such that exactly k of the keys are >= T.  It works by a
// coarse bucket histogram over the top 11 key bits (kept up to date while
// candidates are appended) followed by 8-bit radix passes inside the
// bucket that holds the k-th key.
#pragma once

#include <stdint.h>

#include "ptx.cuh"

namespace fp4idx {

constexpr int kHistBins = 2048;
constexpr int kHistShift = 53;  // bucket = key >> 53 (sign, exponent, 2 mantissa bits)

// Group of kThreads threads (a multiple of 32, <= 1024) that synchronise
// with a named barrier: barrier 0 is __syncthreads, kBarrierId < 0 takes the
// barrier id from `bar` at run time; a group of one warp uses __syncwarp.
template <int kThreads, int kBarrierId>
struct Group {
  static_assert(kThreads % 32 == 0, "whole warps");
  static constexpr int kSize = kThreads;
  int tid;  // 0 .. kThreads-1
  int bar = kBarrierId;
  __device__ __forceinline__ void sync() const {
    if constexpr (kThreads == 32)
      __syncwarp();  // a one-warp group
    else if constexpr (kBarrierId == 0)
      __syncthreads();
    else if constexpr (kBarrierId > 0)
      asm volatile("bar.sync %0, %1;" ::"n"(kBarrierId), "n"(kThreads) : "memory");
    else
      asm volatile("bar.sync %0, %1;" ::"r"(bar), "n"(kThreads) : "memory");
  }
};

// Scratch for selections: warp partial sums and a few broadcast words.
struct SelectScratch {
  uint32_t warp_sum[32];
  uint32_t digit_hist[256];
  uint32_t bcast[4];
};

// Exclusive suffix sum over the group: returns sum of v over threads with a
// larger tid.  Also returns the group total in *total.
template <int kThreads, int kBarrierId>
__device__ __forceinline__ uint32_t group_excl_suffix(const Group<kThreads, kBarrierId>& g, uint32_t v,
                                                      SelectScratch* sc, uint32_t* total) {
  const int lane = g.tid & 31, wid = g.tid >> 5;
  constexpr int kWarps = kThreads / 32;
  uint32_t incl = v;  // inclusive suffix within the warp
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    uint32_t y = __shfl_down_sync(0xffffffffu, incl, o);
    if (lane + o < 32) incl += y;
  }
  if (lane == 0) sc->warp_sum[wid] = incl;
  g.sync();
  uint32_t after = 0, all = 0;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) {
    uint32_t s = sc->warp_sum[w];
    all += s;
    if (w > wid) after += s;
  }
  g.sync();
  *total = all;
  return after + incl - v;
}

// Exclusive prefix sum over all kThreads threads of the CTA (__syncthreads):
// returns the sum of v over threads with a smaller threadIdx.x and the CTA
// total in *total.  ws holds kThreads / 32 words.
template <int kThreads>
__device__ __forceinline__ uint32_t cta_excl_prefix(uint32_t v, uint32_t* ws, uint32_t* total) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  uint32_t incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) ws[wid] = incl;
  __syncthreads();
  uint32_t before = 0, all = 0;
#pragma unroll
  for (int w = 0; w < kThreads / 32; ++w) {
    const uint32_t x = ws[w];
    before += w < wid ? x : 0u;
    all += x;
  }
  __syncthreads();
  *total = all;
  return before + incl - v;
}

// Bucket histogram with 16-bit counters, two per 32-bit word (a row's
// candidate buffer never holds 65,536 keys).
struct Hist16 {
  uint32_t* w;  // kHistBins / 2 words
  __device__ __forceinline__ uint32_t operator()(int b) const { return (w[b >> 1] >> ((b & 1) * 16)) & 0xFFFFu; }
  __device__ __forceinline__ void add(int b) const { atomicAdd(&w[b >> 1], 1u << ((b & 1) * 16)); }
  // Single thread: overwrite one counter.
  __device__ __forceinline__ void set(int b, uint32_t v) const {
    const int sh = (b & 1) * 16;
    w[b >> 1] = (w[b >> 1] & ~(0xFFFFu << sh)) | (v << sh);
  }
};

// Bucket of the k-th largest key given a bucket histogram hist(b) (k >= 1
// and total >= k).  Returns the bucket and writes the count of keys in
// higher buckets to *above.  Every thread of the group gets the same answer.
template <int kThreads, int kBarrierId, class HistGet>
__device__ uint32_t find_kth_bucket(const Group<kThreads, kBarrierId>& g, const HistGet& hist,
                                    uint32_t k, SelectScratch* sc, uint32_t* above) {
  constexpr int kPer = kHistBins / kThreads;
  static_assert(kHistBins % kThreads == 0, "bins per thread");
  const int b0 = g.tid * kPer;
  uint32_t s = 0;
#pragma unroll 4
  for (int i = 0; i < kPer; ++i) s += hist(b0 + i);
  if (g.tid == 0) {  // answer when fewer than k keys exist: keep everything
    sc->bcast[0] = 0;
    sc->bcast[1] = 0;
  }
  uint32_t total;
  uint32_t after = group_excl_suffix(g, s, sc, &total);
  if (after < k && after + s >= k) {
    uint32_t acc = after;
    for (int i = kPer - 1; i >= 0; --i) {
      uint32_t h = hist(b0 + i);
      if (acc + h >= k) {
        sc->bcast[0] = static_cast<uint32_t>(b0 + i);
        sc->bcast[1] = acc;
        break;
      }
      acc += h;
    }
  }
  g.sync();
  uint32_t bucket = sc->bcast[0];
  *above = sc->bcast[1];
  g.sync();
  return bucket;
}

// Exact threshold inside one bucket: among keys with (key >> 53) == bucket,
// find T such that exactly `rank` of them are >= T (1 <= rank <= their
// count).  `for_each` visits every key of the source once per call.
template <int kThreads, int kBarrierId, class ForEach>
__device__ uint64_t select_in_bucket(const Group<kThreads, kBarrierId>& g, uint32_t bucket,
                                     uint32_t rank, SelectScratch* sc, ForEach for_each) {
  uint64_t prefix = bucket;
  int sh = kHistShift;
  while (sh > 0) {
    const int w = sh >= 8 ? 8 : sh;
    const int lo = sh - w;
    for (int i = g.tid; i < 256; i += kThreads) sc->digit_hist[i] = 0;
    g.sync();
    const uint64_t pref = prefix;
    for_each([&](uint64_t key) {
      if ((key >> sh) == pref) atomicAdd(&sc->digit_hist[(key >> lo) & ((1u << w) - 1u)], 1u);
    });
    g.sync();
    // digits owned by this thread: [d0, d0 + per)
    constexpr int kPer = (256 + kThreads - 1) / kThreads;
    const int d0 = g.tid * kPer;
    uint32_t s = 0;
    for (int i = 0; i < kPer; ++i)
      if (d0 + i < 256) s += sc->digit_hist[d0 + i];
    uint32_t total;
    uint32_t after = group_excl_suffix(g, s, sc, &total);
    if (after < rank && after + s >= rank) {
      uint32_t acc = after;
      for (int i = kPer - 1; i >= 0; --i) {
        if (d0 + i >= 256) continue;
        uint32_t h = sc->digit_hist[d0 + i];
        if (acc + h >= rank) {
          sc->bcast[0] = static_cast<uint32_t>(d0 + i);
          sc->bcast[1] = rank - acc;
          sc->bcast[2] = h;
          break;
        }
        acc += h;
      }
    }
    g.sync();
    const uint32_t digit = sc->bcast[0];
    rank = sc->bcast[1];
    const uint32_t eq = sc->bcast[2];
    g.sync();
    prefix = (prefix << w) | digit;
    sh = lo;
    if (eq == rank) return prefix << sh;  // every key with this prefix is kept
  }
  return prefix;
}

}  // namespace fp4idx
