// topk_merge.cu -- exact top-k of each query row: from the per-CTA partial
// candidate lists written by the scorer in top-k mode (the merge), or
// straight from the row's logits (the short-context plan).
//
// Every scorer CTA kept, for each row of each item it touched, a superset of
// the top-k of the keys it scored.  The union of those lists therefore holds
// the row's global top-k; this kernel selects it exactly (bucket histogram, then
// radix passes inside the bucket of the k-th key) and writes logical
// positions, values and the valid count.  One CTA per query row.  The row's
// partial lists are read with one warp per list and, when the union fits,
// copied into shared memory so that every later pass runs from there.
#include <cstdint>
#include <cstring>

#include "score_kernel.cuh"

namespace fp4idx {
namespace {

constexpr int kMergeThreads = 512;
constexpr int kMergeWarps = kMergeThreads / 32;

// kLocal: candidate keys held in shared memory.  Rows whose union is larger
// run the same selection from global memory (L2).  The large variant serves
// few rows with many partial lists (long decode); the small one lets three
// CTAs share an SM when there are many rows (prefill).
template <int kLocal>
struct MergeSmem {
  uint32_t hist[kHistBins];
  int32_t slot_cnt[kMaxMergeSlots];
  int32_t slot_off[kMaxMergeSlots + 1];
  int64_t slot_part[kMaxMergeSlots];
  SelectScratch sc;
  int32_t info[8];
  uint64_t out[2048];
  uint64_t buf[kLocal];
};

// The n_out keys >= T of a row (from shared memory when `local`, else
// through for_each_global), optionally sorted by (value desc, position asc),
// written as logical positions / values / valid count of row t.
template <int kLocal, class ForEachGlobal>
__device__ void gather_sort_write(MergeSmem<kLocal>* sm, const Group<kMergeThreads, 0>& g, uint64_t T, int n_out,
                                  bool local, int M, ForEachGlobal&& for_each_global, uint32_t flags, int t, int k,
                                  int32_t* indices, float* values, int32_t* valid_count) {
  const int tid = g.tid;
  if (tid == 0) sm->info[3] = 0;
  g.sync();
  // one slot reservation per group of converged lanes, not per kept key
  auto keep = [&](uint64_t key) {
    const unsigned act = __activemask();
    const bool want = key >= T;
    const unsigned m = __ballot_sync(act, want);
    if (m) {
      const int lane = tid & 31;
      const int leader = __ffs(m) - 1;
      uint32_t o = 0;
      if (lane == leader) o = atomicAdd(reinterpret_cast<uint32_t*>(&sm->info[3]), static_cast<uint32_t>(__popc(m)));
      o = __shfl_sync(act, o, leader) + static_cast<uint32_t>(__popc(m & ((1u << lane) - 1u)));
      if (want && o < 2048u) sm->out[o] = key;
    }
  };
  if (local) {
    for (int e = tid; e < M; e += kMergeThreads) keep(sm->buf[e]);
  } else {
    for_each_global([&](uint64_t key, int) { keep(key); });
  }
  g.sync();

  if (flags & 1u) {
    int P2 = 1;
    while (P2 < n_out) P2 <<= 1;
    for (int i = n_out + tid; i < P2; i += kMergeThreads) sm->out[i] = 0;
    g.sync();
    for (int size = 2; size <= P2; size <<= 1) {
      for (int stride = size >> 1; stride > 0; stride >>= 1) {
        for (int i = tid; i < P2; i += kMergeThreads) {
          const int j = i ^ stride;
          if (j > i) {
            const uint64_t a = sm->out[i], c = sm->out[j];
            const bool desc = (i & size) == 0;
            if (desc ? (a < c) : (a > c)) {
              sm->out[i] = c;
              sm->out[j] = a;
            }
          }
        }
        g.sync();
      }
    }
  }

  const int64_t row = static_cast<int64_t>(t) * k;
  for (int j = tid; j < k; j += kMergeThreads) {
    const bool have = j < n_out;
    const uint64_t key = have ? sm->out[j] : 0;
    indices[row + j] = have ? key_pos(key) : -1;
    if (values) values[row + j] = have ? key_value(key) : -INFINITY;
  }
  if (tid == 0 && valid_count) valid_count[t] = n_out;
}

template <int kMergeLocal>
__global__ void __launch_bounds__(kMergeThreads) topk_merge_kernel(const __grid_constant__ MergeParams mp) {
  const ScoreParams& p = mp.sp;
  extern __shared__ uint8_t smem_raw[];
  using Smem = MergeSmem<kMergeLocal>;
  Smem* sm = reinterpret_cast<Smem*>((reinterpret_cast<uintptr_t>(smem_raw) + 15) & ~uintptr_t(15));
  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  const int t = blockIdx.x;
  const int k = p.k;
  const int cap = topk_part_capacity(k);  // keys per partial list
  const int R = mp.rows_per_cta;
  Group<kMergeThreads, 0> g{tid};

  // Only the shared-memory clear overlaps the previous kernel: every global
  // input (the problem metadata too) may be written by it.
  for (int i = tid; i < kHistBins; i += kMergeThreads) sm->hist[i] = 0;
  pdl_wait();  // item starts and partial lists come from the scorer before this kernel

  // request of row t: largest b with cu_seqlens_q[b] <= t
  int lo = 0, hi = p.num_seqs - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (__ldg(p.cu_seqlens_q + mid) <= t) lo = mid; else hi = mid - 1;
  }
  const int b = lo;
  const int q_local = t - __ldg(p.cu_seqlens_q + b);
  const int item = b * p.row_groups + q_local / R;
  const int r = q_local % R;
  // tile range of the row's item in the scorer's concatenated unit space
  // (an item with tiles holds its tiles, then p.item_overhead units of no tile)
  const int items = p.num_seqs * p.row_groups;
  const int32_t P = __ldg(p.item_start + item), total = __ldg(p.item_start + items);
  const int32_t tiles = max(__ldg(p.item_start + item + 1) - P - p.item_overhead, 0);
  const int C = p.score_ctas;
  const int32_t chunk = total > 0 ? (total + C - 1) / C : 1;
  const int c_lo = tiles > 0 ? P / chunk : 0;
  const int nslots = tiles > 0 ? min((P + tiles - 1) / chunk - c_lo + 1, kMaxMergeSlots) : 0;

  // partial lists of this row: count and global offset of each
  for (int i = tid; i < nslots; i += kMergeThreads) {
    const int c = c_lo + i;
    const int s = static_cast<int64_t>(c) * chunk >= P ? c : C + item;
    const int64_t part = static_cast<int64_t>(s) * R + r;
    sm->slot_part[i] = part;
    sm->slot_cnt[i] = min(max(__ldg(p.part_count + part), 0), cap);
  }
  g.sync();
  if (tid == 0) {
    int32_t acc = 0;
    for (int i = 0; i < nslots; ++i) {
      sm->slot_off[i] = acc;
      acc += sm->slot_cnt[i];
    }
    sm->slot_off[nslots] = acc;
  }
  g.sync();
  const int M = sm->slot_off[nslots];
  const bool local = M <= kMergeLocal;
  const int n_out = M < k ? M : k;

  // visit every candidate in global memory, eight loads in flight per lane
  // so that a long list is not a chain of L2 round trips: with fewer lists
  // than warps (a prefill row has one or two) every thread works on each
  // list in turn, else one warp per list
  auto for_each_global = [&](auto&& fn) {
    constexpr int U = 8;
    if (nslots < kMergeWarps) {
      for (int i = 0; i < nslots; ++i) {
        const uint64_t* keys = p.part_keys + sm->slot_part[i] * cap;
        const int n = sm->slot_cnt[i];
        const int off = sm->slot_off[i];
        for (int e0 = tid; e0 < n; e0 += kMergeThreads * U) {
          uint64_t v[U];
#pragma unroll
          for (int u = 0; u < U; ++u) {
            const int e = e0 + kMergeThreads * u;
            v[u] = e < n ? __ldg(keys + e) : 0;
          }
#pragma unroll
          for (int u = 0; u < U; ++u) {
            const int e = e0 + kMergeThreads * u;
            if (e < n) fn(v[u], off + e);
          }
        }
      }
      return;
    }
    for (int i = warp; i < nslots; i += kMergeWarps) {
      const uint64_t* keys = p.part_keys + sm->slot_part[i] * cap;
      const int n = sm->slot_cnt[i];
      const int off = sm->slot_off[i];
      for (int e0 = lane; e0 < n; e0 += 32 * U) {
        uint64_t v[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int e = e0 + 32 * u;
          v[u] = e < n ? __ldg(keys + e) : 0;
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int e = e0 + 32 * u;
          if (e < n) fn(v[u], off + e);
        }
      }
    }
  };
  // pass 1: bucket histogram (and the copy into shared memory when it fits)
  for_each_global([&](uint64_t key, int at) {
    atomicAdd(&sm->hist[key >> kHistShift], 1u);
    if (local) sm->buf[at] = key;
  });
  g.sync();

  auto hist_get = [&](int bin) { return sm->hist[bin]; };
  uint64_t T = 0;
  if (M > k) {
    uint32_t above = 0;
    const uint32_t bkt = find_kth_bucket(g, hist_get, static_cast<uint32_t>(k), &sm->sc, &above);
    const uint32_t rank = static_cast<uint32_t>(k) - above;
    if (local) {
      T = select_in_bucket(g, bkt, rank, &sm->sc, [&](auto&& fn) {
        for (int e = tid; e < M; e += kMergeThreads) fn(sm->buf[e]);
      });
    } else if (sm->hist[bkt] <= static_cast<uint32_t>(kMergeLocal)) {
      if (tid == 0) sm->info[2] = 0;
      g.sync();
      for_each_global([&](uint64_t key, int) {
        if ((key >> kHistShift) == bkt) {
          const uint32_t o = atomicAdd(reinterpret_cast<uint32_t*>(&sm->info[2]), 1u);
          if (o < static_cast<uint32_t>(kMergeLocal)) sm->buf[o] = key;
        }
      });
      g.sync();
      const int nbuf = min(sm->info[2], kMergeLocal);
      T = select_in_bucket(g, bkt, rank, &sm->sc, [&](auto&& fn) {
        for (int e = tid; e < nbuf; e += kMergeThreads) fn(sm->buf[e]);
      });
    } else {
      T = select_in_bucket(g, bkt, rank, &sm->sc,
                           [&](auto&& fn) { for_each_global([&](uint64_t key, int) { fn(key); }); });
    }
  }

  gather_sort_write(sm, g, T, n_out, local, M, for_each_global, mp.flags, t, k, mp.indices, mp.values,
                    mp.valid_count);
}

// Exact top-k of row t straight from its logits (the short-context plan):
// every visible position's key (value, position) is built from logits[t][s],
// a NaN logit becomes key 0 (never selected), and the same bucket + radix
// selection as the merge runs over them -- in shared memory when the row
// fits, else re-reading the logits.
constexpr int kSelectLocal = 20480;

__global__ void __launch_bounds__(kMergeThreads) topk_select_kernel(const __grid_constant__ MergeParams mp) {
  const ScoreParams& p = mp.sp;
  extern __shared__ uint8_t smem_raw[];
  using Smem = MergeSmem<kSelectLocal>;
  Smem* sm = reinterpret_cast<Smem*>((reinterpret_cast<uintptr_t>(smem_raw) + 15) & ~uintptr_t(15));
  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int t = blockIdx.x;
  const int k = p.k;
  Group<kMergeThreads, 0> g{tid};

  pdl_wait();  // the logits (and any metadata) may come from the kernel before this one
  // request of row t and its visible key count
  int lo = 0, hi = p.num_seqs - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (__ldg(p.cu_seqlens_q + mid) <= t) lo = mid; else hi = mid - 1;
  }
  ItemInfo it;
  it.b = lo;
  it.k_len = max(__ldg(p.cu_seqlens_k + lo + 1) - __ldg(p.cu_seqlens_k + lo), 0);
  const int M = static_cast<int>(min(static_cast<int64_t>(row_visible(p, it, t)), p.ld));
  const bool local = M <= kSelectLocal;
  const float* row_logits = p.logits + static_cast<int64_t>(t) * p.ld;
  // a NaN logit or a position the candidate mask clears has no rank: key 0
  const uint8_t* row_mask = p.cand_mask ? p.cand_mask + static_cast<int64_t>(t) * p.mask_ld : nullptr;
  auto key_of = [&](float v, int s) -> uint64_t {
    return isnan(v) || (row_mask && __ldg(row_mask + s) == 0) ? 0ull : topk_key(v, static_cast<uint32_t>(s));
  };
  // the row's keys, four float4 loads in flight per thread (rows are 16-byte
  // aligned: ld % 4 == 0 and a 16-byte aligned base)
  auto for_each_global = [&](auto&& fn) {
    constexpr int U = 4;
    const float4* row4 = reinterpret_cast<const float4*>(row_logits);
    const int M4 = M >> 2;
    for (int e0 = tid; e0 < M4; e0 += kMergeThreads * U) {
      float4 v[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int e = e0 + kMergeThreads * u;
        v[u] = e < M4 ? __ldg(row4 + e) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int e = e0 + kMergeThreads * u;
        if (e < M4) {
          fn(key_of(v[u].x, 4 * e), 4 * e);
          fn(key_of(v[u].y, 4 * e + 1), 4 * e + 1);
          fn(key_of(v[u].z, 4 * e + 2), 4 * e + 2);
          fn(key_of(v[u].w, 4 * e + 3), 4 * e + 3);
        }
      }
    }
    for (int e = 4 * M4 + tid; e < M; e += kMergeThreads) fn(key_of(__ldg(row_logits + e), e), e);
  };

  for (int i = tid; i < kHistBins; i += kMergeThreads) sm->hist[i] = 0;
  if (tid == 0) sm->info[4] = 0;
  g.sync();
  // pass 1: keys (into shared memory when the row fits), bucket histogram, non-NaN count
  uint32_t mine = 0;
  for_each_global([&](uint64_t key, int at) {
    if (local) sm->buf[at] = key;
    if (key != 0) {
      atomicAdd(&sm->hist[key >> kHistShift], 1u);
      ++mine;
    }
  });
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mine += __shfl_xor_sync(0xffffffffu, mine, o);
  if (lane == 0) atomicAdd(reinterpret_cast<uint32_t*>(&sm->info[4]), mine);
  g.sync();
  const int n_valid = sm->info[4];
  const int n_out = min(n_valid, k);

  auto hist_get = [&](int bin) { return sm->hist[bin]; };
  uint64_t T = 1;  // keeps every non-NaN key (key 0 marks NaN)
  if (n_valid > k) {
    uint32_t above = 0;
    const uint32_t bkt = find_kth_bucket(g, hist_get, static_cast<uint32_t>(k), &sm->sc, &above);
    const uint32_t rank = static_cast<uint32_t>(k) - above;
    if (local) {
      T = select_in_bucket(g, bkt, rank, &sm->sc, [&](auto&& fn) {
        for (int e = tid; e < M; e += kMergeThreads) fn(sm->buf[e]);
      });
    } else {
      T = select_in_bucket(g, bkt, rank, &sm->sc,
                           [&](auto&& fn) { for_each_global([&](uint64_t key, int) { fn(key); }); });
    }
  }
  gather_sort_write(sm, g, T, n_out, local, M, for_each_global, mp.flags, t, k, mp.indices, mp.values,
                    mp.valid_count);
}

// ---------------------------------------------------------------------------
// Rows of at most 16,384 visible keys, sorted output (unsorted output takes
// the cluster kernel below): one 1024-thread CTA per row holds 16
// keys per thread in registers and finds the k-th largest 64-bit key by
// radix levels (11-bit digits), each level counting only the keys that still
// match the prefix; a level whose digit bucket holds exactly the remaining
// rank ends the search.  Then one uniform pass writes the keys >= the
// threshold.  Logits of one row often share a few exponent buckets, so the
// digit counters (16-bit, two per word) come in 8 copies, lane l of every
// warp counting into copy l % 8: at most 4 lanes of a warp update one word,
// and the padded copy stride puts lanes that hold the same digit in
// different copies on different banks.
// ---------------------------------------------------------------------------
constexpr int kSmallThreads = 1024;
constexpr int kSmallPer = 16;
constexpr int kSmallMaxKeys = kSmallThreads * kSmallPer;
constexpr int kSmallCopies = 8;
constexpr int kSmallRow = 1025;  // words per copy (1,024 + 1 of padding)

struct SmallSelectSmem {
  uint32_t hist[kSmallCopies][kSmallRow];  // [lane % 8][digit / 2], digit & 1 selects the half-word
  uint32_t warp_sum[33];
  uint32_t bcast[4];
  uint32_t win_count[4];
  uint64_t out[2048];
};

// Block-wide (1024 threads) exclusive prefix and total of v; `ws` holds 33
// words.  Ends with a barrier, so ws may be reused after it.
__device__ __forceinline__ uint32_t block_excl_prefix(uint32_t v, uint32_t* ws, uint32_t* total) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  uint32_t incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) ws[wid] = incl;
  __syncthreads();
  if (wid == 0) {  // warp 0 turns the 32 warp totals into exclusive offsets
    const uint32_t x = ws[lane];
    uint32_t y = x;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t z = __shfl_up_sync(0xffffffffu, y, o);
      if (lane >= o) y += z;
    }
    ws[lane] = y - x;
    if (lane == 31) ws[32] = y;
  }
  __syncthreads();
  const uint32_t before = ws[wid];
  *total = ws[32];
  __syncthreads();
  return before + incl - v;
}

// One radix level: the keys flagged in `in` are counted by digit (dig[i] <
// 2^W); the digit holding the rank-th largest counted key is returned in d,
// the counted keys in higher digits are taken off rank, eq = keys in digit d,
// total = all counted keys.
template <int W>
__device__ __forceinline__ void small_level(SmallSelectSmem& sm, uint32_t* my_hist, const uint32_t (&dig)[kSmallPer],
                                            uint32_t in, uint32_t& rank, uint32_t& total, uint32_t& d, uint32_t& eq) {
#pragma unroll
  for (int i = 0; i < kSmallPer; ++i)
    if ((in >> i) & 1u) atomicAdd(&my_hist[dig[i] >> 1], 1u << ((dig[i] & 1u) * 16));
  __syncthreads();
  // this thread's digits 2 tid and 2 tid + 1, summed over the copies (which
  // it clears for the next level)
  constexpr uint32_t nb = 1u << W;
  const uint32_t tid = threadIdx.x;
  const uint32_t d0 = 2u * tid;
  uint32_t c0 = 0, c1 = 0;
  if (d0 < nb) {
#pragma unroll
    for (int c = 0; c < kSmallCopies; ++c) {
      const uint32_t x = sm.hist[c][tid];
      c0 += x & 0xFFFFu;
      c1 += x >> 16;
      sm.hist[c][tid] = 0;
    }
  }
  const uint32_t sloc = c0 + c1;
  const uint32_t pre = block_excl_prefix(sloc, sm.warp_sum, &total);
  const uint32_t after = total - pre - sloc;  // counted keys in higher digits
  if (after < rank && after + sloc >= rank) {
    const bool upper = after + c1 >= rank;
    sm.bcast[0] = upper ? d0 + 1 : d0;
    sm.bcast[1] = upper ? after : after + c1;
    sm.bcast[2] = upper ? c1 : c0;
  }
  __syncthreads();
  d = sm.bcast[0];
  rank -= sm.bcast[1];
  eq = sm.bcast[2];
}

__global__ void __launch_bounds__(kSmallThreads) topk_select_small_kernel(const __grid_constant__ MergeParams mp) {
  const ScoreParams& p = mp.sp;
  extern __shared__ uint8_t smem_raw[];
  SmallSelectSmem& sm = *reinterpret_cast<SmallSelectSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 15) & ~uintptr_t(15));
  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int t = blockIdx.x;
  const int k = p.k;
  uint32_t* my_hist = sm.hist[lane % kSmallCopies];

  // The cleared counters come first: they touch shared memory only, so they
  // overlap the scorer's tail (this kernel may start before the scorer
  // completes).  Every global read -- the problem metadata too, which the
  // previous kernel may have written -- waits for it.  The row's stored
  // logits are then loaded at once (they lie inside the row's ld entries
  // whatever its visible length).
  const int cap = static_cast<int>(min(p.ld, static_cast<int64_t>(kSmallMaxKeys)));
  const float4* row4 = reinterpret_cast<const float4*>(p.logits + static_cast<int64_t>(t) * p.ld);
  for (int i = tid; i < kSmallCopies * kSmallRow; i += kSmallThreads) (&sm.hist[0][0])[i] = 0;
  if (tid == 0) {
    sm.bcast[3] = 0;
    sm.win_count[0] = 0;
  }
  pdl_wait();  // the logits come from the kernel before this one
  pdl_launch_dependents();  // the next kernel's on-chip setup may overlap this one
  int lo = 0, hi = p.num_seqs - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (__ldg(p.cu_seqlens_q + mid) <= t) lo = mid; else hi = mid - 1;
  }
  ItemInfo it;
  it.b = lo;
  it.k_len = max(__ldg(p.cu_seqlens_k + lo + 1) - __ldg(p.cu_seqlens_k + lo), 0);
  const int M = min(row_visible(p, it, t), cap);
  float4 v[4];
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const int e = tid + kSmallThreads * u;
    v[u] = 4 * e < cap ? __ldg(row4 + e) : make_float4(0.f, 0.f, 0.f, 0.f);
  }

  // Key i of this thread (position 4 (tid + 1024 (i / 4)) + i % 4) as the
  // two halves of its 64-bit top-k key: kh = order-preserving bits of the
  // logit, kl = ~position (bits 31..14 all ones, positions < 2^14).  Bit i
  // of `present`: the position is visible, not cleared by the candidate
  // mask, and the logit not NaN.
  uint32_t kh[kSmallPer], kl[kSmallPer];
  uint32_t present = 0;
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const int pos = 4 * (tid + kSmallThreads * u);
    const float f[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const bool ok = pos + c < M && !isnan(f[c]) &&
                      (!p.cand_mask || __ldg(p.cand_mask + static_cast<int64_t>(t) * p.mask_ld + pos + c) != 0);
      const uint64_t key = topk_key(f[c], static_cast<uint32_t>(pos + c));
      kh[4 * u + c] = static_cast<uint32_t>(key >> 32);
      kl[4 * u + c] = static_cast<uint32_t>(key);
      present |= ok ? 1u << (4 * u + c) : 0u;
    }
  }
  __syncthreads();

  // Radix levels over the key: the 32 value bits as 11 + 11 + 10, then the
  // low 14 bits of ~position as 7 + 7.  Each level counts only the keys
  // matching the prefix fixed so far; the first level's total is the number
  // of present keys; a level whose digit holds exactly the remaining rank
  // ends the search (every key with that prefix is in the top-k).
  uint32_t dig[kSmallPer];
  uint32_t rank = static_cast<uint32_t>(k), total = 0, d = 0, eq = 0;
  // The first level first counts only the keys within kWindow digits (six
  // binades) below the largest key's digit: when they are at least k, the
  // k-th key is among them and the other keys never touch the counters.
  // Otherwise (or with fewer than k keys) the level is redone over all keys.
  constexpr uint32_t kWindow = 24;
  uint32_t top = 0, n_present = static_cast<uint32_t>(__popc(present));
#pragma unroll
  for (int i = 0; i < kSmallPer; ++i) {
    dig[i] = kh[i] >> 21;
    if ((present >> i) & 1u) top = max(top, dig[i]);
  }
  top = __reduce_max_sync(0xffffffffu, top);
  n_present = __reduce_add_sync(0xffffffffu, n_present);
  if (lane == 0) {
    atomicMax(&sm.bcast[3], top);
    atomicAdd(&sm.win_count[0], n_present);
  }
  __syncthreads();
  const uint32_t n_valid = sm.win_count[0];
  const bool all_kept = n_valid <= static_cast<uint32_t>(k);
  if (!all_kept) {
    const uint32_t lo_digit = sm.bcast[3] > kWindow ? sm.bcast[3] - kWindow : 0u;
    uint32_t in = 0;
#pragma unroll
    for (int i = 0; i < kSmallPer; ++i) in |= dig[i] >= lo_digit ? 1u << i : 0u;
    small_level<11>(sm, my_hist, dig, in & present, rank, total, d, eq);
    if (total < static_cast<uint32_t>(k)) {
      rank = static_cast<uint32_t>(k);
      small_level<11>(sm, my_hist, dig, present, rank, total, d, eq);
    }
  }
  uint32_t Th = 0, Tl = 0;  // threshold key: exactly k present keys are >= (Th, Tl)
  if (!all_kept) {
    uint32_t P = d;  // 11-bit prefix
    Th = P << 21;
    if (eq != rank) {
      uint32_t in = 0;
#pragma unroll
      for (int i = 0; i < kSmallPer; ++i) {
        in |= (kh[i] >> 21) == P ? 1u << i : 0u;
        dig[i] = (kh[i] >> 10) & 0x7FFu;
      }
      small_level<11>(sm, my_hist, dig, in & present, rank, total, d, eq);
      P = (P << 11) | d;  // 22 bits
      Th = P << 10;
      if (eq != rank) {
        in = 0;
#pragma unroll
        for (int i = 0; i < kSmallPer; ++i) {
          in |= (kh[i] >> 10) == P ? 1u << i : 0u;
          dig[i] = kh[i] & 0x3FFu;
        }
        small_level<10>(sm, my_hist, dig, in & present, rank, total, d, eq);
        Th = (P << 10) | d;  // all 32 value bits
        Tl = 0xFFFFC000u;
        if (eq != rank) {
          in = 0;
#pragma unroll
          for (int i = 0; i < kSmallPer; ++i) {
            in |= kh[i] == Th ? 1u << i : 0u;
            dig[i] = (kl[i] >> 7) & 0x7Fu;
          }
          small_level<7>(sm, my_hist, dig, in & present, rank, total, d, eq);
          const uint32_t P2 = d;
          Tl = 0xFFFFC000u | (P2 << 7);
          if (eq != rank) {
            in = 0;
#pragma unroll
            for (int i = 0; i < kSmallPer; ++i) {
              in |= (kh[i] == Th && ((kl[i] >> 7) & 0x7Fu) == P2) ? 1u << i : 0u;
              dig[i] = kl[i] & 0x7Fu;
            }
            small_level<7>(sm, my_hist, dig, in & present, rank, total, d, eq);
            Tl |= d;
          }
        }
      }
    }
  }
  const int n_out = static_cast<int>(min(n_valid, static_cast<uint32_t>(k)));

  // the n_out keys >= the threshold, at offsets from a block prefix of
  // per-thread counts
  uint32_t mask = present;
  if (!all_kept) {
#pragma unroll
    for (int i = 0; i < kSmallPer; ++i)
      if (!(kh[i] > Th || (kh[i] == Th && kl[i] >= Tl))) mask &= ~(1u << i);
  }
  uint32_t total_kept;
  uint32_t o = block_excl_prefix(static_cast<uint32_t>(__popc(mask)), sm.warp_sum, &total_kept);
  const int64_t row = static_cast<int64_t>(t) * k;
  if (mp.flags & 1u) {
#pragma unroll
    for (int i = 0; i < kSmallPer; ++i)
      if ((mask >> i) & 1u) {
        if (o < 2048u) sm.out[o] = (static_cast<uint64_t>(kh[i]) << 32) | kl[i];
        ++o;
      }
    int P2 = 1;
    while (P2 < n_out) P2 <<= 1;
    __syncthreads();
    for (int i = n_out + tid; i < P2; i += kSmallThreads) sm.out[i] = 0;
    __syncthreads();
    for (int size = 2; size <= P2; size <<= 1) {
      for (int stride = size >> 1; stride > 0; stride >>= 1) {
        for (int i = tid; i < P2; i += kSmallThreads) {
          const int j = i ^ stride;
          if (j > i) {
            const uint64_t a = sm.out[i], c = sm.out[j];
            const bool desc = (i & size) == 0;
            if (desc ? (a < c) : (a > c)) {
              sm.out[i] = c;
              sm.out[j] = a;
            }
          }
        }
        __syncthreads();
      }
    }
    for (int j = tid; j < k; j += kSmallThreads) {
      const bool have = j < n_out;
      const uint64_t kk = have ? sm.out[j] : 0;
      mp.indices[row + j] = have ? key_pos(kk) : -1;
      if (mp.values) mp.values[row + j] = have ? key_value(kk) : -INFINITY;
    }
  } else {
    // unsorted: kept keys are placed in shared memory at their output slots,
    // then written out in order (coalesced stores)
#pragma unroll
    for (int i = 0; i < kSmallPer; ++i)
      if ((mask >> i) & 1u) {
        if (o < 2048u) sm.out[o] = (static_cast<uint64_t>(kh[i]) << 32) | kl[i];
        ++o;
      }
    __syncthreads();
    for (int j = tid; j < k; j += kSmallThreads) {
      const bool have = j < n_out;
      const uint64_t kk = have ? sm.out[j] : 0;
      mp.indices[row + j] = have ? key_pos(kk) : -1;
      if (mp.values) mp.values[row + j] = have ? key_value(kk) : -INFINITY;
    }
  }
  if (tid == 0 && mp.valid_count) mp.valid_count[t] = n_out;
}

// ---------------------------------------------------------------------------
// The same rows, unsorted output: one cluster of 8 CTAs per row, so that a
// row's keys are counted by eight SMs.  CTA r of the cluster holds positions
// [2048 r, 2048 r + 2048), eight keys per thread in registers, as 46-bit
// search keys: the 32 order-preserving value bits, then the low 14 bits of
// ~position (positions are < 2^14 here, so the dropped bits of ~position are
// all ones and the order is that of the full top-k key).
//
// A radix level counts the keys it is given into each CTA's own digit
// counters.  After a cluster barrier, CTA r sums digits [r per, (r+1) per)
// over the eight CTAs' counters (distributed shared memory), scans them, and
// stores their total in every CTA; after a second barrier every CTA knows
// which CTA's digits hold the rank-th key and finds the digit by reading
// that CTA's scanned sums.  All CTAs take every decision from the same
// exchanged data, so they pass the same barriers, and a cluster barrier
// costs about as much as a pass over the keys, so there are few of them.
//
// The first level counts the top 16 bits of the keys within 1,024 digits
// (eight binades) of the largest, with stores instead of remote reads.  Each
// CTA counts within 1,024 digits of its own largest key and, before the
// first barrier, stores each count at the digit's residue mod 1,024 in the
// CTA owning that residue, and its largest digit and number of selectable
// keys in every CTA.  The row's window (the 1,024 digits below the largest
// of all) holds one digit of each residue and lies inside every CTA's own
// window wherever that CTA has keys, so an owner sums, per residue, the
// counts of the CTAs whose largest digit is at or above the window's digit
// of that residue, and stores the sums in every CTA; after the second
// barrier every CTA scans the whole window by itself.  When fewer than k
// keys lie in the window, an 11-bit level over every key takes its place.
// Further levels narrow the digit until it holds exactly the remaining rank,
// or at most kClCand keys: those are gathered into every CTA (a region per
// source CTA), with each CTA's count of keys above the digit, and the
// rank-th of them is found by direct comparison; every CTA then knows each
// CTA's count of kept keys, so the output offsets need no further exchange.
// ---------------------------------------------------------------------------
constexpr int kClCtas = 8;
constexpr int kClThreads = 256;
constexpr int kClPer = 8;            // keys per thread
constexpr int kClCand = kClThreads;  // gathered keys: one per thread when ranked
constexpr int kClWin = 1024;         // first-level window (digits)
constexpr int kClRows = 12;          // exchange rows: start (2), at most 7 levels, output, gathered counts (2)
constexpr int kClAboveRow = kClRows - 1;
constexpr int kClCandRow = kClRows - 2;
static_assert(kClCtas * kClThreads * kClPer == kSmallMaxKeys, "the cluster covers every short row");

struct ClusterSelectSmem {
  uint32_t hist[2048];              // this CTA's digit counters
  uint32_t bsum[kClThreads];        // owned digits: counts summed over the cluster
  uint32_t babove[kClThreads];      // owned digits: counted keys in the higher owned digits
  uint64_t cand[kClCtas][kClCand];  // gathered keys of the final digit, by source CTA
  uint64_t flat[kClCand];           // the same keys, regions in order
  uint32_t inc[kClCtas][kClWin / kClCtas];  // owner: first-level counts of its residues, by source CTA
  uint32_t gh[kClWin];              // first-level counts of the window, by residue
  uint32_t xchg[kClRows][kClCtas];  // [exchange][source CTA]
  uint32_t ws[kClThreads / 32];
  uint32_t kc[kClCtas];             // gathered keys kept, by source CTA
  uint32_t bc[3];
  uint32_t cand_n, lmax, lcnt, labove;  // cand_n: this CTA's gathered keys
  uint64_t thr;
};

// Exclusive prefix of v over the CTA's threads and its total.  ws (one word
// per warp) is read after the barrier inside; the caller separates two uses
// by a barrier.
__device__ __forceinline__ uint32_t cl_prefix(uint32_t v, uint32_t* ws, uint32_t* total) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  uint32_t incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) ws[wid] = incl;
  __syncthreads();
  uint32_t before = 0, tot = 0;
#pragma unroll
  for (int w = 0; w < kClThreads / 32; ++w) {
    const uint32_t x = ws[w];
    before += w < wid ? x : 0u;
    tot += x;
  }
  *total = tot;
  return before + incl - v;
}

// One radix level over the cluster.  Key i of this thread is counted under
// digit dig(i) (< nbins) when bit i of `in` is set.  When the cluster counted
// at least `rank` keys: d = the digit holding the rank-th largest counted
// key, rank -= the counted keys in higher digits, eq = the keys counted in d.
// total = all counted keys (d, rank, eq unchanged when total < rank).  The
// counters are zero on entry and on return.
template <class Dig>
__device__ __forceinline__ void cluster_level(ClusterSelectSmem& sm, uint32_t r, int xrow, uint32_t in, int nbins,
                                              Dig dig, uint32_t& rank, uint32_t& d, uint32_t& eq,
                                              uint32_t& total) {
  const int tid = threadIdx.x;
#pragma unroll
  for (int i = 0; i < kClPer; ++i)
    if ((in >> i) & 1u) atomicAdd(&sm.hist[dig(i)], 1u);
  cluster_sync();  // every CTA's counters are complete
  const int per = (nbins + kClCtas - 1) / kClCtas;
  const int b = static_cast<int>(r) * per + tid;
  uint32_t s = 0;
  if (tid < per && b < nbins) {
    uint32_t a[kClCtas];
#pragma unroll
    for (int c = 0; c < kClCtas; ++c) a[c] = dsmem_ld_u32(dsmem_addr(&sm.hist[b], c));
#pragma unroll
    for (int c = 0; c < kClCtas; ++c) s += a[c];
  }
  uint32_t tot;
  const uint32_t pre = cl_prefix(s, sm.ws, &tot);
  if (tid < per) {
    sm.bsum[tid] = s;
    sm.babove[tid] = tot - pre - s;  // owned digits are ascending with tid
  }
  if (tid < kClCtas) dsmem_st_u32(dsmem_addr(&sm.xchg[xrow][r], tid), tot);
  cluster_sync();  // every owner's total and scanned sums are in place
  // the owner of the rank-th key's digit: CTAs own ascending digit ranges
  uint32_t acc = 0, ro = 0, rk = 0;
  bool found = false;
#pragma unroll
  for (int c = kClCtas - 1; c >= 0; --c) {
    const uint32_t x = sm.xchg[xrow][c];
    if (!found && acc + x >= rank) {
      found = true;
      ro = static_cast<uint32_t>(c);
      rk = rank - acc;
    }
    acc += x;
  }
  total = acc;
  // every CTA read this CTA's counters before the barrier
  for (int i = tid; i < nbins; i += kClThreads) sm.hist[i] = 0;
  if (found && tid < per) {
    const uint32_t x = dsmem_ld_u32(dsmem_addr(&sm.bsum[tid], ro));
    const uint32_t above = dsmem_ld_u32(dsmem_addr(&sm.babove[tid], ro));
    if (above < rk && above + x >= rk) {
      sm.bc[0] = ro * static_cast<uint32_t>(per) + static_cast<uint32_t>(tid);
      sm.bc[1] = rk - above;
      sm.bc[2] = x;
    }
  }
  __syncthreads();
  if (found) {
    d = sm.bc[0];
    rank = sm.bc[1];
    eq = sm.bc[2];
  }
}

__global__ void __launch_bounds__(kClThreads) topk_select_cluster_kernel(const __grid_constant__ MergeParams mp) {
  const ScoreParams& p = mp.sp;
  __shared__ ClusterSelectSmem sm;
  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const uint32_t r = cluster_ctarank();
  const int t = static_cast<int>(blockIdx.x / kClCtas);
  const int k = p.k;

  // This CTA's own state first (shared memory only, so it overlaps the
  // scorer's tail); the arrive publishes it to the cluster, whose CTAs touch
  // it only after the matching wait.
  for (int i = tid; i < 2048; i += kClThreads) sm.hist[i] = 0;
  if (tid < kClCtas) sm.kc[tid] = 0;
  if (tid == 0) {
    sm.cand_n = 0;
    sm.lmax = 0;
    sm.lcnt = 0;
    sm.labove = 0;
    sm.thr = 0;
  }
  cluster_arrive();
  pdl_wait();  // the logits come from the kernel before this one
  pdl_launch_dependents();
  int lo = 0, hi = p.num_seqs - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (__ldg(p.cu_seqlens_q + mid) <= t) lo = mid; else hi = mid - 1;
  }
  ItemInfo it;
  it.b = lo;
  it.k_len = max(__ldg(p.cu_seqlens_k + lo + 1) - __ldg(p.cu_seqlens_k + lo), 0);
  const int cap = static_cast<int>(min(p.ld, static_cast<int64_t>(kSmallMaxKeys)));
  const int M = min(row_visible(p, it, t), cap);
  const float4* row4 = reinterpret_cast<const float4*>(p.logits + static_cast<int64_t>(t) * p.ld);
  float4 v[2];
#pragma unroll
  for (int u = 0; u < 2; ++u) {
    const int e = static_cast<int>(r) * (kClThreads * 2) + tid + kClThreads * u;
    v[u] = 4 * e < cap ? __ldg(row4 + e) : make_float4(0.f, 0.f, 0.f, 0.f);
  }
  // Key i of this thread: position 4 (512 r + tid + 256 (i / 4)) + i % 4.
  // Bit i of `present`: visible, not cleared by the candidate mask, not NaN.
  uint64_t K[kClPer];
  uint32_t present = 0, top = 0;
#pragma unroll
  for (int u = 0; u < 2; ++u) {
    const int pos = 4 * (static_cast<int>(r) * (kClThreads * 2) + tid + kClThreads * u);
    const float f[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const bool ok = pos + c < M && !isnan(f[c]) &&
                      (!p.cand_mask || __ldg(p.cand_mask + static_cast<int64_t>(t) * p.mask_ld + pos + c) != 0);
      const uint64_t key = topk_key(f[c], static_cast<uint32_t>(pos + c));
      const uint64_t s46 = ((key >> 32) << 14) | (key & 0x3FFFu);
      K[4 * u + c] = s46;
      present |= ok ? 1u << (4 * u + c) : 0u;
      if (ok) top = max(top, static_cast<uint32_t>(s46 >> 30));
    }
  }
  top = __reduce_max_sync(0xffffffffu, top);
  const uint32_t cnt = __reduce_add_sync(0xffffffffu, static_cast<uint32_t>(__popc(present)));
  __syncthreads();  // the zeroed state above is visible to the whole CTA
  if (lane == 0) {
    atomicMax(&sm.lmax, top);
    atomicAdd(&sm.lcnt, cnt);
  }
  __syncthreads();
  // first level, counting half: the top 16 bits within 1,024 digits of this
  // CTA's largest
  const uint32_t lmax = sm.lmax;
  const uint32_t lwlo = lmax >= 1023u ? lmax - 1023u : 0u;
#pragma unroll
  for (int i = 0; i < kClPer; ++i) {
    const uint32_t dg = static_cast<uint32_t>(K[i] >> 30);
    if (((present >> i) & 1u) && dg >= lwlo) atomicAdd(&sm.hist[dg - lwlo], 1u);
  }
  __syncthreads();
  cluster_wait();  // every CTA of the cluster has set up its state
  // each count to the owner of its digit's residue (and cleared)
#pragma unroll
  for (int j = 0; j < kClWin / kClThreads; ++j) {
    const uint32_t idx = static_cast<uint32_t>(tid + kClThreads * j);
    const uint32_t x = sm.hist[idx];
    sm.hist[idx] = 0;
    const uint32_t rho = (lwlo + idx) & (kClWin - 1);
    dsmem_st_u32(dsmem_addr(&sm.inc[r][rho % (kClWin / kClCtas)], rho / (kClWin / kClCtas)), x);
  }
  if (tid < kClCtas) {
    dsmem_st_u32(dsmem_addr(&sm.xchg[0][r], static_cast<uint32_t>(tid)), lmax);
    dsmem_st_u32(dsmem_addr(&sm.xchg[1][r], static_cast<uint32_t>(tid)), sm.lcnt);
  }
  cluster_sync();  // counters complete; every CTA's largest digit and count in place
  uint32_t gmax = 0, n_valid = 0;
#pragma unroll
  for (int c = 0; c < kClCtas; ++c) {
    gmax = max(gmax, sm.xchg[0][c]);
    n_valid += sm.xchg[1][c];
  }

  int xrow = 2;
  const bool all_kept = n_valid <= static_cast<uint32_t>(k);
  bool counted = all_kept;  // every CTA's count of kept keys known without an exchange
  uint32_t base = 0, n_all = n_valid;
  if (all_kept) {
#pragma unroll
    for (int c = 0; c < kClCtas; ++c) base += c < static_cast<int>(r) ? sm.xchg[1][c] : 0u;
  }
  uint64_t T46 = 0;  // kept: present keys >= T46 (every present key when all_kept)
  if (!all_kept) {
    uint32_t rank = static_cast<uint32_t>(k), d = 0, eq = 0, total = 0;
    // the row's window [wlo, gmax]: this CTA owns residues
    // [128 r, 128 r + 128); the window's digit of residue rho is
    // wlo + ((rho - wlo) mod 1024), counted by CTA c when c's largest digit
    // is at or above it (c's window [lwlo_c, lmax_c] then holds it, as
    // lwlo_c <= wlo)
    const uint32_t wlo = gmax >= 1023u ? gmax - 1023u : 0u;
    constexpr int kOwn = kClWin / kClCtas;
    if (tid < kOwn) {
      const uint32_t rho = r * kOwn + static_cast<uint32_t>(tid);
      const uint32_t g = wlo + ((rho - wlo) & (kClWin - 1));
      uint32_t s = 0;
#pragma unroll
      for (int c = 0; c < kClCtas; ++c) s += g <= sm.xchg[0][c] ? sm.inc[c][tid] : 0u;
#pragma unroll
      for (int c = 0; c < kClCtas; ++c) dsmem_st_u32(dsmem_addr(&sm.gh[rho], static_cast<uint32_t>(c)), s);
    }
    cluster_sync();  // the window's counts are in every CTA
    {
      // digits wlo + 4 tid .. + 3 of the window
      constexpr int kQ = kClWin / kClThreads;
      uint32_t c4[kQ], s4 = 0;
#pragma unroll
      for (int q = 0; q < kQ; ++q) {
        c4[q] = sm.gh[(wlo + kQ * tid + q) & (kClWin - 1)];
        s4 += c4[q];
      }
      uint32_t tot;
      uint32_t a = cl_prefix(s4, sm.ws, &tot);
      a = tot - a - s4;  // window keys in the digits of higher threads
      total = tot;
      if (total >= rank) {
#pragma unroll
        for (int q = kQ - 1; q >= 0; --q) {
          if (a < rank && a + c4[q] >= rank) {
            sm.bc[0] = static_cast<uint32_t>(kQ * tid + q);
            sm.bc[1] = rank - a;
            sm.bc[2] = c4[q];
          }
          a += c4[q];
        }
      }
      __syncthreads();
      if (total >= rank) {
        d = sm.bc[0];
        rank = sm.bc[1];
        eq = sm.bc[2];
      }
    }
    uint64_t pre;
    int sh;
    if (total >= rank) {
      pre = wlo + d;
      sh = 30;
    } else {
      cluster_level(sm, r, xrow++, present, 2048, [&](int i) { return static_cast<uint32_t>(K[i] >> 35); }, rank,
                    d, eq, total);
      pre = d;
      sh = 35;
    }
    bool ranked = false;
    // sh > 0 while eq != rank (a full 46-bit prefix matches one key); the
    // level count is bounded all the same (at most four levels follow)
    for (int lv = 0; lv < 6 && eq != rank && sh > 0; ++lv) {
      if (eq <= static_cast<uint32_t>(kClCand)) {
        // gather the eq keys of the digit into every CTA, with this CTA's
        // count of keys above the digit, then rank them
        uint32_t n_above = 0;
#pragma unroll
        for (int i = 0; i < kClPer; ++i) {
          const bool sel = (present >> i) & 1u;
          const uint64_t dg = K[i] >> sh;
          n_above += sel && dg > pre ? 1u : 0u;
          const bool mine = sel && dg == pre;
          const uint32_t m = __ballot_sync(0xffffffffu, mine);
          if (m) {  // one slot reservation per warp
            const int leader = __ffs(m) - 1;
            uint32_t b0 = 0;
            if (lane == leader) b0 = atomicAdd(&sm.cand_n, static_cast<uint32_t>(__popc(m)));
            b0 = __shfl_sync(0xffffffffu, b0, leader);
            const uint32_t slot = b0 + static_cast<uint32_t>(__popc(m & ((1u << lane) - 1u)));
            if (mine && slot < static_cast<uint32_t>(kClCand)) {
#pragma unroll
              for (int c = 0; c < kClCtas; ++c) dsmem_st_u64(dsmem_addr(&sm.cand[r][slot], c), K[i]);
            }
          }
        }
        n_above = __reduce_add_sync(0xffffffffu, n_above);
        if (lane == 0) atomicAdd(&sm.labove, n_above);
        __syncthreads();
        if (tid < kClCtas) {
          dsmem_st_u32(dsmem_addr(&sm.xchg[kClAboveRow][r], static_cast<uint32_t>(tid)), sm.labove);
          dsmem_st_u32(dsmem_addr(&sm.xchg[kClCandRow][r], static_cast<uint32_t>(tid)), sm.cand_n);
        }
        cluster_sync();  // the last access to another CTA's shared memory on this path is before it
        // candidate tid of the regions taken in order (eq of them, at most kClCand)
        uint32_t ncs[kClCtas];
#pragma unroll
        for (int c = 0; c < kClCtas; ++c) ncs[c] = min(sm.xchg[kClCandRow][c], static_cast<uint32_t>(kClCand));
        uint64_t x = 0;
        int src = 0;
        if (tid < static_cast<int>(eq)) {
          int j = tid;
#pragma unroll
          for (int c = 0; c < kClCtas; ++c)
            if (src == c && j >= static_cast<int>(ncs[c])) {
              j -= static_cast<int>(ncs[c]);
              src = c + 1;
            }
          if (src < kClCtas) x = sm.cand[src][j];
          sm.flat[tid] = x;
        }
        __syncthreads();
        if (tid < static_cast<int>(eq) && src < kClCtas) {
          uint32_t above = 0;
          for (uint32_t jj = 0; jj < eq; ++jj) above += sm.flat[jj] > x ? 1u : 0u;
          if (above == rank - 1) sm.thr = x;
        }
        __syncthreads();
        T46 = sm.thr;
        // kept gathered keys by source CTA
        if (tid < static_cast<int>(eq) && src < kClCtas && x >= T46) atomicAdd(&sm.kc[src], 1u);
        __syncthreads();
        n_all = 0;
#pragma unroll
        for (int c = 0; c < kClCtas; ++c) {
          const uint32_t n = sm.xchg[kClAboveRow][c] + sm.kc[c];
          base += c < static_cast<int>(r) ? n : 0u;
          n_all += n;
        }
        counted = true;
        ranked = true;
        break;
      }
      const int w = sh < 11 ? sh : 11;
      const int shn = sh - w;
      uint32_t in = 0;
#pragma unroll
      for (int i = 0; i < kClPer; ++i) in |= (K[i] >> sh) == pre ? 1u << i : 0u;
      cluster_level(sm, r, xrow++, in & present, 1 << w,
                    [&](int i) { return static_cast<uint32_t>(K[i] >> shn) & ((1u << w) - 1u); }, rank, d, eq,
                    total);
      pre = (pre << w) | d;
      sh = shn;
    }
    if (!ranked) T46 = pre << sh;
  }

  uint32_t keep = present;
  if (!all_kept) {
#pragma unroll
    for (int i = 0; i < kClPer; ++i)
      if (K[i] < T46) keep &= ~(1u << i);
  }
  uint32_t ctot;
  uint32_t o = cl_prefix(static_cast<uint32_t>(__popc(keep)), sm.ws, &ctot);
  if (!counted) {
    if (tid < kClCtas) dsmem_st_u32(dsmem_addr(&sm.xchg[xrow][r], static_cast<uint32_t>(tid)), ctot);
    cluster_sync();  // the last access to another CTA's shared memory on this path is before it
    base = 0;
    n_all = 0;
#pragma unroll
    for (int c = 0; c < kClCtas; ++c) {
      const uint32_t x = sm.xchg[xrow][c];
      base += c < static_cast<int>(r) ? x : 0u;
      n_all += x;
    }
  }
  o += base;
  const int n_out = static_cast<int>(min(n_all, static_cast<uint32_t>(k)));
  const int64_t row = static_cast<int64_t>(t) * k;
#pragma unroll
  for (int i = 0; i < kClPer; ++i)
    if ((keep >> i) & 1u) {
      if (o < static_cast<uint32_t>(k)) {
        const uint64_t key = ((K[i] >> 14) << 32) | 0xFFFFC000u | (K[i] & 0x3FFFu);
        mp.indices[row + o] = key_pos(key);
        if (mp.values) mp.values[row + o] = key_value(key);
      }
      ++o;
    }
  for (int j = n_out + static_cast<int>(r) * kClThreads + tid; j < k; j += kClCtas * kClThreads) {
    mp.indices[row + j] = -1;
    if (mp.values) mp.values[row + j] = -INFINITY;
  }
  if (r == 0 && tid == 0 && mp.valid_count) mp.valid_count[t] = n_out;
}

// Launch with programmatic stream serialization: the kernel's CTAs may be
// scheduled once the previous kernel of the stream (the scorer, which
// signals early) allows it; the kernel itself waits (pdl_wait) for that
// kernel's completion before it reads the scorer's output.
cudaError_t launch_dependent(void (*kern)(MergeParams), int grid, int threads, int smem_bytes, cudaStream_t stream,
                             const MergeParams& p) {
  cudaLaunchConfig_t cfg;
  std::memset(&cfg, 0, sizeof(cfg));
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(static_cast<unsigned>(threads));
  cfg.dynamicSmemBytes = static_cast<size_t>(smem_bytes);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, p);
}

template <int kLocal>
cudaError_t launch_merge_t(const MergeParams& p, int rows, cudaStream_t stream) {
  const int bytes = static_cast<int>(sizeof(MergeSmem<kLocal>) + 16);
  cudaError_t e = cudaFuncSetAttribute(topk_merge_kernel<kLocal>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e != cudaSuccess) return e;
  return launch_dependent(topk_merge_kernel<kLocal>, rows, kMergeThreads, bytes, stream, p);
}

}  // namespace

cudaError_t launch_topk_select(const MergeParams& p, int rows, cudaStream_t stream) {
  if (rows <= 0) return cudaSuccess;
  if (p.sp.max_seqlen_k <= kSmallMaxKeys && !(p.flags & 1u) &&
      static_cast<int64_t>(rows) * kClCtas <= static_cast<int64_t>(INT32_MAX)) {
    cudaLaunchConfig_t cfg;
    std::memset(&cfg, 0, sizeof(cfg));
    cfg.gridDim = dim3(static_cast<unsigned>(rows * kClCtas));
    cfg.blockDim = dim3(kClThreads);
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = kClCtas;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, topk_select_cluster_kernel, p);
  }
  if (p.sp.max_seqlen_k <= kSmallMaxKeys) {
    const int sbytes = static_cast<int>(sizeof(SmallSelectSmem) + 16);
    cudaError_t e = cudaFuncSetAttribute(topk_select_small_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, sbytes);
    if (e != cudaSuccess) return e;
    return launch_dependent(topk_select_small_kernel, rows, kSmallThreads, sbytes, stream, p);
  }
  const int bytes = static_cast<int>(sizeof(MergeSmem<kSelectLocal>) + 16);
  cudaError_t e = cudaFuncSetAttribute(topk_select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e != cudaSuccess) return e;
  return launch_dependent(topk_select_kernel, rows, kMergeThreads, bytes, stream, p);
}

cudaError_t launch_topk_merge(const MergeParams& p, int rows, bool many_rows, cudaStream_t stream) {
  if (rows <= 0) return cudaSuccess;
  return many_rows ? launch_merge_t<8192>(p, rows, stream) : launch_merge_t<20480>(p, rows, stream);
}

}  // namespace fp4idx
