// block_kernel.cu -- per-128-key block max of the unweighted FP4 dot, sm_103a.
//
//   scores[h][kb][t] = max over visible s in [128 kb, 128 kb + 128) of q[t,h] . k[s, hk(h)]
//                      (-inf when the block holds no visible key)
// (M3-indexer README, "数学语义" and "输出 shape 和类型"; hk(h) = h / (Hq/Hkv)).
//
// Queries on the MMA M dimension.  One item = (request b, K head hk, RT query
// rows).  Its 128 MMA rows are the g = Hq/Hkv query heads of group hk times
// the RT rows (row m = h_local * RT + t_local), brought in by one 3-D TMA box.
// A tile is one 128-key block of the item: D[m, n] = Q_real[m] . K_real[128 kb + n]
// lands in TMEM lane m, column n, so an epilogue thread owns one (head, row)
// and reduces the block along its 128 columns without shuffles.  Blocks after
// the last visible key of every row of the item are not computed; their
// scores are written as -inf.
//
// Warp roles (160 + 128 * kGroups threads):
//   warps 0, 4  producers, alternate tiles: per tile the K codes by TMA
//               (64-byte swizzle) and the page's raw K scales by one bulk
//               copy, into a kStages-deep ring; warp 0 also loads Q codes of
//               each item by TMA and Q scales by cp.async (double buffered,
//               one item ahead).
//   warp 1      MMA: TMEM owner; one thread waits for the tiles' scales and
//               free accumulators and issues, two tiles at a time with their
//               K halves interleaved, K = 64 block-scaled MMAs into a
//               triple-buffered accumulator, nothing else.
//   warps 2, 3  scales, alternate tiles: Q scales -> TMEM once per item
//               (warp 2); per tile the raw K scales are transposed into the
//               128-row scale layout (each row: the 32x4x4 atom line of its
//               lane) and one tcgen05.cp 128x128b/256b moves them to TMEM.
//   warps 5..   epilogue, one group of four warps (one per TMEM lane
//               quadrant) per accumulator buffer, so three tiles drain at
//               once: tcgen05.ld of the 128 columns, masked max
//               (NaN-propagating), one fp32 store per (head, row).
//
// Work split: the tiles of all items are concatenated and cut into one equal
// contiguous chunk per CTA; every output element is produced by exactly one
// tile, so no cross-CTA combination is needed.
#include "formats.cuh"
#include "internal.h"
#include "ptx.cuh"
#include "topk_smem.cuh"  // Group

namespace fp4idx {
namespace {

constexpr int kStages = 16;
constexpr int kAccBufs = 3;
constexpr int kKsfSlots = 8;  // K-scale slots (TMEM and staging); > kAccBufs (see the scale warps)
constexpr int kGroups = kAccBufs;  // epilogue group e drains accumulator e
constexpr int kEpiWarp0 = 5;
constexpr int kThreads = 32 * kEpiWarp0 + 128 * kGroups;  // producers, MMA, scale warps, epilogue groups
constexpr uint32_t kTmemCols = 512;
static_assert(kAccBufs < kKsfSlots, "K-scale slot reuse");

struct BlockCta {
  uint32_t tmem_base;
  int32_t abort;
  int32_t item0;        // item holding the first tile of this CTA's chunk
  int32_t item0_start;  // global tile index where item0 starts
  int32_t total_tiles;
  int32_t chunk;
  int32_t pad[2];
};

template <int FMT>
struct BlockLayout {
  using F = FmtTraits<FMT>;
  static constexpr uint32_t kCodes = 0;                                // kStages x 8 KB K codes
  static constexpr uint32_t kQ = kCodes + kStages * 8192;              // 2 x 8 KB Q codes
  static constexpr uint32_t kKraw = kQ + 2 * 8192;                     // kStages x 128 keys x G raw K scales
  static constexpr uint32_t kKsf = kKraw + kStages * 128 * F::G;       // kKsfSlots x kAtoms x 2048 (128 rows)
  static constexpr uint32_t kQsf = kKsf + kKsfSlots * F::kAtoms * 2048;  // 2 x kAtoms x 512
  static constexpr uint32_t kBars = kQsf + 2 * F::kAtoms * 512;
  static constexpr int kNumBars = 2 * kStages + 2 * kAccBufs + 6 + kKsfSlots;
  static constexpr uint32_t kState = kBars + kNumBars * 8;
  static constexpr uint32_t kScan = (kState + sizeof(BlockCta) + 15) / 16 * 16;
  static constexpr uint32_t kEnd = kScan + kThreads / 32 * 4;
  static constexpr uint32_t bytes() { return kEnd + 1024; }  // + alignment slack
  // TMEM columns
  static constexpr uint32_t kAccCol = 0;                      // kAccBufs x 128
  static constexpr uint32_t kQsfCol = 128 * kAccBufs;         // 2 item slots x 8
  static constexpr uint32_t kKsfCol = kQsfCol + 16;           // kKsfSlots x 8
  static_assert(kKsfCol + 8 * kKsfSlots <= kTmemCols, "TMEM columns");
};

// ---------------------------------------------------------------------------
// Items: i = (b * Hkv + hk) * row_tiles + rt.
// ---------------------------------------------------------------------------
struct BlockItem {
  int32_t b, hk, q0, q_len, row0, nrows, k_len, maxvis, tiles;
  int64_t table_base;
};

__device__ __forceinline__ int32_t clamp_vis(int64_t v, int32_t k_len) {
  return static_cast<int32_t>(v < 0 ? 0 : (v > k_len ? k_len : v));
}

// Visible key count of row t of the item (rule of the public header).
__device__ __forceinline__ int32_t row_vis(const BlockParams& p, const BlockItem& it, int32_t t) {
  if (p.visible_len) return clamp_vis(__ldg(p.visible_len + t), it.k_len);
  if (p.causal) {
    const int64_t off = p.qo_offset ? static_cast<int64_t>(__ldg(p.qo_offset + it.b))
                                    : static_cast<int64_t>(it.k_len) - it.q_len;
    return clamp_vis(static_cast<int64_t>(t - it.q0) + off + 1, it.k_len);
  }
  return it.k_len;
}

__device__ BlockItem block_item(const BlockParams& p, int32_t i) {
  BlockItem it;
  const int per_seq = p.num_kv_heads * p.row_tiles;
  it.b = i / per_seq;
  const int rem = i - it.b * per_seq;
  it.hk = rem / p.row_tiles;
  const int rt = rem - it.hk * p.row_tiles;
  it.q0 = __ldg(p.cu_seqlens_q + it.b);
  it.q_len = __ldg(p.cu_seqlens_q + it.b + 1) - it.q0;
  it.row0 = it.q0 + (rt << p.rt_shift);
  const int n = it.q_len - (rt << p.rt_shift);
  const int RT = 1 << p.rt_shift;
  it.nrows = n < 0 ? 0 : (n > RT ? RT : n);
  it.k_len = __ldg(p.cu_seqlens_k + it.b + 1) - __ldg(p.cu_seqlens_k + it.b);
  if (it.k_len < 0) it.k_len = 0;
  it.table_base = p.page_offsets ? static_cast<int64_t>(__ldg(p.page_offsets + it.b))
                                 : static_cast<int64_t>(it.b) * p.table_stride;
  // Largest visible count over the item's rows: the last row for the causal
  // rule (visibility grows with the row), every row for explicit lengths.
  it.maxvis = 0;
  if (it.nrows > 0) {
    if (p.visible_len) {
      for (int r = 0; r < it.nrows; ++r) it.maxvis = max(it.maxvis, row_vis(p, it, it.row0 + r));
    } else {
      it.maxvis = row_vis(p, it, it.row0 + it.nrows - 1);
    }
  }
  // At least one tile (computed or not) so that some CTA writes the item's -inf blocks.
  it.tiles = it.nrows > 0 ? max(1, (it.maxvis + kTileKeys - 1) / kTileKeys) : 0;
  return it;
}

__device__ __forceinline__ bool tile_computed(const BlockItem& it, int j) {
  return j * kTileKeys < it.maxvis;
}

// Cooperative over kThreads threads: total tiles, this CTA's equal chunk of
// them and the item holding the chunk's first tile (item0 = -1 when the CTA
// has no tiles).
__device__ void block_plan(const BlockParams& p, int tid, uint32_t* ws, BlockCta* st) {
  const int items = p.num_seqs * p.num_kv_heads * p.row_tiles;
  const int per = (items + kThreads - 1) / kThreads;
  const int i0 = tid * per, i1 = min(items, i0 + per);
  int32_t s = 0;
  for (int i = i0; i < i1; ++i) s += block_item(p, i).tiles;
  if (tid == 0) st->item0 = -1;  // ordered before the writes below by the scan's barriers
  uint32_t total_u;
  const int32_t pre = static_cast<int32_t>(cta_excl_prefix<kThreads>(static_cast<uint32_t>(s), ws, &total_u));
  const int32_t total = static_cast<int32_t>(total_u);
  const int32_t chunk = (total + static_cast<int32_t>(gridDim.x) - 1) / static_cast<int32_t>(gridDim.x);
  const int64_t x = static_cast<int64_t>(blockIdx.x) * chunk;
  if (tid == 0) {
    st->total_tiles = total;
    st->chunk = chunk;
  }
  if (x < total && pre <= x && x < pre + s) {
    int32_t acc = pre;
    for (int i = i0; i < i1; ++i) {
      const int32_t ti = block_item(p, i).tiles;
      if (x < acc + ti) {
        st->item0 = i;
        st->item0_start = acc;
        break;
      }
      acc += ti;
    }
  }
  __syncthreads();
}

// Visit the (item, tile range) segments of this CTA's chunk in order.
template <class Fn>
__device__ __forceinline__ void block_segments(const BlockParams& p, const BlockCta* st, Fn&& f) {
  const int items = p.num_seqs * p.num_kv_heads * p.row_tiles;
  int64_t x = static_cast<int64_t>(blockIdx.x) * st->chunk;
  const int64_t end = min(static_cast<int64_t>(st->total_tiles), x + st->chunk);
  if (x >= end || st->item0 < 0) return;
  int32_t i = st->item0;
  int64_t start = st->item0_start;
  while (x < end && i < items) {
    const BlockItem it = block_item(p, i);
    const int64_t lo = x - start;
    const int64_t hi = min(end, start + it.tiles) - start;
    if (hi > lo) {
      f(i, it, static_cast<int>(lo), static_cast<int>(hi));
      x = start + hi;
    }
    start += it.tiles;
    ++i;
  }
}

__device__ __forceinline__ float max2n(float a, float b) {
  float d;
  asm("max.NaN.f32 %0, %1, %2;" : "=f"(d) : "f"(a), "f"(b));
  return d;
}
__device__ __forceinline__ float max3n(float a, float b, float c) {
  float d;
  asm("max.NaN.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// Fold 64 columns into four running maxima (three-input max, four chains).
__device__ __forceinline__ void block_max_accum(const uint32_t (&v)[64], float (&m)[4]) {
#pragma unroll
  for (int i = 0; i < 64; i += 8) {
#pragma unroll
    for (int c = 0; c < 4; ++c) m[c] = max3n(m[c], __uint_as_float(v[i + 2 * c]), __uint_as_float(v[i + 2 * c + 1]));
  }
}

// Same over the columns i of this half with (i - off) in [0, span): off is
// the first visible column relative to the half.  Masked columns are
// replaced by -inf by selection, so whatever they hold never reaches the max.
__device__ __forceinline__ void block_max_accum_range(const uint32_t (&v)[64], int off, int span, float (&m)[4]) {
  const uint32_t n = span > 0 ? static_cast<uint32_t>(span) : 0u;
#pragma unroll
  for (int i = 0; i < 64; i += 8) {
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const int i0 = i + 2 * c, i1 = i0 + 1;
      const float a = static_cast<uint32_t>(i0 - off) < n ? __uint_as_float(v[i0]) : -INFINITY;
      const float b = static_cast<uint32_t>(i1 - off) < n ? __uint_as_float(v[i1]) : -INFINITY;
      m[c] = max3n(m[c], a, b);
    }
  }
}

template <int FMT>
__global__ void __launch_bounds__(kThreads, 1) block_score_kernel(const __grid_constant__ BlockParams p) {
  using L = BlockLayout<FMT>;
  using F = FmtTraits<FMT>;
  constexpr int G = F::G;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  const uint32_t bar0 = smem_u32(smem + L::kBars);
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (kStages + s); };
  auto accf_bar = [&](int a) { return bar0 + 8u * (2 * kStages + a); };
  auto acce_bar = [&](int a) { return bar0 + 8u * (2 * kStages + kAccBufs + a); };
  auto qfull_bar = [&](uint32_t qb) { return bar0 + 8u * (2 * kStages + 2 * kAccBufs + qb); };
  auto qempty_bar = [&](uint32_t qb) { return bar0 + 8u * (2 * kStages + 2 * kAccBufs + 2 + qb); };
  auto sfready_bar = [&](int slot) { return bar0 + 8u * (2 * kStages + 2 * kAccBufs + 4 + slot); };
  // Q scales of item slot qb in TMEM (committed by scale warp 2)
  auto qsf_bar = [&](uint32_t qb) { return bar0 + 8u * (2 * kStages + 2 * kAccBufs + 4 + kKsfSlots + qb); };

  BlockCta* st = reinterpret_cast<BlockCta*>(smem + L::kState);
  uint32_t* scan = reinterpret_cast<uint32_t*>(smem + L::kScan);
  volatile int* abort_flag = &st->abort;

  // ---- this CTA's chunk of the concatenated tile space
  if (threadIdx.x == 0) {
    st->abort = 0;
    // the first TMA waits for its descriptor: fetch both while the CTA plans
    prefetch_tmap(&p.tmap_k);
    prefetch_tmap(&p.tmap_q);
  }
  block_plan(p, threadIdx.x, scan, st);
  if (st->item0 < 0) return;  // uniform: no work for this CTA

  // ---- one-time setup
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(full_bar(s), 1);  // the producer's expect-tx arrive; TMA and bulk copies complete the bytes
      mbar_init(empty_bar(s), 1);
    }
    for (int a = 0; a < kAccBufs; ++a) {
      mbar_init(accf_bar(a), 1);
      mbar_init(acce_bar(a), 4);  // one arrive per warp of the group that owns the tile
    }
    for (uint32_t qb = 0; qb < 2; ++qb) {
      mbar_init(qfull_bar(qb), 1 + 32);
      // freed by the MMA thread's commit (its MMAs read Q) and the scale
      // warp's arrive (it has seen this load), so a buffer is never reloaded
      // before both consumers observed the previous load's phase
      mbar_init(qempty_bar(qb), 2);
    }
    for (int sl = 0; sl < kKsfSlots; ++sl) mbar_init(sfready_bar(sl), 1);
    for (uint32_t qb = 0; qb < 2; ++qb) mbar_init(qsf_bar(qb), 1);
    fence_barrier_init();
  }
  if (warp == 1) tmem_alloc<kTmemCols>(smem_u32(&st->tmem_base));
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = st->tmem_base;

  const uint32_t codes_s = smem_u32(smem + L::kCodes);
  const uint32_t q_s = smem_u32(smem + L::kQ);
  const uint32_t kraw_s = smem_u32(smem + L::kKraw);
  const uint8_t* kraw = smem + L::kKraw;
  uint8_t* ksf_rows = smem + L::kKsf;
  uint8_t* qsf_atoms = smem + L::kQsf;
  const int pshift = p.page_shift;
  const int page = p.page_size;
  const int slots = kTileKeys >> pshift;  // pages per tile: 2 (64-key pages) or 1 (128)
  const int rt_shift = p.rt_shift;

  if (warp == 0 || warp == 4) {
    // ================================================================ producers
    // Two warps take alternate tiles (each tile's barrier wait, expect_tx and
    // copies are a serial chain of ~500 cycles in one warp); warp 0 also
    // loads each item's Q.
    const uint32_t pidx = warp == 0 ? 0u : 1u;
    uint32_t tile_iter = 0, item_iter = 0;
    bool ok = true;
    block_segments(p, st, [&](int, const BlockItem& it, int lo, int hi) {
      if (!ok) return;
      // -- Q of the item: codes by TMA, scales by cp.async into the atom
      if (pidx == 0) {
      const uint32_t qb = item_iter & 1u, qph = (item_iter >> 1) & 1u;
      ok = warp_wait(qempty_bar(qb), qph ^ 1u, abort_flag, p.err);
      if (!ok) return;
      if (lane == 0) {
        mbar_arrive_expect_tx(qfull_bar(qb), 128 * kCodeBytes);
        tma_load_3d(q_s + qb * 8192u, &p.tmap_q, 0, it.row0, it.hk << p.group_shift, qfull_bar(qb));
      }
      {
        uint8_t* atom = qsf_atoms + qb * F::kAtoms * 512 + lane * 16;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int m = 32 * q + lane;
          const int t_local = m & ((1 << rt_shift) - 1);
          const int h = (it.hk << p.group_shift) + (m >> rt_shift);
          // rows past the item's last row read row0's scales (results discarded)
          const int64_t t = it.row0 + (t_local < it.nrows ? t_local : 0);
          const uint8_t* src = p.q_scale + t * p.q_scale_row_stride + h * G;
          cp_async_4(smem_u32(atom + 4 * q), src);
          if constexpr (G == 8) cp_async_4(smem_u32(atom + 512 + 4 * q), src + 4);
        }
        cp_async_arrive(qfull_bar(qb));
      }
      ++item_iter;
      }
      // -- K tiles: lane l caches the physical id of logical page base + l
      const int32_t npages = (it.k_len + page - 1) >> pshift;
      const int32_t* table = p.block_table + it.table_base;
      auto fetch = [&](int32_t b) -> int32_t {
        const int32_t lp = b + lane;
        return lp < npages ? __ldg(table + lp) : -1;
      };
      int32_t base = (lo * slots) & ~31;
      int32_t cur_ids = fetch(base), next_ids = fetch(base + 32);
      for (int j = lo; j < hi; ++j) {
        if (!tile_computed(it, j)) continue;
        const int32_t lp0 = j * slots;
        if (lp0 >= base + 32) {  // warp-uniform
          base += 32;
          cur_ids = next_ids;
          next_ids = fetch(base + 32);
        }
        if ((tile_iter & 1u) != pidx) {  // the other producer's tile
          ++tile_iter;
          continue;
        }
        const int32_t phys0 = __shfl_sync(0xffffffffu, cur_ids, lp0 - base);
        const int32_t phys1 = __shfl_sync(0xffffffffu, cur_ids, lp0 - base + (slots - 1));
        auto page_ok = [&](int sl, int32_t ph_id) {
          return ((lp0 + sl) << pshift) < it.k_len && ph_id >= 0 && ph_id < p.num_pages;
        };
        const bool ok0 = page_ok(0, phys0);
        const bool ok1 = slots == 2 && page_ok(1, phys1);
        if (lane < slots && ((lp0 + lane) << pshift) < it.k_len && !(lane == 0 ? ok0 : ok1))
          atomicOr(p.err, kErrPageRange);
        // (page, K head) blocks of the two slots (< 2^31 for resolved pages: checked on the host)
        const int32_t row0k = ok0 ? static_cast<int32_t>(static_cast<int64_t>(phys0) * p.num_kv_heads + it.hk) : 0;
        const int32_t row1k = ok1 ? static_cast<int32_t>(static_cast<int64_t>(phys1) * p.num_kv_heads + it.hk) : 0;
        const uint32_t bytes = static_cast<uint32_t>((ok0 ? 1 : 0) + (ok1 ? 1 : 0)) * page * (kCodeBytes + G);
        const int s = tile_iter % kStages;
        const uint32_t ph = (tile_iter / kStages) & 1u;
        ok = warp_wait(empty_bar(s), ph ^ 1u, abort_flag, p.err);
        if (!ok) return;
        if (lane == 0) mbar_arrive_expect_tx(full_bar(s), bytes);
        __syncwarp();
        if (lane < slots && (lane == 0 ? ok0 : ok1)) {
          const int32_t blk = lane == 0 ? row0k : row1k;
          tma_load_3d(codes_s + s * 8192 + ((lane * kCodeBytes) << pshift), &p.tmap_k, 0, 0, blk, full_bar(s));
          // the page's scales are contiguous: [page keys][G]
          bulk_load(kraw_s + s * (128 * G) + ((lane * G) << pshift),
                    p.kscale_base + static_cast<int64_t>(blk) * p.kscale_block_stride, static_cast<uint32_t>(page * G),
                    full_bar(s));
        }
        ++tile_iter;
      }
    });
    if (!ok && lane == 0) {
      // Let copies already in flight land before the CTA can exit.
      volatile int never = 0;
      const uint32_t first = tile_iter > static_cast<uint32_t>(kStages) ? tile_iter - kStages : 0;
      for (uint32_t u = first; u < tile_iter; ++u)
        if ((u & 1u) == pidx) mbar_wait(full_bar(u % kStages), (u / kStages) & 1u, &never, p.err);
      for (uint32_t u = item_iter > 2u ? item_iter - 2u : 0u; u < item_iter; ++u)
        mbar_wait(qfull_bar(u & 1u), (u >> 1) & 1u, &never, p.err);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ================================================================ MMA issuer
    // One thread does nothing but wait and issue: an MMA issue holds the
    // issuing thread for most of the MMA's duration, so any other per-tile
    // work here would leave the tensor pipe idle.
    if (lane == 0) {
      const uint64_t q_desc0 = desc_kmajor_sw64(q_s);
      const uint64_t k_desc0 = desc_kmajor_sw64(codes_s);
      uint32_t tile_iter = 0, item_iter = 0;
      int acc_sel = 0;           // tile_iter % kAccBufs
      uint32_t acc_phase = 0;    // bit a: phase of accumulator a's next use
      uint32_t sf_phase = 0;     // bit slot: phase of the scale slot's next use
      uint32_t qsf_phase = 0;    // bit qb: phase of the Q-scale slot's next use
      bool ok = true;
      int last_acc = -1;
      uint32_t last_acc_phase = 0;
      block_segments(p, st, [&](int, const BlockItem& it, int lo, int hi) {
        if (!ok) return;
        const uint32_t qb = item_iter & 1u;
        const uint32_t qsf_t = tmem + L::kQsfCol + qb * 8u;
        const uint64_t adesc = q_desc0 + static_cast<uint64_t>((qb * 8192u) >> 4);
        // the item's Q scales (copied by scale warp 2 when the segment computes a tile)
        if (tile_computed(it, lo)) {
          if (!(ok = mbar_wait(qsf_bar(qb), (qsf_phase >> qb) & 1u, abort_flag, p.err))) return;
          qsf_phase ^= 1u << qb;
        }
        // Tiles go to the tensor pipe in pairs with their K halves interleaved
        // (A0 B0 A1 B1): back-to-back dependent MMAs on one accumulator stall
        // the pipe, two independent chains keep it busy (measured: ~226
        // instead of ~565 cycles per tile).  Computed tiles are a prefix of
        // the segment.
        const int jend = min(hi, (it.maxvis + kTileKeys - 1) / kTileKeys);
        for (int j = lo; j < jend && ok; j += 2) {
          const int n = min(2, jend - j);
          int sg[2], slot[2], a[2];
          uint32_t aph[2];
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            const uint32_t ti = tile_iter + u;
            sg[u] = ti % kStages;
            slot[u] = ti % kKsfSlots;
            a[u] = u == 0 ? acc_sel : (acc_sel == kAccBufs - 1 ? 0 : acc_sel + 1);
            aph[u] = (acc_phase >> a[u]) & 1u;
          }
          // scale slot ready implies the stage's codes landed (the scale warp waited for them)
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            if (u >= n || !ok) continue;
            ok = mbar_wait(sfready_bar(slot[u]), (sf_phase >> slot[u]) & 1u, abort_flag, p.err);
            sf_phase ^= 1u << slot[u];
          }
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            if (u >= n || !ok) continue;
            ok = mbar_wait(acce_bar(a[u]), aph[u] ^ 1u, abort_flag, p.err);
          }
          if (!ok) break;
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < 2; ++kk) {
            constexpr uint32_t sf1 = F::kScaleVec == 2 ? 2u : 0u;
            const uint32_t idesc =
                kk == 0 ? idesc_fp4(128, 128, F::kUe8m0, 0, 0) : idesc_fp4(128, 128, F::kUe8m0, sf1, sf1);
            const uint32_t col = F::kScaleVec == 2 ? 0u : 4u * kk;
#pragma unroll
            for (int u = 0; u < 2; ++u) {
              if (u >= n) continue;
              const uint32_t ksf_t = tmem + L::kKsfCol + slot[u] * 8u;
              const uint32_t d = tmem + L::kAccCol + a[u] * 128u;
              const uint64_t bdesc = k_desc0 + static_cast<uint64_t>((sg[u] * 8192) >> 4);
              tc_mma_fp4<F::kScaleVec>(d, adesc + 2u * kk, bdesc + 2u * kk, idesc, qsf_t + col, ksf_t + col,
                                       static_cast<uint32_t>(kk));
            }
          }
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            if (u >= n) continue;
            tc_commit(empty_bar(sg[u]));
            tc_commit(accf_bar(a[u]));
            last_acc = a[u];
            last_acc_phase = aph[u];
            acc_phase ^= 1u << a[u];
            acc_sel = a[u] == kAccBufs - 1 ? 0 : a[u] + 1;
          }
          tile_iter += n;
        }
        if (!ok) return;
        // Q buffer and Q-scale slot free once this item's MMAs complete.
        tc_commit(qempty_bar(qb));
        ++item_iter;
      });
      if (!ok && last_acc >= 0) {
        // Outstanding MMAs must finish before TMEM is released.
        volatile int never = 0;
        mbar_wait(accf_bar(last_acc), last_acc_phase, &never, p.err);
      }
    }
    __syncwarp();
  } else if (warp == 2 || warp == 3) {
    // ================================================================ scale warps
    // Per item: Q scales (atoms written by the producer's cp.async) -> TMEM.
    // Per tile: raw K scales [128 keys][G] -> 128 rows of the scale layout
    // (row r holds the 32x4x4 atom line r % 32: the words of keys l, 32+l,
    // 64+l, 96+l, l = r % 32; NVFP4's K half 1 in the second 16 bytes), one
    // tcgen05.cp into TMEM slot tile % kKsfSlots, committed to that slot's
    // barrier.  The slot (TMEM and shared staging) is reused by tile
    // i + kKsfSlots only after the MMA of tile i completed (its stage's
    // empty barrier), which also completes the copy that read the staging.
    // Two warps take alternate tiles; warp 2 also copies each item's Q scales.
    const uint32_t sidx = warp == 2 ? 0u : 1u;
    const uint64_t ksf_desc0 = desc_sf_rows(smem_u32(ksf_rows));
    const uint64_t qsf_desc0 = desc_sf_atom(smem_u32(qsf_atoms));
    uint32_t tile_iter = 0, item_iter = 0;
    bool ok = true;
    block_segments(p, st, [&](int, const BlockItem& it, int lo, int hi) {
      if (!ok) return;
      const uint32_t qb = item_iter & 1u, qph = (item_iter >> 1) & 1u;
      if (sidx == 0) {
      ok = warp_wait(qfull_bar(qb), qph, abort_flag, p.err);
      if (!ok) return;
      if (lane == 0) {
        // Q scales were written by cp.async (generic proxy): make them
        // visible to the tensor core's copy.  The previous user of this Q
        // slot (item - 2) finished: the producer waited for it (qempty)
        // before loading this item's Q.  Copied only when some tile of the
        // segment is computed (otherwise no MMA reads them, and no barrier
        // would track the copy).
        if (tile_computed(it, lo)) {
          fence_proxy_async_smem();
          tc_fence_after();
          const uint32_t qsf_t = tmem + L::kQsfCol + qb * 8u;
#pragma unroll
          for (int at = 0; at < F::kAtoms; ++at)
            tc_cp_32x128b_warpx4(qsf_t + 4u * at, qsf_desc0 + static_cast<uint64_t>(((qb * F::kAtoms + at) * 512) >> 4));
          tc_commit(qsf_bar(qb));
        }
        mbar_arrive(qempty_bar(qb));
      }
      __syncwarp();
      }
      for (int j = lo; j < hi; ++j) {
        if (!tile_computed(it, j)) continue;
        if ((tile_iter & 1u) != sidx) {  // the other scale warp's tile
          ++tile_iter;
          continue;
        }
        const int s = tile_iter % kStages;
        const uint32_t ph = (tile_iter / kStages) & 1u;
        const int slot = tile_iter % kKsfSlots;
        bool got = false;
        if (lane == 0) {
          got = mbar_wait(full_bar(s), ph, abort_flag, p.err);
          if (got && tile_iter >= static_cast<uint32_t>(kKsfSlots)) {
            const uint32_t u = tile_iter - kKsfSlots;  // previous user of the slot
            got = mbar_wait(empty_bar(u % kStages), (u / kStages) & 1u, abort_flag, p.err);
          }
        }
        ok = __shfl_sync(0xffffffffu, got, 0);
        if (!ok) break;
        {
          const uint8_t* raw = kraw + s * (128 * G);
          uint8_t* rows = ksf_rows + slot * (F::kAtoms * 2048);
          if constexpr (G == 4) {
            const uint32_t* r32 = reinterpret_cast<const uint32_t*>(raw);
            const uint4 v = make_uint4(r32[lane], r32[32 + lane], r32[64 + lane], r32[96 + lane]);
#pragma unroll
            for (int q = 0; q < 4; ++q) *reinterpret_cast<uint4*>(rows + (32 * q + lane) * 16) = v;
          } else {
            const uint2* r64 = reinterpret_cast<const uint2*>(raw);
            const uint2 a0 = r64[lane], a1 = r64[32 + lane], a2 = r64[64 + lane], a3 = r64[96 + lane];
            const uint4 lo4 = make_uint4(a0.x, a1.x, a2.x, a3.x), hi4 = make_uint4(a0.y, a1.y, a2.y, a3.y);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              *reinterpret_cast<uint4*>(rows + (32 * q + lane) * 16) = lo4;
              *reinterpret_cast<uint4*>(rows + 2048 + (32 * q + lane) * 16) = hi4;
            }
          }
          fence_proxy_async_smem();
        }
        __syncwarp();
        if (lane == 0) {
          tc_fence_after();
          const uint32_t ksf_t = tmem + L::kKsfCol + slot * 8u;
          const uint64_t sdesc = ksf_desc0 + static_cast<uint64_t>((slot * F::kAtoms * 2048) >> 4);
          if constexpr (G == 4) tc_cp_128x128b(ksf_t, sdesc);
          else tc_cp_128x256b(ksf_t, sdesc);
          tc_commit(sfready_bar(slot));
        }
        __syncwarp();
        ++tile_iter;
      }
      ++item_iter;
    });
    if (lane == 0) {
      // copies still in flight must land before TMEM is released
      volatile int never = 0;
      const uint32_t first = tile_iter > static_cast<uint32_t>(kKsfSlots) ? tile_iter - kKsfSlots : 0;
      for (uint32_t u = first; u < tile_iter; ++u)
        if ((u & 1u) == sidx) mbar_wait(sfready_bar(u % kKsfSlots), (u / kKsfSlots) & 1u, &never, p.err);
    }
    __syncwarp();
  } else {
    // ================================================================ epilogue
    const int e = (warp - kEpiWarp0) >> 2;  // group e owns accumulator e: tiles with tile_iter % kAccBufs == e
    Group<128, -1> g{static_cast<int>(threadIdx.x) - 32 * kEpiWarp0 - e * 128, 1 + e};
    const int quad = warp & 3;
    const int m = quad * 32 + lane;  // TMEM lane = MMA row
    const int h_local = m >> rt_shift;
    const int t_local = m & ((1 << rt_shift) - 1);
    int sel = 0;              // tile_iter % kAccBufs, kept incrementally
    uint32_t own_phase = 0;   // phase of accumulator e for this group's next tile
    bool ok = true;
    const int64_t T = p.num_rows;
    const uint32_t taddr = tmem + (static_cast<uint32_t>(quad * 32) << 16) + L::kAccCol + e * 128u;
    block_segments(p, st, [&](int, const BlockItem& it, int lo, int hi) {
      const int32_t t = it.row0 + t_local;
      const bool row_valid = t_local < it.nrows && t < p.num_rows;
      const int h = (it.hk << p.group_shift) + h_local;
      const int32_t vis = row_valid ? row_vis(p, it, t) : 0;
      float* out = p.scores + static_cast<int64_t>(h) * p.ktiles * T + t;  // + kb * T
      const int nreal = (it.maxvis + kTileKeys - 1) / kTileKeys;
      for (int j = lo; j < hi; ++j) {
        bool owner;
        if (tile_computed(it, j)) {
          owner = sel == e;
          if (owner) {
            // page ids of the tile, loaded while the accumulator is awaited
            const int32_t lp0 = j * slots;
            int32_t ph_id[2] = {0, 0};
            for (int sl = 0; sl < slots; ++sl)
              if (((lp0 + sl) << pshift) < it.k_len) ph_id[sl] = __ldg(p.block_table + it.table_base + lp0 + sl);
            if (g.tid == 0 && ok && !mbar_wait(accf_bar(e), own_phase, abort_flag, p.err)) st->abort = 1;
            own_phase ^= 1u;
            g.sync();
            // warp-uniform: tcgen05.ld below is a whole-warp instruction
            ok = __all_sync(0xffffffffu, ok && !*abort_flag);
            if (ok) {
              // columns [lo_c, hi_c) are visible keys of this row in pages that resolved
              int lo_c = 0;
              int hi_c = vis - j * kTileKeys;
              hi_c = hi_c < 0 ? 0 : (hi_c > kTileKeys ? kTileKeys : hi_c);
              for (int sl = 0; sl < slots; ++sl) {
                if (((lp0 + sl) << pshift) >= it.k_len) break;
                if (ph_id[sl] < 0 || ph_id[sl] >= p.num_pages) {
                  if (sl == 0) lo_c = page;  // 64-key pages: the second half may still count
                  else hi_c = min(hi_c, page);
                  if (slots == 1) hi_c = 0;
                }
              }
              const bool full = __all_sync(0xffffffffu, lo_c == 0 && hi_c == kTileKeys);
              tc_fence_after();
              // two halves of 64 columns keep the live registers low; the
              // accumulator is released after the second half is loaded
              float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
              for (int half = 0; half < 2; ++half) {
                uint32_t v[64];
                tmem_ld_x32(taddr + 64 * half, *reinterpret_cast<uint32_t(*)[32]>(&v[0]));
                tmem_ld_x32(taddr + 64 * half + 32, *reinterpret_cast<uint32_t(*)[32]>(&v[32]));
                tmem_wait_ld();
                reg_fence(v);
                if (half == 1) {
                  // every lane's loads completed (wait::ld); one arrive per warp
                  tc_fence_before();
                  __syncwarp();
                  if (lane == 0) mbar_arrive(acce_bar(e));
                }
                if (full) block_max_accum(v, mx);
                else block_max_accum_range(v, lo_c - 64 * half, hi_c - lo_c, mx);
              }
              const float r = max2n(max2n(mx[0], mx[1]), max2n(mx[2], mx[3]));
              if (row_valid && j < p.ktiles) out[static_cast<int64_t>(j) * T] = r;
            }
          }
          sel = sel == kAccBufs - 1 ? 0 : sel + 1;
        } else {
          owner = e == 0;  // a tile nothing is computed for: group 0 writes its -inf
        }
        if (j == it.tiles - 1 && owner && row_valid) {
          for (int kb = nreal; kb < p.ktiles; ++kb) out[static_cast<int64_t>(kb) * T] = -INFINITY;
        }
      }
    });
  }

  // ---- teardown
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc<kTmemCols>(tmem);
  }
}

template <int FMT>
cudaError_t launch_fmt(const BlockParams& p, dim3 grid, cudaStream_t stream) {
  using L = BlockLayout<FMT>;
  // At least ~120 KB so that one CTA (and one 512-column TMEM allocation) runs per SM.
  const uint32_t bytes = L::bytes() < 120u * 1024u ? 120u * 1024u : L::bytes();
  if (bytes > 232448u) return cudaErrorInvalidConfiguration;
  auto kern = block_score_kernel<FMT>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes));
  if (e != cudaSuccess) return e;
  kern<<<grid, kThreads, bytes, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_block_scores(const BlockParams& p, int format, dim3 grid, cudaStream_t stream) {
  return format == 0 ? launch_fmt<0>(p, grid, stream) : launch_fmt<1>(p, grid, stream);
}

}  // namespace fp4idx
