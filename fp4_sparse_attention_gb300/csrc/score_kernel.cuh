// score_kernel.cuh -- keys-on-M FP4 indexer scorer for sm_103a.
//
// logit(t, s) = sum_h w[t,h] * max(q[t,h] . k[s], 0)  (CURRENT_ISSUE...,
// "TL;DR"), evaluated as one tcgen05 block-scaled FP4 MMA per 128-key tile:
//
//   D[key, r*H + h] = sum_d K_real[key, d] * Q_real[row r, head h, d]
//
// with the 128 keys of a tile on the MMA M dimension (TMEM lanes) and the
// R rows x H heads of one request on N (TMEM columns).  The head sum then is
// a serial loop inside one thread: thread = key, no shuffles.
//
// Warp roles (128 + 128 * groups threads):
//   warp 0 and the last warp: producers, each owning alternate tiles:
//             resolve pages through the block table, issue the TMA gather of
//             K codes (64-byte swizzle) and one bulk copy of each page's raw
//             scales into a kStages-deep shared-memory ring; warp 0 also
//             loads Q per item (double buffered).
//   warp 1    MMA: owns the TMEM allocation; one thread waits for a tile's
//             scales and a free accumulator and issues two K=64 MMAs into a
//             triple-buffered fp32 accumulator, nothing else (an MMA issue
//             holds its thread, so other work there idles the tensor pipe).
//   warp 2    scales: Q scales -> 32x4x4 atoms -> TMEM per item; per tile
//             the raw K scales -> 128-row scale layout -> one tcgen05.cp.
//   warps 3.. epilogue, groups of four warps (one per TMEM lane quadrant):
//             one query row per group for top-k, several rows per group for
//             logits; tcgen05.ld of the rows' H accumulator columns, ReLU * w
//             summed over heads (packed fp32x2 FMAs, four independent
//             chains), visibility mask, then either the fp32 logits store or
//             the streaming top-k append (candidate buffers in shared memory
//             for two-row CTAs, in the workspace for four-row ones).  Each
//             group synchronises on its own named barrier, only every few
//             tiles, so one row's candidate compaction never stalls another.
//
// The barrier initialisation and TMEM allocation come before any global
// access, so under programmatic stream serialisation they overlap the
// previous kernel; griddepcontrol.wait then orders the rest after it.
//
// Work split: the tiles of all (request, row-group) items are concatenated
// and cut into gridDim.x equal contiguous chunks, one per CTA, so long and
// short requests balance across the GPU.  A CTA that crosses an item
// boundary reloads Q and, for top-k, flushes its per-row candidates.
#pragma once

#include <cstring>

#include "formats.cuh"
#include "internal.h"
#include "ptx.cuh"
#include "topk_smem.cuh"

namespace fp4idx {

constexpr int kEpiThreads = 128;  // one epilogue group: four warps, one per TMEM lane quadrant

// Time attribution for profiling builds (-DFP4IDX_STAMPS only; product
// builds compile none of it): every warp of a role attributes the clock64
// cycles since its previous stamp to one category of its role; the sums are
// added to fp4idx_stamps[role][category] at the end of the kernel (category
// 7 counts tiles).  Roles: 0 producers, 1 MMA thread, 2 scale warp,
// 3 epilogue warps.
#ifdef FP4IDX_STAMPS
constexpr int kStampCats = 8;
static __device__ unsigned long long fp4idx_stamps[4 * kStampCats];
#define FP4IDX_STAMP_INIT() \
  unsigned long long stamp_acc_[kStampCats] = {}; \
  long long stamp_t_ = clock64()
#define FP4IDX_STAMP(c)                 \
  do {                                  \
    const long long n_ = clock64();     \
    stamp_acc_[c] += n_ - stamp_t_;     \
    stamp_t_ = n_;                      \
  } while (0)
#define FP4IDX_STAMP_COUNT() (stamp_acc_[7] += 1)
#define FP4IDX_STAMP_DONE(role)                                                      \
  do {                                                                               \
    if ((threadIdx.x & 31) == 0)                                                     \
      for (int c_ = 0; c_ < kStampCats; ++c_)                                        \
        atomicAdd(&fp4idx_stamps[(role) * kStampCats + c_], stamp_acc_[c_]);         \
  } while (0)
#else
#define FP4IDX_STAMP_INIT() do { } while (0)
#define FP4IDX_STAMP(c) do { } while (0)
#define FP4IDX_STAMP_COUNT() do { } while (0)
#define FP4IDX_STAMP_DONE(role) do { } while (0)
#endif
constexpr uint32_t kTmemCols = 512;
constexpr int kAccBufs = 3;  // accumulator buffers: the MMA may run two tiles ahead of the epilogue

// Per-CTA bookkeeping in shared memory.
struct CtaState {
  uint32_t tmem_base;
  int32_t abort;
  int32_t item0;        // item holding the first tile of this CTA's chunk
  int32_t item0_start;  // global tile index where item0 starts
  int32_t total_tiles;  // work units over all items (tiles, plus per-item units in top-k mode)
  int32_t chunk;        // tiles per CTA
  int32_t pad[2];
};

template <int R, int NREG>
struct RowState {  // top-k: candidates each epilogue warp appended to its region of each row
  int32_t wc[2][R][NREG];  // double buffered: publication p writes wc[p & 1]
};


template <int H, int R, int FMT, int MODE>
struct ScoreLayout {
  static constexpr int G = FmtTraits<FMT>::G;
  static constexpr int kAtoms = FmtTraits<FMT>::kAtoms;
  // MXFP4: the K tile's codes arrive in the strided key order (MMA row
  // m = 32c + l holds key 4l + c), so the tile's raw scale bytes -- 128
  // keys x 4 B, as the pages hold them -- already are the 32-line atom the
  // MMA reads (line l, word c = key 4l + c = row 32c + l).  The MMA thread
  // copies them into TMEM itself: no scale warp work per tile, no shared-
  // memory staging.  NVFP4's 8 scale bytes per key do not line up that way
  // and keep the scale warps' per-tile transposition.
  static constexpr bool kDirectSf = FMT == 0;
  // Top-k with two rows per CTA (64 heads): each row's candidate buffer
  // lives in shared memory (a compaction then reads and writes it at
  // shared-memory latency), kCandCap keys per row -- large, so that a row
  // rarely needs a compaction at all (about 3k insertions before the first).
  // With four rows the buffers would leave too shallow a K ring (measured:
  // long decode 286 -> 400 us with 3,072-key buffers and 8 stages), so they
  // stay in the workspace (L2) there.
  static constexpr bool kSmemCand = MODE == kModeTopk && R < 4;
  static constexpr int kCandCap = kSmemCand ? (FMT == 0 ? 8192 : 6144) : 0;
  static constexpr uint32_t kCandBytes = static_cast<uint32_t>(R) * kCandCap * 8;
  // Everything but the K ring, and the ring: as deep as shared memory allows
  // (a loaded HBM round trip for a random page is ~2 us, so ~70+ KB in
  // flight per SM), at most 20 stages.
  static constexpr uint32_t kFixedBytes = 2 * (((H * R * 64 + 1023) / 1024) * 1024) + (kDirectSf ? 0 : 4 * kAtoms * 2048) +
                                          2 * kAtoms * 512 + 4096 + (160 + kEpiThreads * 4) * 4 + 4 * 1280 +
                                          (MODE == kModeTopk ? R * kHistBins * 2 + R * H * 4 : 0) + kCandBytes + 2048;
  static constexpr int kStagesFit = static_cast<int>((232448u - 1024u - kFixedBytes) / (8192u + 128u * G)) & ~1;
  static constexpr int kStages = kStagesFit < 20 ? kStagesFit : 20;
  static_assert(kStages >= 4, "K ring depth");
  // Rows of the item per epilogue group of four warps.  Logits: 64
  // accumulator columns per thread and tile, so the per-tile fixed work
  // (barrier poll, TMEM load, fences) is shared by several rows.  Top-k: one
  // row per group, as each row's insert and compaction chain is serial
  // within its group and more groups overlap more of them.
  static constexpr int kRowsPerGroup =
      MODE == kModeTopk ? 1 : (R < 64 / H ? R : (64 / H < 1 ? 1 : 64 / H));
  static_assert(R % kRowsPerGroup == 0, "rows split evenly over the groups");
  static constexpr int kGroups = R / kRowsPerGroup;
  // Two-row top-k CTAs (64 heads) give each row two sets of four warps that
  // take alternate tiles (tile parity), so the per-tile epilogue chain of a
  // row runs on twice the warps; a row's checks, compactions and flush stay
  // cooperative over both sets (eight warps, eight append regions).
  static constexpr int kSets = MODE == kModeTopk && R == 2 ? 2 : 1;
  static constexpr int kEpiGroups = kGroups * kSets;
  static constexpr int kRegions = 4 * kSets;
  // warp 0 and kProducer2Warp: producers; warp 1: MMA; warp 2 (and
  // kScale2Warp, when there are two): scales (alternate tiles); warps 3 ..
  // 3 + 4 * kEpiGroups - 1: epilogue.  Registers are reserved for whole
  // groups of four warps, so the CTA is rounded up to a multiple of four
  // warps (the extra ones idle); a second scale warp is used where that
  // leaves the epilogue enough registers.
  static constexpr int kEpiWarp0 = 3;
  static constexpr int kProducer2Warp = kEpiWarp0 + 4 * kEpiGroups;
  static constexpr int kScaleWarps = kDirectSf || (kProducer2Warp + 1) % 4 == 0 ? 1 : 2;
  static constexpr int kScale2Warp = kProducer2Warp + 1;
  static constexpr int kWarpsUsed = kProducer2Warp + kScaleWarps;
  static constexpr int kThreads = ((kWarpsUsed + 3) / 4) * 4 * 32;
  // registers per thread with one CTA of kThreads on an SM (a multiple of 8)
  static constexpr int kMaxRegs = (65536 / kThreads) / 8 * 8 > 255 ? 255 : (65536 / kThreads) / 8 * 8;
  static_assert(kStages % 2 == 0, "the two producers own alternate stages");
  static constexpr int N = H * R;
  static_assert(N % 16 == 0 && N >= 16 && N <= 128, "MMA N");
  // K-scale slots (TMEM and shared staging): tile i uses slot i % kSfaSlots;
  // direct scales use the accumulator's index (the accumulator's release
  // then also frees the slot)
  static constexpr int kSfaSlots = kDirectSf ? kAccBufs : 4;
  static constexpr uint32_t kCodes = 0;                                  // kStages x 8 KB
  static constexpr uint32_t kQBytes = ((N * 64 + 1023) / 1024) * 1024;
  static constexpr uint32_t kQ = kCodes + kStages * 8192;                // 2 x N x 64 B (double buffered)
  static constexpr uint32_t kKraw = kQ + 2 * kQBytes;                    // kStages x 128 keys x G raw K scales
  static constexpr uint32_t kSfaRows = kKraw + kStages * 128 * G;        // kSfaSlots x kAtoms x 2048 (128 rows)
  static constexpr uint32_t kSfb = kSfaRows + (kDirectSf ? 0 : kSfaSlots * kAtoms * 2048); // 2 x kAtoms x 512 Q-scale atoms
  static constexpr uint32_t kBars = kSfb + 2 * kAtoms * 512;             // mbarriers
  static constexpr int kNumBars = 2 * kStages + 2 * kAccBufs + 4 + kSfaSlots + 2;
  static constexpr uint32_t kState = kBars + kNumBars * 8;
  static constexpr uint32_t kRows = (kState + sizeof(CtaState) + 15) / 16 * 16;
  static constexpr uint32_t kScan = (kRows + sizeof(RowState<R, kRegions>) + 15) / 16 * 16;  // kThreads ints
  static constexpr uint32_t kScratch = kScan + kThreads * 4;                      // per group
  static constexpr uint32_t kHist = (kScratch + kGroups * sizeof(SelectScratch) + 15) / 16 * 16;
  static constexpr uint32_t kCand = (kHist + (MODE == kModeTopk ? R * kHistBins * 2 : 0) + 15) / 16 * 16;
  // top-k: the item rows' head weights (the epilogue reads them from here,
  // not from registers, which the top-k state needs)
  static constexpr uint32_t kW = kCand + kCandBytes;
  static constexpr uint32_t kEnd = kW + (MODE == kModeTopk ? R * H * 4 : 0);
  static constexpr uint32_t bytes() { return kEnd + 1024; }
  static_assert(kEnd + 1024 <= 232448u, "shared memory");
  // TMEM columns
  static constexpr uint32_t kAccCol = 0;                  // kAccBufs accumulators of 128 columns
  static constexpr uint32_t kSfbCol = 128 * kAccBufs;     // two Q-scale slots of 8 columns
  static constexpr uint32_t kSfaCol = kSfbCol + 16;       // kSfaSlots K-scale slots of 8 columns
  static_assert(kSfaCol + 8 * kSfaSlots <= kTmemCols, "TMEM columns");
};

// ---------------------------------------------------------------------------
// Items: item i = (request b, row group g), i = b * row_groups + g.
// ---------------------------------------------------------------------------
struct ItemInfo {
  int32_t b, row0, nrows, k_len;
  int32_t maxvis;  // largest visible key count over the item's rows
  int64_t table_base;
};

// Visible key count of row t (rule of the public header).
__device__ __forceinline__ int32_t row_visible(const ScoreParams& p, const ItemInfo& it, int32_t t) {
  int64_t vis;
  if (p.visible_len) {
    vis = __ldg(p.visible_len + t);
  } else if (p.causal) {
    const int q0 = __ldg(p.cu_seqlens_q + it.b), q1 = __ldg(p.cu_seqlens_q + it.b + 1);
    const int64_t off = p.qo_offset ? static_cast<int64_t>(__ldg(p.qo_offset + it.b))
                                    : static_cast<int64_t>(it.k_len) - (q1 - q0);
    vis = static_cast<int64_t>(t - q0) + off + 1;
  } else {
    vis = it.k_len;
  }
  if (vis < 0) vis = 0;
  if (vis > it.k_len) vis = it.k_len;
  return static_cast<int32_t>(vis);
}

__device__ __forceinline__ ItemInfo item_info(const ScoreParams& p, int32_t i, int rows_per_cta) {
  ItemInfo it;
  it.b = i / p.row_groups;
  const int g = i - it.b * p.row_groups;
  const int q0 = __ldg(p.cu_seqlens_q + it.b), q1 = __ldg(p.cu_seqlens_q + it.b + 1);
  it.row0 = q0 + g * rows_per_cta;
  const int n = q1 - it.row0;
  it.nrows = n < 0 ? 0 : (n > rows_per_cta ? rows_per_cta : n);
  it.k_len = __ldg(p.cu_seqlens_k + it.b + 1) - __ldg(p.cu_seqlens_k + it.b);
  if (it.k_len < 0) it.k_len = 0;
  it.table_base = p.page_offsets ? static_cast<int64_t>(__ldg(p.page_offsets + it.b))
                                 : static_cast<int64_t>(it.b) * p.table_stride;
  // the causal rule grows with the row: its last row sees the most
  it.maxvis = 0;
  if (it.nrows > 0) {
    if (p.visible_len) {
      for (int r = 0; r < it.nrows; ++r) it.maxvis = max(it.maxvis, row_visible(p, it, it.row0 + r));
    } else {
      it.maxvis = row_visible(p, it, it.row0 + it.nrows - 1);
    }
  }
  return it;
}

// Tiles an item contributes to the concatenated work space: every output
// column for logits, the tiles holding some visible key for top-k.
template <int MODE>
__device__ __forceinline__ int32_t item_tiles(const ScoreParams& p, const ItemInfo& it) {
  if (it.nrows <= 0) return 0;
  if constexpr (MODE == kModeLogits) return p.total_tiles;
  return (it.maxvis + kTileKeys - 1) / kTileKeys;
}

// Units an item occupies in the concatenated work space: its tiles plus,
// when it has any, p.item_overhead units without a tile (its fixed cost).
template <int MODE>
__device__ __forceinline__ int32_t item_units(const ScoreParams& p, const ItemInfo& it) {
  const int32_t t = item_tiles<MODE>(p, it);
  return t > 0 ? t + p.item_overhead : 0;
}

// Whether tile j of the item holds a key some row of it can see; logits
// tiles past that are written as -inf without loading or computing.
__device__ __forceinline__ bool tile_has_visible(const ItemInfo& it, int j) {
  return static_cast<int64_t>(j) * kTileKeys < it.maxvis;
}

// Cooperative over kNT threads (tid in [0, kNT), all of the CTA): the total
// of the item units, this CTA's equal chunk of them and the item holding the
// chunk's first unit with that item's start (item0 = -1 when the CTA has no
// units).  `ws` holds kNT / 32 words.  With `starts` != nullptr the start of
// every item (and the total, at index items) is also written there, for the
// merge.
template <int MODE, int kNT>
__device__ void plan_items(const ScoreParams& p, int rows_per_cta, int tid, uint32_t* ws, CtaState* st,
                           int32_t* starts) {
  const int items = p.num_seqs * p.row_groups;
  const int per = (items + kNT - 1) / kNT;
  const int i0 = tid * per;
  const int i1 = min(items, i0 + per);
  int32_t s = 0;
  for (int i = i0; i < i1; ++i) s += item_units<MODE>(p, item_info(p, i, rows_per_cta));
  if (tid == 0) st->item0 = -1;  // ordered before the writes below by the scan's barriers
  uint32_t total_u;
  const int32_t pre = static_cast<int32_t>(cta_excl_prefix<kNT>(static_cast<uint32_t>(s), ws, &total_u));
  const int32_t total = static_cast<int32_t>(total_u);
  const int32_t chunk = (total + static_cast<int32_t>(gridDim.x) - 1) / static_cast<int32_t>(gridDim.x);
  const int64_t x = static_cast<int64_t>(blockIdx.x) * chunk;
  if (tid == 0) {
    st->total_tiles = total;
    st->chunk = chunk;
    if (starts) starts[items] = total;
  }
  if (starts) {
    int32_t acc = pre;
    for (int i = i0; i < i1; ++i) {
      starts[i] = acc;
      acc += item_units<MODE>(p, item_info(p, i, rows_per_cta));
    }
  }
  if (x < total && pre <= x && x < pre + s) {
    int32_t acc = pre;
    for (int i = i0; i < i1; ++i) {
      const int32_t ti = item_units<MODE>(p, item_info(p, i, rows_per_cta));
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

// Visit the (item, tile range) segments of this CTA's chunk in order:
// f(item, info, lo, hi, own) with tiles [lo, hi) of the item; own is true
// when the chunk starts at or after the item's first unit (the item is the
// chunk's first), false when the item starts inside the chunk.  The merge
// finds a CTA's partial list of an item by the same rule.
template <int MODE, int R, class F>
__device__ __forceinline__ void for_each_segment(const ScoreParams& p, const CtaState* st, F&& f) {
  const int items = p.num_seqs * p.row_groups;
  const int64_t x = static_cast<int64_t>(blockIdx.x) * st->chunk;
  const int64_t end = min(static_cast<int64_t>(st->total_tiles), x + st->chunk);
  if (x >= end || st->item0 < 0) return;
  int32_t i = st->item0;
  int64_t start = st->item0_start;
  while (start < end && i < items) {
    const ItemInfo it = item_info(p, i, R);
    const int32_t units = item_units<MODE>(p, it);
    const int64_t tiles = units > 0 ? units - p.item_overhead : 0;
    const int64_t lo = max(x - start, int64_t(0));
    const int64_t hi = min(end - start, tiles);
    if (hi > lo) f(i, it, static_cast<int>(lo), static_cast<int>(hi), x >= start);
    start += units;
    ++i;
  }
}

// ---------------------------------------------------------------------------
// Scale-factor atoms.  tcgen05 reads a block scale of MMA row m from TMEM
// lane m%32, column m/32; tcgen05.cp 32x128b.warpx4 fills 4 columns from a
// 512-byte atom whose 16-byte line l holds, for row groups j = 0..3, the
// four scale bytes of row 32j + l.
// ---------------------------------------------------------------------------
// Q scales of the item's rows (B row n = r*H + h) into the atom layout.
template <int H, int R, int FMT>
__device__ __forceinline__ void q_scale_atoms(const ScoreParams& p, const ItemInfo& it, uint8_t* atoms,
                                              int lane) {
  constexpr int N = H * R;
  constexpr int G = FmtTraits<FMT>::G;
  uint32_t lo[4], hi[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int n = 32 * j + lane;
    const int r = n / H, h = n % H;
    lo[j] = 0;
    hi[j] = 0;
    if (n < N && r < it.nrows) {
      const uint8_t* src = p.q_scale + static_cast<int64_t>(it.row0 + r) * p.q_scale_row_stride + h * G;
      if constexpr (FMT == 0) {
        lo[j] = __ldg(reinterpret_cast<const uint32_t*>(src));
      } else {
        const uint2 v = __ldg(reinterpret_cast<const uint2*>(src));
        lo[j] = v.x;
        hi[j] = v.y;
      }
    }
  }
  *reinterpret_cast<uint4*>(atoms + lane * 16) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
  if constexpr (FMT == 1)
    *reinterpret_cast<uint4*>(atoms + 512 + lane * 16) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
}

// acc[(i0 + i) % 4] += w2[i0 + i] * (max(v[2i], 0), max(v[2i+1], 0)) for the
// C columns of one TMEM load (head pairs i0 .. i0 + C/2 - 1): the ReLU as a
// NaN-propagating max per value, then packed fp32x2 FMAs in four chains
// fixed by the head pair, so a row's sum does not depend on how its
// columns were loaded.  wrelu_total adds the chains.
template <int C, class W>
__device__ __forceinline__ void wrelu_chunk(const uint32_t (&v)[C], const W& w2, int i0, float2 (&acc)[4]) {
#pragma unroll
  for (int i = 0; i < C / 2; ++i) {
    const float2 x = make_float2(relu_nan(__uint_as_float(v[2 * i])), relu_nan(__uint_as_float(v[2 * i + 1])));
    acc[(i0 + i) % 4] = __ffma2_rn(w2[i0 + i], x, acc[(i0 + i) % 4]);
  }
}
__device__ __forceinline__ float wrelu_total(float2 (&acc)[4]) {
  acc[0] = __fadd2_rn(acc[0], acc[1]);
  acc[2] = __fadd2_rn(acc[2], acc[3]);
  acc[0] = __fadd2_rn(acc[0], acc[2]);
  return acc[0].x + acc[0].y;
}

// Order-preserving 32-bit image of a logit (-0 folded into +0); the high
// half of topk_key().
__device__ __forceinline__ uint32_t ordered_bits(float v) {
  const uint32_t u = __float_as_uint(v + 0.0f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Keep the keys >= T of cand[0, n) in place (order not kept); returns the
// number kept.  All threads of the group call it.
template <class G>
__device__ int compact_keep_ge(const G& g, uint64_t* cand, int n, uint64_t T, SelectScratch* sc) {
  const int lane = g.tid & 31;
  if (g.tid == 0) sc->bcast[3] = 0;
  g.sync();
  constexpr int kPer = 8;
  constexpr int kChunk = G::kSize * kPer;
  for (int base = 0; base < n; base += kChunk) {
    uint64_t v[kPer];
    bool keep[kPer];
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
      const int idx = base + j * G::kSize + g.tid;
      keep[j] = false;
      v[j] = 0;
      if (idx < n) {
        v[j] = cand[idx];
        keep[j] = v[j] >= T;
      }
    }
    g.sync();
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
      const uint32_t m = __ballot_sync(0xffffffffu, keep[j]);
      if (m) {
        const int leader = __ffs(m) - 1;
        uint32_t dst = 0;
        if (lane == leader) dst = atomicAdd(&sc->bcast[3], static_cast<uint32_t>(__popc(m)));
        dst = __shfl_sync(0xffffffffu, dst, leader);
        if (keep[j]) cand[dst + __popc(m & ((1u << lane) - 1u))] = v[j];
      }
    }
    g.sync();
  }
  const int kept = static_cast<int>(sc->bcast[3]);
  g.sync();
  return kept;
}

// Group-cooperative copy of the keys >= T of cand[0, n) to out[0, cap) in any
// order; returns how many keys were >= T (possibly more than cap, of which
// only cap are written).  Loads go out kPer at a time per thread.
template <class G>
__device__ uint32_t copy_keep_ge(const G& g, const uint64_t* cand, int n, uint64_t T, uint64_t* out, int cap,
                                 SelectScratch* sc) {
  const int lane = g.tid & 31;
  if (g.tid == 0) sc->bcast[3] = 0;
  g.sync();
  constexpr int kPer = 8;
  constexpr int kChunk = G::kSize * kPer;
  for (int base = 0; base < n; base += kChunk) {
    uint64_t v[kPer];
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
      const int idx = base + j * G::kSize + g.tid;
      v[j] = idx < n ? cand[idx] : 0;
    }
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
      const bool keep = base + j * G::kSize + g.tid < n && v[j] >= T;
      const uint32_t m = __ballot_sync(0xffffffffu, keep);
      if (m) {
        const int leader = __ffs(m) - 1;
        uint32_t dst = 0;
        if (lane == leader) dst = atomicAdd(&sc->bcast[3], static_cast<uint32_t>(__popc(m)));
        dst = __shfl_sync(0xffffffffu, dst, leader);
        const uint32_t o = dst + __popc(m & ((1u << lane) - 1u));
        if (keep && o < static_cast<uint32_t>(cap)) out[o] = v[j];
      }
    }
  }
  g.sync();
  const uint32_t kept = sc->bcast[3];
  g.sync();
  return kept;
}

// ---------------------------------------------------------------------------
// The kernel.
// ---------------------------------------------------------------------------
template <int H, int R, int FMT, int MODE>
__global__ void __maxnreg__((ScoreLayout<H, R, FMT, MODE>::kMaxRegs)) score_kernel(const __grid_constant__ ScoreParams p) {
  using L = ScoreLayout<H, R, FMT, MODE>;
  constexpr int kThreads = L::kThreads;
  using F = FmtTraits<FMT>;
  constexpr int N = L::N;
  constexpr int G = F::G;
  constexpr int kStages = L::kStages;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBars);
  const uint32_t bar0 = smem_u32(bars);
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (kStages + s); };
  auto accf_bar = [&](int a) { return bar0 + 8u * (2 * kStages + a); };
  auto acce_bar = [&](int a) { return bar0 + 8u * (2 * kStages + kAccBufs + a); };
  auto qfull_bar = [&](uint32_t qb) { return bar0 + 8u * (2 * kStages + 2 * kAccBufs + qb); };
  auto qempty_bar = [&](uint32_t qb) { return bar0 + 8u * (2 * kStages + 2 * kAccBufs + 2 + qb); };
  auto sfready_bar = [&](int slot) { return bar0 + 8u * (2 * kStages + 2 * kAccBufs + 4 + slot); };
  auto qsready_bar = [&](uint32_t qb) { return bar0 + 8u * (2 * kStages + 2 * kAccBufs + 4 + L::kSfaSlots + qb); };

  CtaState* st = reinterpret_cast<CtaState*>(smem + L::kState);
  RowState<R, L::kRegions>* rs = reinterpret_cast<RowState<R, L::kRegions>*>(smem + L::kRows);
  uint32_t* scan = reinterpret_cast<uint32_t*>(smem + L::kScan);
  SelectScratch* sc = reinterpret_cast<SelectScratch*>(smem + L::kScratch);
  uint32_t* hist_words = reinterpret_cast<uint32_t*>(smem + L::kHist);
  const int cap = topk_capacity(p.k);
  const int pcap = topk_part_capacity(p.k);  // keys of one partial list
  volatile int* abort_flag = &st->abort;

  // ---- one-time setup: on-chip only, so it may overlap the previous kernel
  // of the stream (launched with programmatic stream serialization)
  if (threadIdx.x == 0) {
    st->abort = 0;
    // the first TMA waits for its descriptor: fetch both early
    prefetch_tmap(&p.tmap_q);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(full_bar(s), 64);  // one arrive per producer lane, once its copies have landed
      mbar_init(empty_bar(s), 1);
    }
    for (int a = 0; a < kAccBufs; ++a) {
      mbar_init(accf_bar(a), 1);
      mbar_init(acce_bar(a), L::kGroups * 4);  // one arrive per epilogue warp of the tile's set
    }
    for (uint32_t qb = 0; qb < 2; ++qb) {
      mbar_init(qfull_bar(qb), 1);
      // freed by the MMA thread's commit (its MMAs read Q) and the scale
      // warp's arrive (it has seen this load), so a buffer is never reloaded
      // before both consumers observed the previous load's phase
      mbar_init(qempty_bar(qb), 2);
    }
    for (int sl = 0; sl < L::kSfaSlots; ++sl) mbar_init(sfready_bar(sl), 1);
    for (uint32_t qb = 0; qb < 2; ++qb) mbar_init(qsready_bar(qb), 1);  // the item's Q scales are in TMEM
    fence_barrier_init();
  }
  if (warp == 1) tmem_alloc<kTmemCols>(smem_u32(&st->tmem_base));
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = st->tmem_base;
  // every input may come from the previous kernel of the stream
  pdl_wait();

  // ---- plan this CTA's chunk of the concatenated tile space
  // (CTA 0 also publishes every item's tile start for the merge)
  if (MODE == kModeLogits && p.uniform_items) {
    if (threadIdx.x == 0) {
      const int32_t total = p.num_seqs * p.row_groups * p.total_tiles;
      const int32_t chunk = (total + static_cast<int32_t>(gridDim.x) - 1) / static_cast<int32_t>(gridDim.x);
      const int64_t x = static_cast<int64_t>(blockIdx.x) * chunk;
      st->total_tiles = total;
      st->chunk = chunk;
      st->item0 = x < total ? static_cast<int32_t>(x / p.total_tiles) : -1;
      st->item0_start = st->item0 >= 0 ? st->item0 * p.total_tiles : 0;
    }
    __syncthreads();
  } else {
    plan_items<MODE, kThreads>(p, R, threadIdx.x, scan, st, blockIdx.x == 0 ? p.item_start : nullptr);
  }
  // the selection or merge kernel that follows may start its prologue now;
  // it waits for this grid's completion before reading what it wrote
  pdl_launch_dependents();
  if (st->item0 < 0) {  // uniform: no work for this CTA
    if (warp == 1) tmem_dealloc<kTmemCols>(tmem);
    return;
  }

  const uint32_t codes_s = smem_u32(smem + L::kCodes);
  const uint32_t q_s = smem_u32(smem + L::kQ);
  const uint32_t kraw_s = smem_u32(smem + L::kKraw);
  const uint8_t* kraw = smem + L::kKraw;
  uint8_t* sfa_rows = smem + L::kSfaRows;
  uint8_t* sfb_atoms = smem + L::kSfb;

  if (warp == 0 || warp == L::kProducer2Warp) {
    // ================================================================ producers
    // Both producer warps work on every tile: warp 0 copies keys 0..63 of
    // the tile, the last warp keys 64..127 -- one 64-key page each, or one
    // half of a 128-key page -- with 16-byte cp.async copies (a page is far
    // too small for a tensor copy to pay its issue cost): its 4 KB of codes
    // in eight coalesced 512-byte warp copies, each 16-byte chunk placed at
    // its key's MMA row (the strided order for MXFP4) under the operand's
    // 64-byte swizzle, and its 64 G scale bytes unchanged.  Every lane then
    // arrives on the stage's full barrier once its copies have landed
    // (64 arrivals a phase).  Lane l caches the physical id of logical page
    // base + l (and of the next 32, prefetched).  Warp 0 also loads each
    // item's Q codes by TMA.
    const uint32_t pidx = warp == 0 ? 0u : 1u;
    uint32_t tile_iter = 0, item_iter = 0;
    bool ok = true;
    const int pshift = p.page_shift;
    FP4IDX_STAMP_INIT();
    for_each_segment<MODE, R>(p, st, [&](int, const ItemInfo& it, int lo, int hi, int) {
      if (!ok) return;
      if (pidx == 0) {
        const uint32_t qb = item_iter & 1u, qph = (item_iter >> 1) & 1u;
        FP4IDX_STAMP(3);
        ok = warp_wait(qempty_bar(qb), qph ^ 1u, abort_flag, p.err);
        FP4IDX_STAMP(0);
        if (!ok) return;
        if (lane == 0) {
          mbar_arrive_expect_tx(qfull_bar(qb), N * kCodeBytes);
          tma_load_3d(q_s + qb * L::kQBytes, &p.tmap_q, 0, 0, it.row0, qfull_bar(qb));
        }
      }
      ++item_iter;
      const int32_t npages = (it.k_len + p.page_size - 1) >> pshift;
      const int32_t* table = p.block_table + it.table_base;
      auto fetch = [&](int32_t b) -> int32_t {
        const int32_t lp = b + lane;
        return lp < npages ? __ldg(table + lp) : -1;
      };
      const int32_t half = 64 * static_cast<int32_t>(pidx);  // this warp's first key in a tile
      int32_t base = (((lo << 7) + half) >> pshift) & ~31;
      int32_t cur_ids = fetch(base), next_ids = fetch(base + 32);
      for (int j = lo; j < hi; ++j) {
        if (MODE == kModeLogits && !tile_has_visible(it, j)) continue;
        const int32_t key0 = (j << 7) + half;  // first logical position of this warp's 64 keys
        const int32_t lp = key0 >> pshift;     // their page (warp-uniform)
        if (lp >= base + 32) {
          base += 32;
          cur_ids = next_ids;
          next_ids = fetch(base + 32);
        }
        const int32_t phys = __shfl_sync(0xffffffffu, cur_ids, lp - base);
        const bool in_len = key0 < it.k_len;
        const bool good = in_len && phys >= 0 && phys < p.num_pages;
        // one report per page: a 128-key page's first half reports it
        if (lane == 0 && in_len && !good && (key0 & (p.page_size - 1)) == 0) atomicOr(p.err, kErrPageRange);
        const int s = tile_iter % kStages;
        const uint32_t ph = (tile_iter / kStages) & 1u;
        FP4IDX_STAMP(3);
        ok = warp_wait(empty_bar(s), ph ^ 1u, abort_flag, p.err);
        FP4IDX_STAMP(1);
        if (!ok) return;
        if (good) {
          const int32_t in_page = key0 & (p.page_size - 1);
          const uint8_t* codes = p.kcode_base + static_cast<int64_t>(phys) * p.kcode_block_stride + in_page * kCodeBytes;
          const uint32_t dst0 = codes_s + s * 8192;
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const int c = 32 * u + lane;       // 16-byte chunk of the warp's 4 KB
            const int kq = half + (c >> 2);    // key within the tile
            const int m = L::kDirectSf ? 32 * (kq & 3) + (kq >> 2) : kq;  // its MMA row
            const int jj = (c & 3) ^ ((m >> 1) & 3);                       // 64-byte swizzle
            cp_async_16(dst0 + m * kCodeBytes + jj * 16, codes + c * 16);
          }
          if (lane < 4 * G)  // 64 keys x G scale bytes
            cp_async_16(kraw_s + s * (128 * G) + half * G + lane * 16,
                        p.kscale_base + static_cast<int64_t>(phys) * p.kscale_block_stride + in_page * G + lane * 16);
        }
        cp_async_arrive(full_bar(s));
        FP4IDX_STAMP(2);
        FP4IDX_STAMP_COUNT();
        ++tile_iter;
      }
    });
    FP4IDX_STAMP(3);
    FP4IDX_STAMP_DONE(0);
    if (lane == 0 && pidx == 0 && !ok) {
      // Let the Q copies in flight land before the CTA can exit.
      volatile int never = 0;
      for (uint32_t u = item_iter > 2u ? item_iter - 2u : 0u; u < item_iter; ++u)
        mbar_wait(qfull_bar(u & 1u), (u >> 1) & 1u, &never, p.err);
    }
    // this thread's own cp.async copies land before it exits
    cp_async_wait_all();
    __syncwarp();
  } else if (warp == 1) {
    // ================================================================ MMA issuer
    // One thread only waits and issues: an MMA issue holds the issuing
    // thread for most of the MMA's duration, so any other per-tile work here
    // would leave the tensor pipe idle.
    if (lane == 0) {
      const uint64_t a_desc0 = desc_kmajor_sw64(codes_s);
      const uint64_t b_desc0 = desc_kmajor_sw64(q_s);
      uint32_t tile_iter = 0, item_iter = 0;
      uint32_t sf_phase = 0;  // bit slot: phase of the K-scale slot's next use
      bool ok = true;
      int last_acc = -1;
      uint32_t last_acc_phase = 0;
      FP4IDX_STAMP_INIT();
      for_each_segment<MODE, R>(p, st, [&](int, const ItemInfo& it, int lo, int hi, int) {
        if (!ok) return;
        const uint32_t qb = item_iter & 1u;
        // the first scale warp copied (or, with no tile to compute, skipped)
        // this item's Q scales
        if (!(ok = mbar_wait(qsready_bar(qb), (item_iter >> 1) & 1u, abort_flag, p.err))) return;
        const uint32_t sfb_t = tmem + L::kSfbCol + qb * 8u;
        const uint64_t bdesc = b_desc0 + static_cast<uint64_t>((qb * L::kQBytes) >> 4);
        for (int j = lo; j < hi && ok; ++j) {
          if (MODE == kModeLogits && !tile_has_visible(it, j)) continue;
          const int s = tile_iter % kStages;
          const int slot = tile_iter % L::kSfaSlots;
          const int a = tile_iter % kAccBufs;
          const uint32_t aph = (tile_iter / kAccBufs) & 1u;
          FP4IDX_STAMP(3);
          if constexpr (L::kDirectSf) {
            // the stage's codes and raw scales landed
            if (!(ok = mbar_wait(full_bar(s), (tile_iter / kStages) & 1u, abort_flag, p.err))) break;
          } else {
            // a scale warp copied this tile's K scales after the stage's
            // codes landed
            if (!(ok = mbar_wait(sfready_bar(slot), (sf_phase >> slot) & 1u, abort_flag, p.err))) break;
            sf_phase ^= 1u << slot;
          }
          FP4IDX_STAMP(0);
          if (!(ok = mbar_wait(acce_bar(a), aph ^ 1u, abort_flag, p.err))) break;
          FP4IDX_STAMP(1);
          tc_fence_after();
          // the stage was written by cp.async (generic proxy); the MMA and
          // the scale copy read it through the async proxy
          fence_proxy_async_smem();
          const uint32_t sfa_t = tmem + L::kSfaCol + slot * 8u;
          if constexpr (L::kDirectSf) {
            // slot == a: the MMA that last read it finished before the
            // epilogue released accumulator a; the copy completes before
            // the MMAs below read it (tcgen05 operations of one thread run
            // in issue order)
            tc_cp_32x128b_warpx4(sfa_t, desc_sf_atom(kraw_s + s * (128 * G)));
          }
          const uint32_t d = tmem + L::kAccCol + a * 128u;
          const uint64_t adesc = a_desc0 + static_cast<uint64_t>((s * 8192) >> 4);
#pragma unroll
          for (int kk = 0; kk < 2; ++kk) {
            constexpr uint32_t sf1 = F::kScaleVec == 2 ? 2u : 0u;
            const uint32_t idesc = kk == 0 ? idesc_fp4(128, N, F::kUe8m0, 0, 0) : idesc_fp4(128, N, F::kUe8m0, sf1, sf1);
            const uint32_t col = F::kScaleVec == 2 ? 0u : 4u * kk;
            tc_mma_fp4<F::kScaleVec>(d, adesc + 2u * kk, bdesc + 2u * kk, idesc, sfa_t + col, sfb_t + col,
                                     static_cast<uint32_t>(kk));
          }
          tc_commit(empty_bar(s));
          tc_commit(accf_bar(a));
          FP4IDX_STAMP(2);
          FP4IDX_STAMP_COUNT();
          last_acc = a;
          last_acc_phase = aph;
          ++tile_iter;
        }
        if (!ok) return;
        // Q buffer and Q-scale slot free once this item's MMAs complete.
        tc_commit(qempty_bar(qb));
        ++item_iter;
      });
      FP4IDX_STAMP(3);
      FP4IDX_STAMP_DONE(1);
      if (!ok && last_acc >= 0) {
        // Outstanding MMAs must finish before TMEM is released.
        volatile int never = 0;
        mbar_wait(accf_bar(last_acc), last_acc_phase, &never, p.err);
      }
    }
    __syncwarp();
  } else if (warp == 2 || (L::kScaleWarps == 2 && warp == L::kScale2Warp)) {
    // ================================================================ scales
    // Two warps, alternate tiles (warp 2 the even ones).  Per item (warp 2
    // only): the Q scales of its rows -> 32x4x4 atoms -> TMEM slot item % 2
    // (free: the producer loaded this item's Q only after the MMAs of
    // item - 2 completed), committed to the item's Q-scale barrier.  Per
    // tile (NVFP4 only: MXFP4 scales go from the stage to TMEM by the MMA
    // thread): raw K scales [128 keys][G] -> 128
    // rows of the scale layout (row r holds atom line r % 32: the words of
    // keys l, 32+l, 64+l, 96+l, l = r % 32; NVFP4's second K half in the
    // second 16 bytes), one tcgen05.cp 128x128b/256b into TMEM slot
    // tile % kSfaSlots, committed to that slot's barrier.  A slot (TMEM and
    // shared staging) is rewritten only after the MMA of the tile that last
    // used it completed (its stage's empty barrier).
    const uint32_t sidx = warp == 2 ? 0u : 1u;
    const uint32_t smask = L::kScaleWarps == 2 ? 1u : 0u;  // tiles of this warp: (tile & smask) == sidx
    const uint64_t sfa_desc0 = desc_sf_rows(smem_u32(sfa_rows));
    uint32_t tile_iter = 0, item_iter = 0;
    bool ok = true;
    FP4IDX_STAMP_INIT();
    for_each_segment<MODE, R>(p, st, [&](int, const ItemInfo& it, int lo, int hi, int) {
      if (!ok) return;
      FP4IDX_STAMP(4);
      const uint32_t qb = item_iter & 1u, qph = (item_iter >> 1) & 1u;
      if (sidx == 0) {
        ok = warp_wait(qfull_bar(qb), qph, abort_flag, p.err);
        if (!ok) return;
        // Q scales only when some tile of the segment is computed (otherwise
        // no MMA reads them); the barrier is committed either way
        if (MODE != kModeLogits || tile_has_visible(it, lo)) {
          q_scale_atoms<H, R, FMT>(p, it, sfb_atoms + qb * (F::kAtoms * 512), lane);
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            tc_fence_after();
            const uint32_t sfb_t = tmem + L::kSfbCol + qb * 8u;
#pragma unroll
            for (int at = 0; at < F::kAtoms; ++at)
              tc_cp_32x128b_warpx4(sfb_t + 4u * at, desc_sf_atom(smem_u32(sfb_atoms + (qb * F::kAtoms + at) * 512)));
          }
        }
        if (lane == 0) {
          tc_commit(qsready_bar(qb));
          mbar_arrive(qempty_bar(qb));
        }
        __syncwarp();
      }
      FP4IDX_STAMP(0);
      if constexpr (L::kDirectSf) {  // the MMA thread copies the K scales
        ++item_iter;
        return;
      }
      for (int j = lo; j < hi; ++j) {
        if (MODE == kModeLogits && !tile_has_visible(it, j)) continue;
        if ((tile_iter & smask) != sidx) {  // the other scale warp's tile
          ++tile_iter;
          continue;
        }
        const int s = tile_iter % kStages;
        const uint32_t ph = (tile_iter / kStages) & 1u;
        const int slot = tile_iter % L::kSfaSlots;
        bool got = false;
        FP4IDX_STAMP(4);
        if (lane == 0) {
          got = mbar_wait(full_bar(s), ph, abort_flag, p.err);
          FP4IDX_STAMP(1);
          if (got && tile_iter >= static_cast<uint32_t>(L::kSfaSlots)) {
            const uint32_t u = tile_iter - L::kSfaSlots;  // previous user of the slot
            got = mbar_wait(empty_bar(u % kStages), (u / kStages) & 1u, abort_flag, p.err);
          }
          FP4IDX_STAMP(2);
        }
        ok = __shfl_sync(0xffffffffu, got, 0);
        if (!ok) break;
        {
          const uint8_t* raw = kraw + s * (128 * G);
          uint8_t* rows = sfa_rows + slot * (F::kAtoms * 2048);
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
          const uint32_t sfa_t = tmem + L::kSfaCol + slot * 8u;
          const uint64_t sdesc = sfa_desc0 + static_cast<uint64_t>((slot * F::kAtoms * 2048) >> 4);
          if constexpr (G == 4) tc_cp_128x128b(sfa_t, sdesc);
          else tc_cp_128x256b(sfa_t, sdesc);
          tc_commit(sfready_bar(slot));
        }
        __syncwarp();
        FP4IDX_STAMP(3);
        FP4IDX_STAMP_COUNT();
        ++tile_iter;
      }
      ++item_iter;
    });
    FP4IDX_STAMP(4);
    FP4IDX_STAMP_DONE(2);
    if (lane == 0) {
      // copies still in flight must land before TMEM is released
      volatile int never = 0;
      const uint32_t first = tile_iter > static_cast<uint32_t>(L::kSfaSlots) ? tile_iter - L::kSfaSlots : 0;
      for (uint32_t u = first; u < tile_iter && !L::kDirectSf; ++u)
        if ((u & smask) == sidx) mbar_wait(sfready_bar(u % L::kSfaSlots), (u / L::kSfaSlots) & 1u, &never, p.err);
      if (sidx == 0 && item_iter > 0) {
        const uint32_t u = item_iter - 1;
        mbar_wait(qsready_bar(u & 1u), (u >> 1) & 1u, &never, p.err);
      }
    }
    __syncwarp();
  } else if (warp >= L::kWarpsUsed) {
    // spare warp (the CTA is a whole number of four-warp groups)
  } else {
    // ================================================================ epilogue
    constexpr int RG = L::kRowsPerGroup;  // query rows of this group
    constexpr int kG = kEpiThreads * L::kSets;  // threads of a row group (all its sets)
    constexpr int kRegions = L::kRegions;
    const int gi4 = (warp - L::kEpiWarp0) >> 2;  // four-warp group
    const int set = gi4 / L::kGroups;            // the tile parity it takes (two sets)
    const int gi = gi4 - set * L::kGroups;       // its row group
    const int r0 = gi * RG;  // first row of the item this group handles
    Group<kG, -1> g{set * kEpiThreads + static_cast<int>(threadIdx.x) - 32 * L::kEpiWarp0 - gi4 * kEpiThreads, 1 + gi};
    SelectScratch* gsc = sc + gi;
    const int quad = warp & 3;
    const int region = set * 4 + quad;  // this warp's append region of each row
    // key of this thread's accumulator lane 32 quad + lane within the tile
    // (MXFP4: the strided order of the producer's code boxes)
    const int key_local = L::kDirectSf ? 4 * lane + quad : quad * 32 + lane;
    // Candidate buffer of each row (shared memory for two-row CTAs, else the
    // workspace), ccap keys laid out as
    //   [0, seg0)                       keys kept by the last compaction
    //   [seg0 + q * rsz, + wc[q])       keys warp q of the row group appended since
    // with rsz = (ccap - seg0) / kRegions, so an append needs no atomic: each
    // warp owns its region and keeps its count in a register.  The counts
    // are published and checked every `check_every` tiles (a set takes
    // check_every / kSets of them); a region then keeps that many tiles of
    // room (32 keys per tile and warp) above the trigger.
    const int ccap = L::kSmemCand ? L::kCandCap : topk_cand_capacity(p.k);
    // a region is at least ccap / 16 keys; two-row CTAs (two sets, each
    // taking half of the tiles between checks) check every 16 tiles
    const int check_every = ccap >= 4096 ? (L::kSmemCand ? 16 : 8) : 4;
    const int margin = check_every / L::kSets * 32;
    const uint32_t kk = static_cast<uint32_t>(p.k);
    int since_check = 0;
    uint32_t tile_iter = 0;
    bool ok = true;
    auto cand_of = [&](int rr) {
      return L::kSmemCand ? reinterpret_cast<uint64_t*>(smem + L::kCand) + (r0 + rr) * L::kCandCap
                          : p.cand + (static_cast<int64_t>(blockIdx.x) * R + r0 + rr) * ccap;
    };
    // Segmented view of one row's buffer: virtual index i < seg0 + sum(c)
    // -> position in the buffer.
    struct SegView {
      int seg0, rsz, c[kRegions];
      __device__ __forceinline__ int n() const {
        int s = seg0;
#pragma unroll
        for (int q = 0; q < kRegions; ++q) s += c[q];
        return s;
      }
      __device__ __forceinline__ int pos(int i) const {
        if (i < seg0) return i;
        int j = i - seg0;
#pragma unroll
        for (int q = 0; q < kRegions - 1; ++q) {
          if (j < c[q]) return seg0 + q * rsz + j;
          j -= c[q];
        }
        return seg0 + (kRegions - 1) * rsz + j;
      }
      __device__ __forceinline__ int fullest() const {
        int m = 0;
#pragma unroll
        for (int q = 0; q < kRegions; ++q) m = max(m, c[q]);
        return m;
      }
    };
    // Group-cooperative visit of every key of a row's buffer, eight loads in
    // flight per thread.  fn runs only on the lanes that hold a key, so it
    // must not contain warp-synchronous operations.
    auto visit = [&](const uint64_t* cr, const SegView& sv, auto&& fn) {
      const int n = sv.n();
      for (int base = 0; base < n; base += 8 * kG) {
        uint64_t kv[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int e = base + j * kG + g.tid;
          kv[j] = e < n ? cr[sv.pos(e)] : 0;
        }
#pragma unroll
        for (int j = 0; j < 8; ++j)
          if (base + j * kG + g.tid < n) fn(kv[j]);
      }
    };
    // Each row keeps a bucket histogram (top kHistShift.. key bits) of the
    // keys appended to its buffer.  The lower edge of the bucket holding the
    // k-th largest of them is a valid threshold for the row (the k-th
    // largest of any subset of a row's keys is at most its k-th largest), so
    // the threshold rises at every check without touching the buffer.
    auto hist_of = [&](int rr) { return Hist16{hist_words + (r0 + rr) * (kHistBins / 2)}; };
    static_assert(kHistBins == kPoolBins, "pooled and per-CTA buckets agree");
    // Keys >= T of the buffer moved, in place, to [0, kept); returns kept.
    // A round reads 8 * kG keys into registers before writing any:
    // every write lands below the number of keys read so far, and an unread
    // key sits at a position at least its virtual index, so none is
    // overwritten before it is read.
    auto compact = [&](uint64_t* cr, const SegView& sv, uint64_t T) -> int {
      if (g.tid == 0) gsc->bcast[3] = 0;
      g.sync();
      const int n = sv.n();
      for (int base = 0; base < n; base += 8 * kG) {
        uint64_t kv[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int e = base + j * kG + g.tid;
          kv[j] = e < n ? cr[sv.pos(e)] : 0;
        }
        g.sync();
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const bool keep = base + j * kG + g.tid < n && kv[j] >= T;
          const uint32_t m = __ballot_sync(0xffffffffu, keep);
          if (m) {
            const int leader = __ffs(m) - 1;
            uint32_t dst = 0;
            if (lane == leader) dst = atomicAdd(&gsc->bcast[3], static_cast<uint32_t>(__popc(m)));
            dst = __shfl_sync(0xffffffffu, dst, leader);
            if (keep) cr[dst + __popc(m & ((1u << lane) - 1u))] = kv[j];
          }
        }
        g.sync();
      }
      const int kept = static_cast<int>(gsc->bcast[3]);
      g.sync();
      return kept;
    };
    // Region counts are published (each warp's lane 0 writes its counts,
    // then the group barrier) into alternate copies, so a publication never
    // overwrites the copy a slower warp may still be reading: it read it
    // before reaching the barrier of the next publication.
    int pub = 0;
    auto publish = [&](const int (&wcnt)[L::kRowsPerGroup], bool valid) {
      ++pub;
#pragma unroll
      for (int rr = 0; rr < L::kRowsPerGroup; ++rr)
        if (lane == 0) rs->wc[pub & 1][r0 + rr][region] = valid ? wcnt[rr] : 0;
    };
    auto view_of = [&](int rr, int seg0) {
      const int32_t* c = rs->wc[pub & 1][r0 + rr];
      SegView v;
      v.seg0 = seg0;
      v.rsz = (ccap - seg0) / kRegions;
#pragma unroll
      for (int q = 0; q < kRegions; ++q) v.c[q] = c[q];
      return v;
    };
    FP4IDX_STAMP_INIT();
    for_each_segment<MODE, R>(p, st, [&](int item, const ItemInfo& it, int lo, int hi, bool own) {
      // -- this group's rows of the item: weights in registers, visibility
      bool row_valid[RG];
      int32_t t[RG], vis[RG];
      float2 w2[RG][H / 2];  // head weight pairs, see wrelu_chunk
      uint64_t thr[RG];      // each row's buffer accepts keys >= thr
      int seg0[RG];          // keys kept by the row's last compaction (front of its buffer)
      int wcnt[RG];          // keys this warp appended to its region of the row's buffer
      // pooled counts (see pool_raise): this lane's highest appended bucket,
      // the window top and bucket count loaded at the last check, the row's
      // pooled top loaded then
      uint32_t pl_top[RG], pl_win[RG], pl_cnt[RG], pl_next[RG];
#pragma unroll
      for (int rr = 0; rr < RG; ++rr) {
        row_valid[rr] = r0 + rr < it.nrows;
        t[rr] = it.row0 + r0 + rr;
        vis[rr] = row_valid[rr] ? row_visible(p, it, t[rr]) : 0;
        if constexpr (MODE == kModeTopk) {
          // ordered before any read by the group barrier after the histogram clear
          float* ws = reinterpret_cast<float*>(smem + L::kW) + (r0 + rr) * H;
          for (int h = g.tid; h < H; h += kG)
            ws[h] = row_valid[rr] ? __ldg(p.w + static_cast<int64_t>(t[rr]) * p.w_row_stride + h) : 0.0f;
        } else {
#pragma unroll
          for (int i = 0; i < H / 2; ++i) {
            const float* wr = p.w + static_cast<int64_t>(t[rr]) * p.w_row_stride + 2 * i;
            w2[rr][i] = row_valid[rr] ? make_float2(__ldg(wr), __ldg(wr + 1)) : make_float2(0.0f, 0.0f);
          }
        }
        thr[rr] = 0;
        seg0[rr] = 0;
        wcnt[rr] = 0;
        pl_top[rr] = pl_win[rr] = pl_cnt[rr] = pl_next[rr] = 0;
      }
      if constexpr (MODE == kModeTopk) {
#pragma unroll
        for (int rr = 0; rr < RG; ++rr) {
          const Hist16 hr = hist_of(rr);
          for (int e = g.tid; e < kHistBins / 2; e += kG) hr.w[e] = 0;
        }
        g.sync();  // cleared before any warp of the group appends
      }
      since_check = 0;
      // Page ids for the validity check: lane l caches the id of logical
      // page pbase + l and the next 32 are loaded 32 pages ahead, so no
      // table load latency is exposed per tile (a warp's 32 keys share a page).
      const int32_t npages = (it.k_len + p.page_size - 1) >> p.page_shift;
      auto fetch_ids = [&](int32_t b) -> int32_t {
        const int32_t lp = b + lane;
        return lp < npages ? __ldg(p.block_table + it.table_base + lp) : -1;
      };
      int32_t pbase = ((lo << 7) >> p.page_shift) & ~31;
      int32_t ids_cur = fetch_ids(pbase), ids_next = fetch_ids(pbase + 32);
      FP4IDX_STAMP(0);
      for (int j = lo; j < hi; ++j) {
        const bool real = !(MODE == kModeLogits && !tile_has_visible(it, j));
        // with two sets, this group's tiles are those of its parity; the
        // other set's tiles only count toward the checks
        const bool mine = L::kSets == 1 || (tile_iter & 1u) == static_cast<uint32_t>(set);
        if (real && !mine) ++tile_iter;
        if (mine) {
          const int32_t pos = (j << 7) + key_local;
          const int32_t lp0 = (j << 7) >> p.page_shift;  // the tile's first page (warp-uniform)
          if (lp0 >= pbase + 32) {
            pbase += 32;
            ids_cur = ids_next;
            ids_next = fetch_ids(pbase + 32);
          }
          // this lane's page: lp0 or, with 64-key pages, lp0 + 1 (then
          // possibly the first of the next 32)
          const int32_t d = (pos >> p.page_shift) - pbase;
          const int32_t id_a = __shfl_sync(0xffffffffu, ids_cur, d & 31);
          const int32_t id_b = __shfl_sync(0xffffffffu, ids_next, d & 31);
          const int32_t pg_cur = d < 32 ? id_a : id_b;
          float val[RG];
#pragma unroll
          for (int rr = 0; rr < RG; ++rr) val[rr] = -INFINITY;
          if (real) {
            const int a = tile_iter % kAccBufs;
            const uint32_t aph = (tile_iter / kAccBufs) & 1u;
            // Each warp waits for the accumulator itself (no group barrier per
            // tile); ok stays warp-uniform, as tcgen05.ld below is a
            // whole-warp instruction.
            FP4IDX_STAMP(4);
            ok = ok && warp_wait(accf_bar(a), aph, abort_flag, p.err);
            FP4IDX_STAMP(1);
            if (ok) {
              tc_fence_after();
              // each row's H columns in chunks (registers: 32 columns, 16 for
              // the 64-head top-k, whose warps run at 96 registers); the
              // accumulator is released once its last chunk is loaded
              const uint32_t tcol = tmem + (static_cast<uint32_t>(quad * 32) << 16) + L::kAccCol + a * 128u + r0 * H;
              constexpr int kChunk = L::kMaxRegs >= 160 || H < 32 ? H : (MODE == kModeTopk && H == 64 ? 16 : 32);
#pragma unroll
              for (int rr = 0; rr < RG; ++rr) {
                float2 acc[4];
#pragma unroll
                for (int c = 0; c < 4; ++c) acc[c] = make_float2(0.0f, 0.0f);
#pragma unroll
                for (int c0 = 0; c0 < H; c0 += kChunk) {
                  uint32_t v[kChunk];
                  tmem_ld<kChunk>(tcol + rr * H + c0, v);
                  tmem_wait_ld();
                  reg_fence(v);
                  if (rr == RG - 1 && c0 + kChunk == H) {
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(acce_bar(a));
                  }
                  if constexpr (MODE == kModeTopk)
                    wrelu_chunk<kChunk>(v, reinterpret_cast<const float2*>(smem + L::kW) + (r0 + rr) * (H / 2),
                                        c0 / 2, acc);
                  else
                    wrelu_chunk<kChunk>(v, w2[rr], c0 / 2, acc);
                }
                val[rr] = wrelu_total(acc);
              }
              FP4IDX_STAMP(3);
            }
            FP4IDX_STAMP_COUNT();
            ++tile_iter;
          }
          const bool page_good = pos < it.k_len && pg_cur >= 0 && pg_cur < p.num_pages;
          // candidate mask: a cleared position is not a candidate (-inf, never selected)
          bool cand[RG];
#pragma unroll
          for (int rr = 0; rr < RG; ++rr)
            cand[rr] = !p.cand_mask || (pos < vis[rr] && __ldg(p.cand_mask + static_cast<int64_t>(t[rr]) * p.mask_ld + pos) != 0);
          if constexpr (MODE == kModeLogits) {
#pragma unroll
            for (int rr = 0; rr < RG; ++rr)
              if (ok && row_valid[rr] && pos < p.ld)
                p.logits[static_cast<int64_t>(t[rr]) * p.ld + pos] =
                    page_good && pos < vis[rr] && cand[rr] ? val[rr] : -INFINITY;
          } else {
#pragma unroll
            for (int rr = 0; rr < RG; ++rr) {
              // NaN logits are never selected
              const uint64_t key = (static_cast<uint64_t>(ordered_bits(val[rr])) << 32) |
                                   static_cast<uint64_t>(~static_cast<uint32_t>(pos));
              const bool take = ok && page_good && pos < vis[rr] && cand[rr] && !isnan(val[rr]) && key >= thr[rr];
              const uint32_t m = __ballot_sync(0xffffffffu, take);
              if (m) {
                // this warp's region: no other warp writes there
                const int slot_i = wcnt[rr] + __popc(m & ((1u << lane) - 1u));
                const uint32_t bkt = static_cast<uint32_t>(key >> kHistShift);
                if (take) {
                  cand_of(rr)[seg0[rr] + region * ((ccap - seg0[rr]) / kRegions) + slot_i] = key;
                  hist_of(rr).add(static_cast<int>(bkt));
                  if (!L::kSmemCand && p.pool_hist) {
                    red_add_u32(p.pool_hist + static_cast<int64_t>(t[rr]) * kHistBins + bkt, 1u);
                    pl_top[rr] = max(pl_top[rr], bkt);
                  }
                }
                wcnt[rr] += __popc(m);
              }
            }
          }
        }
        if constexpr (MODE == kModeTopk) {
          FP4IDX_STAMP(4);
          if (++since_check < check_every) continue;
          since_check = 0;
          if (!L::kSmemCand && p.pool_hist) {
            // Pooled threshold, per warp and without waiting on memory: the
            // 32 buckets below the top read at the last check hold counts
            // that every CTA scoring a row adds to as it appends keys; each
            // count read is at most the row's count at that moment and every
            // counted key exists, so k keys in buckets >= b make b's lower
            // edge a valid threshold (the k-th largest key of the row is at
            // least that large).  Then this warp's highest bucket is pooled
            // and the next window's counts and top are requested.
#pragma unroll
            for (int rr = 0; rr < RG; ++rr) {
              if (!row_valid[rr]) continue;  // warp-uniform
              const uint32_t wm = __reduce_max_sync(0xffffffffu, pl_top[rr]);
              if (lane == 0 && wm > 0) red_max_u32(p.pool_top + t[rr], wm);
              const int b = static_cast<int>(pl_win[rr]) - 31 + lane;
              const uint32_t c = b >= 0 ? pl_cnt[rr] : 0u;
              uint32_t incl = c;  // keys in this lane's bucket and above
#pragma unroll
              for (int o = 1; o < 32; o <<= 1) {
                const uint32_t y = __shfl_down_sync(0xffffffffu, incl, o);
                if (lane + o < 32) incl += y;
              }
              const uint32_t hit = __ballot_sync(0xffffffffu, incl >= kk && incl - c < kk);
              if (hit) {
                const uint64_t Tp = static_cast<uint64_t>(static_cast<int>(pl_win[rr]) - 31 + (__ffs(hit) - 1))
                                    << kHistShift;
                if (Tp > thr[rr]) thr[rr] = Tp;
              }
              pl_win[rr] = pl_next[rr];
              const int nb = static_cast<int>(pl_win[rr]) - 31 + lane;
              pl_cnt[rr] = nb >= 0 ? ld_relaxed_u32(p.pool_hist + static_cast<int64_t>(t[rr]) * kHistBins + nb) : 0u;
              pl_next[rr] = ld_relaxed_u32(p.pool_top + t[rr]);
            }
          }
          publish(wcnt, true);
          g.sync();
          // -- threshold raise from each row's histogram; compaction of a row
          // whose fullest region is near its end, one row at a time
#pragma unroll 1
          for (int rr = 0; rr < RG; ++rr) {
            int sg = 0;  // rr is uniform across the group: registers of row rr
            uint64_t T = 0;
#pragma unroll
            for (int q = 0; q < RG; ++q)
              if (q == rr) {
                sg = seg0[q];
                T = thr[q];
              }
            const SegView sv = view_of(rr, sg);
            // uniform: read after the barrier.  With pooled counts the warps
            // raise their thresholds from the pool; the row's own bucket is
            // then only needed for a compaction.
            if (sv.n() <= p.k) continue;
            if (!L::kSmemCand && p.pool_hist && sv.fullest() <= sv.rsz - margin) continue;
            const Hist16 hr = hist_of(rr);
            uint32_t above = 0;
            const uint32_t bkt = find_kth_bucket(g, hr, kk, gsc, &above);
            const uint64_t Tb = static_cast<uint64_t>(bkt) << kHistShift;
            T = Tb > T ? Tb : T;
            if (sv.fullest() > sv.rsz - margin) {
              // keep the bucket of the k-th key and above, or exactly the k
              // largest when that would keep more than half the buffer
              uint64_t* cr = cand_of(rr);
              const bool exact = above + hr(static_cast<int>(bkt)) > static_cast<uint32_t>(ccap / 2);
              if (exact) {
                const uint64_t Te = select_in_bucket(g, bkt, kk - above, gsc, [&](auto&& fn) { visit(cr, sv, fn); });
                T = Te > T ? Te : T;  // T may be a warp's higher pooled threshold
              }
              const int left = compact(cr, sv, T);
              // the histogram follows the buffer: buckets below bkt are empty now
              for (int wd = g.tid; wd < static_cast<int>(bkt >> 1); wd += kG) hr.w[wd] = 0;
              g.sync();
              if (g.tid == 0) {
                if (bkt & 1u) hr.set(static_cast<int>(bkt) - 1, 0);
                if (exact) hr.set(static_cast<int>(bkt), kk - above);
              }
              g.sync();
#pragma unroll
              for (int q = 0; q < RG; ++q)
                if (q == rr) {
                  seg0[q] = left;
                  wcnt[q] = 0;
                }
            }
#pragma unroll
            for (int q = 0; q < RG; ++q)
              if (q == rr) thr[q] = T;
          }
          FP4IDX_STAMP(5);
        }
      }
      if constexpr (MODE == kModeTopk) {
        // -- flush each of this group's rows: its candidates go to the row's
        // partial list, a superset of the top k of the keys this CTA scored
        // (the merge selects exactly): only the keys in or above the bucket
        // of the k-th largest, which the row's histogram gives without a
        // pass over the buffer.  (Two-row CTAs with one set of epilogue warps
        // copy every candidate: there the threshold cost the scorer more than
        // it saved the merge; with two sets it saves more, measured.)
        const int slot = own ? static_cast<int>(blockIdx.x) : static_cast<int>(gridDim.x) + item;
        publish(wcnt, ok);
#pragma unroll 1
        for (int rr = 0; rr < RG; ++rr) {
          const uint64_t* cr = cand_of(rr);
          g.sync();
          int sg = 0;
#pragma unroll
          for (int q = 0; q < RG; ++q)
            if (q == rr) sg = ok ? seg0[q] : 0;
          const SegView sv = view_of(rr, sg);
          const int n = sv.n();
          const int64_t part = static_cast<int64_t>(slot) * R + r0 + rr;
          uint64_t* out = p.part_keys + part * pcap;
          int wrote = n;
          if constexpr (L::kSmemCand && L::kSets == 1) {
            // n <= ccap <= pcap: the buffer's keys, in order, eight in
            // flight per thread
            for (int base = 0; base < n; base += 8 * kG) {
              uint64_t kv[8];
#pragma unroll
              for (int j = 0; j < 8; ++j) {
                const int e = base + j * kG + g.tid;
                kv[j] = e < n ? cr[sv.pos(e)] : 0;
              }
#pragma unroll
              for (int j = 0; j < 8; ++j) {
                const int e = base + j * kG + g.tid;
                if (e < n) out[e] = kv[j];
              }
            }
          } else {
            uint64_t T = 0;
#pragma unroll
            for (int q = 0; q < RG; ++q)
              if (q == rr) T = thr[q];
            if (n > p.k) {  // uniform
              uint32_t above = 0;
              const uint64_t Tb = static_cast<uint64_t>(find_kth_bucket(g, hist_of(rr), kk, gsc, &above))
                                  << kHistShift;
              T = Tb > T ? Tb : T;
            }
            // keys >= T, every lane taking part in each ballot
            if (g.tid == 0) gsc->bcast[3] = 0;
            g.sync();
            for (int base = 0; base < n; base += 8 * kG) {
              uint64_t kv[8];
#pragma unroll
              for (int j = 0; j < 8; ++j) {
                const int e = base + j * kG + g.tid;
                kv[j] = e < n ? cr[sv.pos(e)] : 0;
              }
#pragma unroll
              for (int j = 0; j < 8; ++j) {
                const bool keep = base + j * kG + g.tid < n && kv[j] >= T;
                const uint32_t m = __ballot_sync(0xffffffffu, keep);
                if (m) {
                  const int leader = __ffs(m) - 1;
                  uint32_t dst = 0;
                  if (lane == leader) dst = atomicAdd(&gsc->bcast[3], static_cast<uint32_t>(__popc(m)));
                  dst = __shfl_sync(0xffffffffu, dst, leader);
                  if (keep) out[dst + __popc(m & ((1u << lane) - 1u))] = kv[j];
                }
              }
            }
            g.sync();
            wrote = static_cast<int>(gsc->bcast[3]);
            g.sync();
          }
          bool valid_rr = false;
#pragma unroll
          for (int q = 0; q < RG; ++q)
            if (q == rr) valid_rr = row_valid[q];
          if (g.tid == 0) p.part_count[part] = valid_rr ? wrote : 0;
        }
        FP4IDX_STAMP(6);
      }
    });
    FP4IDX_STAMP(0);
    FP4IDX_STAMP_DONE(3);
  }

  // ---- teardown
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc<kTmemCols>(tmem);
  }
}

template <int H, int R, int FMT, int MODE>
cudaError_t launch_score_t(const ScoreParams& p, dim3 grid, cudaStream_t stream) {
  using L = ScoreLayout<H, R, FMT, MODE>;
  const uint32_t want = L::bytes();
  // At least ~120 KB so that one CTA (and one 512-column TMEM allocation) runs per SM.
  const uint32_t bytes = want < 120u * 1024u ? 120u * 1024u : want;
  if (bytes > 232448u) return cudaErrorInvalidConfiguration;
  auto kern = score_kernel<H, R, FMT, MODE>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes));
  if (e != cudaSuccess) return e;
  // programmatic stream serialization: the CTAs may start their on-chip
  // setup while the previous kernel of the stream finishes (pdl_wait orders
  // every global access after it)
  cudaLaunchConfig_t cfg;
  std::memset(&cfg, 0, sizeof(cfg));
  cfg.gridDim = grid;
  cfg.blockDim = dim3(L::kThreads);
  cfg.dynamicSmemBytes = bytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, p);
}

template <int FMT>
cudaError_t launch_score_fmt(const ScoreParams& p, int mode, int heads, dim3 grid, cudaStream_t stream) {
  if (mode == kModeLogits) {
    switch (heads) {
      case 8: return launch_score_t<8, 4, FMT, kModeLogits>(p, grid, stream);
      case 16: return launch_score_t<16, 4, FMT, kModeLogits>(p, grid, stream);
      case 32: return launch_score_t<32, 4, FMT, kModeLogits>(p, grid, stream);
      case 64: return launch_score_t<64, 2, FMT, kModeLogits>(p, grid, stream);
    }
  } else {
    switch (heads) {
      case 8: return launch_score_t<8, 4, FMT, kModeTopk>(p, grid, stream);
      case 16: return launch_score_t<16, 4, FMT, kModeTopk>(p, grid, stream);
      case 32: return launch_score_t<32, 4, FMT, kModeTopk>(p, grid, stream);
      case 64: return launch_score_t<64, 2, FMT, kModeTopk>(p, grid, stream);
    }
  }
  return cudaErrorInvalidValue;
}

}  // namespace fp4idx
