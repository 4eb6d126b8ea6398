// internal.h -- launch parameters shared by the host layer (api.cu) and the
// kernel translation units.  Not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace fp4idx {

constexpr int kHeadDim = 128;
constexpr int kTileKeys = 128;       // keys per MMA tile (M of the scorer MMA)
constexpr int kCodeBytes = 64;       // packed E2M1 bytes per 128-value row

enum Mode : int { kModeLogits = 0, kModeTopk = 1 };

// Keys-on-M scorer: one CTA owns up to R query rows of one request (the MMA
// N dimension is R*H) and a contiguous chunk of 128-key tiles.
struct ScoreParams {
  CUtensorMap tmap_q;   // 3D {64 B, Hq, T}, box {64, H, R}, 64B swizzle
  // codes of (page, K head) block z: page*64 bytes at kcode_base + z * kcode_block_stride
  const uint8_t* kcode_base;
  int64_t kcode_block_stride;
  // scales of (page, K head) block z: page*G bytes at kscale_base + z * kscale_block_stride
  // (separate scale array, or the scale rows of a fused page)
  const uint8_t* kscale_base;
  int64_t kscale_block_stride;
  const uint8_t* cand_mask;  // [T][mask_ld] or nullptr: 0 = not a candidate
  int64_t mask_ld;
  const uint8_t* q_scale;
  int64_t q_scale_row_stride;
  const int32_t* cu_seqlens_q;
  const int32_t* cu_seqlens_k;
  const int32_t* block_table;
  const int32_t* page_offsets;
  int64_t table_stride;
  const int32_t* visible_len;
  const int32_t* qo_offset;
  int32_t causal;
  int32_t page_size;
  int32_t page_shift;       // log2(page_size)
  int64_t num_pages;
  int32_t num_rows;
  int32_t num_heads;
  int32_t num_seqs;
  int32_t row_groups;       // ceil(max_seqlen_q / R) row groups per request
  int32_t max_seqlen_k;     // host bound of every request's key count
  const float* w;
  int64_t w_row_stride;
  int32_t total_tiles;      // logits: output tiles per row group, ceil(ld / 128)
  int32_t uniform_items;    // logits: 1 when every item is known (on the host) to hold
                            // total_tiles tiles, so a CTA plans its chunk without device reads
  int32_t score_ctas;       // grid size of the scorer launch
  // logits output
  float* logits;
  int64_t ld;
  // top-k partials: slot s (s < score_ctas: first segment of CTA s; else
  // score_ctas + item: an item that starts inside a CTA's chunk) x R rows,
  // up to topk_part_capacity(k) keys each (a superset of that slot's top-k).
  int32_t k;
  uint64_t* part_keys;      // [slots * R][topk_part_capacity(k)]
  int32_t* part_count;      // [slots * R]
  uint64_t* cand;           // [score_ctas * R][candidate capacity] streaming candidate buffers
  int32_t* item_start;      // [items + 1] first unit of each item, total last (top-k only)
  // Work units of an item with tiles: its tiles plus this many units that
  // stand for the per-item cost (Q load, weights, flush), so that the equal
  // split of the concatenated units balances CTAs with many short items
  // against CTAs with a few long ones (0: tiles only).
  int32_t item_overhead;
  // Pooled bucket counts of every row (top-k with four-row CTAs and at most
  // kPoolMaxRows rows; nullptr otherwise), zeroed before the launch:
  // pool_hist[t][b] = keys of row t that some CTA appended in bucket b,
  // pool_top[t] = the highest such bucket.
  uint32_t* pool_hist;
  uint32_t* pool_top;
  uint32_t* err;
};

// Merge of the per-CTA top-k partials of each row into the final output.
struct MergeParams {
  ScoreParams sp;
  int32_t rows_per_cta;
  uint32_t flags;
  int32_t* indices;
  float* values;
  int32_t* valid_count;
};

// Queries-on-M block scorer: one item = (request b, K head hk, RT query
// rows); its M = 128 MMA rows are the g = Hq/Hkv heads of group hk x RT rows
// (row m = h_local * RT + t_local, RT = 128 / g).  Tiles are the item's
// 128-key blocks; the tiles of all items are split evenly across CTAs.
struct BlockParams {
  CUtensorMap tmap_k;   // 3D {64 B, page, num_pages*Hkv blocks}, box {64, page, 1}, 64B swizzle
  CUtensorMap tmap_q;   // 3D {64 B, T (q_row_stride), Hq (64 B)}, box {64, RT, g}, 64B swizzle
  const uint8_t* kscale_base;  // as ScoreParams
  int64_t kscale_block_stride;
  const uint8_t* q_scale;
  int64_t q_scale_row_stride;
  const int32_t* cu_seqlens_q;
  const int32_t* cu_seqlens_k;
  const int32_t* block_table;
  const int32_t* page_offsets;
  int64_t table_stride;
  const int32_t* visible_len;
  const int32_t* qo_offset;
  int32_t causal;
  int32_t page_size;
  int32_t page_shift;
  int64_t num_pages;
  int32_t num_rows;
  int32_t num_heads;
  int32_t num_kv_heads;
  int32_t num_seqs;
  int32_t group_shift;  // log2(Hq / Hkv)
  int32_t rt_shift;     // log2(RT) = 7 - group_shift
  int32_t row_tiles;    // ceil(max_seqlen_q / RT)
  int32_t ktiles;       // output blocks per (head, row): ceil(max_seqlen_k / 128)
  float* scores;        // [Hq][ktiles][T]
  uint32_t* err;
};

// Launchers (defined in the kernel translation units).  Return cudaSuccess
// or the launch error.
cudaError_t launch_score_mx(const ScoreParams& p, int mode, int heads, dim3 grid, cudaStream_t stream);
cudaError_t launch_score_nv(const ScoreParams& p, int mode, int heads, dim3 grid, cudaStream_t stream);
inline cudaError_t launch_score(const ScoreParams& p, int format, int mode, int heads, dim3 grid,
                                cudaStream_t stream) {
  return format == 0 ? launch_score_mx(p, mode, heads, grid, stream)
                     : launch_score_nv(p, mode, heads, grid, stream);
}
// Partial lists one row can have: at most one per scorer CTA.
constexpr int kMaxMergeSlots = 256;
// many_rows: the small-shared-memory variant (several CTAs per SM).
cudaError_t launch_topk_merge(const MergeParams& p, int rows, bool many_rows, cudaStream_t stream);
// Exact top-k of each row from p.sp.logits [T][p.sp.ld] (visibility from the problem).
cudaError_t launch_topk_select(const MergeParams& p, int rows, cudaStream_t stream);
cudaError_t launch_block_scores(const BlockParams& p, int format, dim3 grid, cudaStream_t stream);
// MXFP4 K-cache writer (fp4idx_store_k, fp4idx_store_k_fused) and query
// quantiser (fp4idx_quantize_q: no slots, one-token pages).
struct StoreParams {
  const uint16_t* keys;     // [N][Hkv][128] bf16 words, token stride key_row_stride
  int64_t key_row_stride;
  const int32_t* slots;     // [N], or nullptr: token i at slot i
  uint8_t* k;               // [P][Hkv][page][64], or the fused table [P][Hkv][page*68]
  uint8_t* k_scale;         // [P][Hkv][page][4] (nullptr with the fused table)
  int32_t fused;
  int64_t num_pages;
  int32_t num_tokens;
  int32_t num_kv_heads;
  int32_t page_size;
  uint32_t* err;
};
cudaError_t launch_store_k(const StoreParams& p, cudaStream_t stream);

// Physical slots of selected positions (fp4idx_topk_slots).
struct SlotParams {
  const int32_t* indices;   // [T][k]
  int32_t* slots;           // [T][ncols]
  const int32_t* cu_seqlens_q;
  const int32_t* cu_seqlens_k;
  const int32_t* block_table;
  const int32_t* page_offsets;
  int64_t table_stride;
  int32_t num_seqs;
  int32_t num_pages;
  int32_t page_size;
  int32_t page_shift;
  int32_t offset_bits;
  int32_t k;
  int32_t ncols;
};
cudaError_t launch_topk_slots(const SlotParams& p, int32_t rows, cudaStream_t stream);

// Top-k blocks of each (head, row) column of [H][Kt][T] block scores, k <= 32.
cudaError_t launch_block_topk(const float* scores, int32_t H, int32_t Kt, int32_t T, int32_t k, int32_t* indices,
                              float* values, int32_t* valid_count, int sms, cudaStream_t stream);

// Cache metadata of a per-token slot table (fp4idx_pages_from_token_table).
struct TokenTableParams {
  const int32_t* req;        // [T]
  const int32_t* req_table;  // [B][req_stride]
  int64_t req_stride;
  int32_t num_rows;
  int32_t num_reqs;
  int32_t page_size;
  int64_t num_pages;
  int32_t* cu_seqlens_q;     // [B+1]
  int32_t* cu_seqlens_k;     // [B+1]
  int32_t* block_table;      // [B][pages per request]
  int32_t table_pages;       // ceil(req_stride / page_size)
  uint32_t* err;
};
cudaError_t launch_token_table(const TokenTableParams& p, cudaStream_t stream);

// Sets the message fp4idx_last_error_message() returns on this thread.
void set_last_error(const char* fmt, ...);

constexpr int kPoolMaxRows = 2048;
constexpr int kPoolBins = 2048;  // the streaming top-k's bucket count (kHistBins)

// Twice k rounded to whole tiles, at least 1,024.
__host__ __device__ constexpr int topk_capacity(int k) {
  return 2 * ((k + 127) / 128) * 128 < 1024 ? 1024 : 2 * ((k + 127) / 128) * 128;
}
// Keys a scorer CTA's streaming candidate buffer holds per row when it lives
// in the workspace: four times k (rounded), so a buffer is compacted only
// after about three times k insertions.
__host__ __device__ constexpr int topk_cand_capacity(int k) { return 2 * topk_capacity(k); }
// Keys of one partial list: a scorer CTA writes a row's whole candidate
// buffer there (no selection in the scorer), so a list holds as many keys
// as the largest candidate buffer (shared memory 8,192, or the workspace
// buffer).
__host__ __device__ constexpr int topk_part_capacity(int k) {
  return topk_cand_capacity(k) > 8192 ? topk_cand_capacity(k) : 8192;
}
// Work units (128-key tiles) standing for one item's fixed cost -- its
// setup and the flush of its candidates -- in the top-k scorer's split
// (measured: 12 balances the causal prefill, whose items range from one
// tile to 256; long decode items are indifferent to it).
constexpr int kTopkItemOverhead = 12;

// Query rows per scorer CTA for a head count (the MMA N is rows * heads).
inline int score_rows_per_cta(int heads) { return heads >= 64 ? 2 : 4; }

}  // namespace fp4idx
