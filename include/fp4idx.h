/*
 * fp4idx.h -- C ABI of the GB300 (sm_103a) FP4 lightning-indexer scorer.
 *
 * The scorer reads FP4 queries and a paged FP4 key cache and computes, for
 * every query row t and logical key position s of its request,
 *
 *     dot(t, h, s)  = sum_{d<128} Q_real[t,h,d] * K_real[s,hk(h),d]
 *     logit(t, s)   = sum_h w[t,h] * max(dot(t,h,s), 0)        (s visible)
 *                   = -inf                                      (s not visible)
 *
 * (CURRENT_ISSUE_FROM_OUTSIDE_CONSULTANT.md, "TL;DR": I[t,s] = sum_h w_h *
 * ReLU(q.K); M3-indexer README, "数学语义": Q_real/K_real are E2M1 values times
 * their block scale, hk = h / (Hq/Hkv)).  Three outputs are offered: the full
 * logits, the per-128-key block max of dot (M3-indexer README, "输出 shape 和
 * 类型"), and the top-k positions of each row.  Around them: the top-k blocks
 * of a block-score tensor, the physical cache slots of selected positions
 * (the sparse-attention consumer's input) and the MXFP4 K-cache writer (the
 * producer of the cache).
 *
 * Formats (M3-indexer README, "FP4 和 scale layout"; SGLang PR 42861,
 * "Modifications"):
 *   FP4IDX_MXFP4: E2M1 codes, one E8M0 scale per 32 values (G = 4 per row of
 *                 128); scale value 2^(code-127), codes 1..254.
 *   FP4IDX_NVFP4: E2M1 codes, one E4M3 scale per 16 values (G = 8), no
 *                 tensor-level global scale; codes 0x00..0x7E.
 * Two E2M1 codes per byte, the low nibble holding the even element.  The
 * head dimension is fixed at 128 (64 bytes of codes per row).
 *
 * Memory and ownership.  Every pointer in fp4idx_problem_t, the weights, the
 * outputs and the workspace are DEVICE pointers owned by the caller; the
 * library never allocates, frees or retains them.  The library reads no
 * device memory on the host and performs no host<->device synchronisation
 * in any call but fp4idx_get_error, so the calls can be captured in a CUDA
 * graph; the device metadata (sequence bounds, block
 * table, visible lengths) is read on the device at run time, so replays see
 * updated contents.
 *
 * Errors.  Argument checks run on the host before any launch and return
 * FP4IDX_EINVAL / FP4IDX_EUNSUPPORTED / FP4IDX_EWORKSPACE without touching
 * the device.  A block-table entry outside [0, num_pages) is found on the
 * device: the keys of that page are treated as invisible and bit
 * FP4IDX_ERR_PAGE_RANGE is set in the device error word; a pipeline wait
 * that exceeds its time limit sets FP4IDX_ERR_TIMEOUT and the kernel returns
 * early.  fp4idx_get_error() reads that word.  No kernel traps.
 * fp4idx_last_error_message() gives a human-readable reason for the last
 * non-OK status returned on the calling thread.
 */
#ifndef FP4IDX_H
#define FP4IDX_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum fp4idx_format {
  FP4IDX_MXFP4 = 0,
  FP4IDX_NVFP4 = 1
} fp4idx_format_t;

typedef enum fp4idx_status {
  FP4IDX_OK = 0,
  FP4IDX_EINVAL = 1,        /* malformed argument: null pointer, size, stride or alignment */
  FP4IDX_EUNSUPPORTED = 2,  /* well-formed but outside what the kernels implement          */
  FP4IDX_EWORKSPACE = 3,    /* workspace missing or smaller than the size query returned   */
  FP4IDX_ECUDA = 4,         /* a CUDA runtime or driver call failed                        */
  FP4IDX_EDEVICE = 5        /* current device is not an sm_103 GPU                         */
} fp4idx_status_t;

/* Bits of the device error word. */
#define FP4IDX_ERR_PAGE_RANGE 0x1u  /* block-table entry outside [0, num_pages)   */
#define FP4IDX_ERR_TIMEOUT    0x2u  /* a pipeline wait exceeded its time limit    */
#define FP4IDX_ERR_TOKEN_TABLE 0x4u /* fp4idx_pages_from_token_table: a page of a
                                       request's slots is not one cache page in
                                       order, or the rows' requests are not
                                       non-decreasing                            */

/* Key-cache layouts (fp4idx_problem_t.kv_layout). */
#define FP4IDX_KV_SPLIT 0  /* k [P][Hkv][page][64] and k_scale [P][Hkv][page][G]     */
#define FP4IDX_KV_FUSED 1  /* one table [P][Hkv][page*(64+G)]: codes, then scales   */

/* Flags of fp4idx_topk. */
#define FP4IDX_TOPK_SORTED 0x1u     /* order each row by (value desc, index asc)  */
#define FP4IDX_TOPK_STREAMING 0x2u  /* fp4idx_topk: always the streaming plan     */

/*
 * The problem: queries, the paged key cache and the visibility rule.
 *
 *   num_seqs B, num_rows T = cu_seqlens_q[B] (host copy supplied by the
 *   caller), num_heads Hq, num_kv_heads Hkv (Hq % Hkv == 0), page_size 64 or
 *   128 tokens, num_pages = physical pages in the cache.
 *
 *   q        [T][Hq][64] bytes, row t at q + t*q_row_stride (q_row_stride a
 *            multiple of 16, >= Hq*64); 128-byte aligned base.
 *   q_scale  [T][Hq][G] bytes, row t at q_scale + t*q_scale_row_stride (>= Hq*G).
 *   k        [num_pages][Hkv][page_size][64] bytes, 128-byte aligned.
 *   k_scale  [num_pages][Hkv][page_size][G] bytes, 16-byte aligned.
 *   cu_seqlens_q, cu_seqlens_k  [B+1] int32 exclusive prefix sums of the
 *            per-request query rows and key counts (M3-indexer README,
 *            "输入 shape 和类型"); k_len[b] bounds the visible keys only.
 *   block_table  logical page j of request b is the physical page
 *            block_table[base(b) + j], base(b) = page_offsets[b] when
 *            page_offsets != NULL (the README's kv_indices + cu_page_offsets
 *            form), else b * table_stride (a [B][table_stride] table).
 *   max_seqlen_q, max_seqlen_k  host upper bounds of q_len[b], k_len[b];
 *            they size grids and outputs and must hold for the device data.
 *
 *   kv_layout  FP4IDX_KV_SPLIT (0): k and k_scale as above.  FP4IDX_KV_FUSED (1):
 *            k is one table of page*(64+G) bytes per (page, K head) --
 *            [num_pages][Hkv][page_size*(64+G)], 128-byte aligned: the page's
 *            64-byte code rows, then its G-byte scale rows -- and k_scale is
 *            unused (SGLang PR 42861, bench_fp4_index_scorer.py: a K table of
 *            PAGE_SIZE * 68 bytes per page; the order inside a page is not
 *            printed there, this is the order read).
 *   cand_mask  NULL, or [T][mask_ld] bytes (mask_ld >= max_seqlen_k): position
 *            s of row t is a candidate only when cand_mask[t*mask_ld + s] != 0;
 *            other positions are -inf in the logits and never selected (the
 *            candidate-mask argument of SGLang PR 42861's fp4_index_logits_paged,
 *            None in its benchmark).  Used by the weighted-ReLU calls
 *            (logits, top-k); fp4idx_block_scores ignores it.
 *
 * Visible keys of row t in request b (q_local = t - cu_seqlens_q[b]):
 *   visible_len != NULL:  vis = clamp(visible_len[t], 0, k_len[b])
 *                          (SGLang PR 42861: a per-row visible length)
 *   causal:               vis = clamp(q_local + off + 1, 0, k_len[b]),
 *                          off = qo_offset ? qo_offset[b] : k_len[b]-q_len[b]
 *                          (M3-indexer README, "数学语义": bottom-right causal)
 *   otherwise:            vis = k_len[b]
 * Positions [0, vis) are visible.  qo_offset with causal == 0 is EINVAL.
 */
typedef struct fp4idx_problem {
  int32_t format;           /* fp4idx_format_t */
  int32_t num_seqs;
  int32_t num_rows;
  int32_t num_heads;
  int32_t num_kv_heads;
  int32_t page_size;
  int64_t num_pages;
  int64_t table_stride;
  int32_t max_seqlen_q;
  int32_t max_seqlen_k;
  const uint8_t* q;
  const uint8_t* q_scale;
  int64_t q_row_stride;
  int64_t q_scale_row_stride;
  const uint8_t* k;
  const uint8_t* k_scale;
  const int32_t* cu_seqlens_q;
  const int32_t* cu_seqlens_k;
  const int32_t* block_table;
  const int32_t* page_offsets;
  const int32_t* visible_len;
  int32_t causal;
  const int32_t* qo_offset;
  int32_t kv_layout;          /* FP4IDX_KV_SPLIT or FP4IDX_KV_FUSED (0 = split) */
  const uint8_t* cand_mask;   /* [T][mask_ld] or NULL */
  int64_t mask_ld;
} fp4idx_problem_t;

/*
 * Full weighted-ReLU logits (CURRENT_ISSUE..., "TL;DR"; SGLang PR 42861,
 * fp4_index_logits_paged: [rows, cap] fp32 with -inf where invisible).
 *   w       [T][Hq] fp32 head weights, row stride w_row_stride floats (>= Hq).
 *   logits  [T][ld] fp32; every column s in [0, ld) of every row is written:
 *           logit(t, s) for s < vis(t), -inf otherwise.  ld % 4 == 0, ld >= 1.
 * Supported: num_kv_heads == 1; num_heads in {8, 16, 32, 64}.
 */
fp4idx_status_t fp4idx_logits(const fp4idx_problem_t* problem, const float* w,
                              int64_t w_row_stride, float* logits, int64_t ld,
                              void* stream);

/*
 * Per-128-key block max of the unweighted dot (M3-indexer README,
 * "数学语义" / "输出 shape 和类型"):
 *   scores[h][kb][t] = max over visible s in [128*kb, 128*kb+128) of dot(t,h,s),
 *                      -inf when the block has no visible key,
 *   for kb < ceil(max_seqlen_k / 128).  scores is [Hq][Ktiles][T] fp32.
 * Supported: Hq/Hkv <= 128 with Hq % Hkv == 0, num_heads <= 128.
 */
fp4idx_status_t fp4idx_block_scores(const fp4idx_problem_t* problem, float* scores,
                                    void* stream);

/*
 * Top-k blocks of every (head, row) column of a block-score tensor (M3-indexer
 * README, "输出 shape 和类型": the block-score call returns the scores only,
 * and a caller that needs a top-k takes it along Ktiles, dim 1).
 *   scores       [Hq][ktiles][T] fp32, device, as written by fp4idx_block_scores.
 *   indices      [Hq][T][k] int32, device: for each (h, t) the block numbers of
 *                the min(k, n) largest scores, n = the blocks of the column
 *                whose score is neither -inf (no visible key) nor NaN; order
 *                (score desc, block asc); -1 after them.
 *   values       [Hq][T][k] fp32 scores of those blocks (-inf padding), or NULL.
 *   valid_count  [Hq][T] int32 = min(k, n), or NULL.
 * Every pointer is caller-owned device memory (4-byte aligned); no workspace,
 * no synchronisation (graph-capturable).  EINVAL for NULL scores / indices or
 * a non-positive size, EUNSUPPORTED for k > 128, or k > 32 with ktiles > 1024.
 * For k <= 32 the scores are read 16 bytes at a time when num_rows is a
 * multiple of 4 and scores is 16-byte aligned, else 4 bytes at a time.
 */
fp4idx_status_t fp4idx_block_topk(const float* scores, int32_t num_heads, int32_t ktiles,
                                  int32_t num_rows, int32_t k, int32_t* indices, float* values,
                                  int32_t* valid_count, void* stream);

/*
 * Top-k positions of each row's logits (CURRENT_ISSUE..., "Fix (production
 * target)": ReLU + per-head weight epilogue followed by a top-k; the output
 * convention is that of a sparse-attention consumer: logical positions, -1
 * padding, a valid count).
 *   indices      [T][k] int32: the min(k, vis(t)) positions with the largest
 *                logits, ties broken by the lower position; -1 after them.
 *                Order: (value desc, index asc) when flags has
 *                FP4IDX_TOPK_SORTED, otherwise unspecified.
 *   values       [T][k] fp32 logits of those positions (-inf padding), or NULL.
 *   valid_count  [T] int32 = min(k, vis(t)), or NULL.  (A position whose
 *                logit is NaN -- only possible with NaN/inf scale codes,
 *                outside the formats' contract -- has no rank and is never
 *                selected; it does not count towards vis(t) here.)
 *   flags        FP4IDX_TOPK_SORTED; FP4IDX_TOPK_STREAMING forces the
 *                streaming plan below (the results are the same).
 *   workspace    device scratch of at least fp4idx_topk_workspace_bytes();
 *                may be NULL when that size is 0.  Contents need no
 *                initialisation and are meaningless after the call.
 * Plans, chosen from host scalars only: short contexts (max_seqlen_k <=
 * 16,384 and T * max_seqlen_k <= 2^24) write the rows' logits into the
 * workspace and select from them; otherwise the scorer keeps a streaming
 * top-k per CTA and a merge selects each row's top-k, so full logits never
 * reach memory.
 * Supported: num_kv_heads == 1; num_heads in {8, 16, 32, 64}; 1 <= k <= 2048.
 * fp4idx_topk_workspace_bytes returns 0 for an invalid problem or a k
 * outside 1..2048 (fp4idx_topk then returns the matching status).
 */
size_t fp4idx_topk_workspace_bytes(const fp4idx_problem_t* problem, int32_t k);
fp4idx_status_t fp4idx_topk(const fp4idx_problem_t* problem, const float* w,
                            int64_t w_row_stride, int32_t k, uint32_t flags,
                            int32_t* indices, float* values, int32_t* valid_count,
                            void* workspace, size_t workspace_bytes, void* stream);

/*
 * The two phases of fp4idx_topk's streaming plan, for callers that schedule
 * them separately (fp4idx_topk with FP4IDX_TOPK_STREAMING is exactly
 * fp4idx_topk_score followed by fp4idx_topk_merge on the same stream,
 * problem, k and workspace).
 *   fp4idx_topk_score  runs the scorer and leaves, in the workspace, a
 *                      superset of the top-k of every row within each CTA's
 *                      share of the keys.
 *   fp4idx_topk_merge  selects each row's exact top-k from those partials and
 *                      writes indices / values / valid_count as fp4idx_topk.
 * The workspace must not be modified between the two calls.
 */
fp4idx_status_t fp4idx_topk_score(const fp4idx_problem_t* problem, const float* w,
                                  int64_t w_row_stride, int32_t k, void* workspace,
                                  size_t workspace_bytes, void* stream);
fp4idx_status_t fp4idx_topk_merge(const fp4idx_problem_t* problem, int32_t k, uint32_t flags,
                                  int32_t* indices, float* values, int32_t* valid_count,
                                  void* workspace, size_t workspace_bytes, void* stream);

/*
 * Full logits and their top-k in one call: fp4idx_logits into the caller's
 * logits [T][ld] (ld >= max_seqlen_k), then each row's exact top-k selected
 * from those logits (same outputs as fp4idx_topk; flags: FP4IDX_TOPK_SORTED).
 * No workspace: the logits are the intermediate.  For a step that needs both
 * outputs (e.g. the verify rows of a short context), one scorer pass
 * instead of two.
 * Supported: as fp4idx_logits and fp4idx_topk.
 */
fp4idx_status_t fp4idx_logits_topk(const fp4idx_problem_t* problem, const float* w,
                                   int64_t w_row_stride, float* logits, int64_t ld, int32_t k,
                                   uint32_t flags, int32_t* indices, float* values,
                                   int32_t* valid_count, void* stream);

/*
 * fp4idx_topk without a caller-supplied workspace, for callers that cannot
 * allocate device memory: an engine that reserved the GPU's memory up front
 * for its own pool (another cudaMalloc fails or fragments it), or a
 * latency-critical loop that cannot take the synchronisation cudaMalloc and
 * cudaFree imply.  The pages describe no such entry point; it exists only
 * for these callers.
 *
 * Results are those of fp4idx_topk (same arguments, minus the workspace).
 * The scratch is a fixed 128 MiB array inside the library's device memory,
 * held by every GPU that loads the library until the process exits.  A
 * problem whose fp4idx_topk_workspace_bytes() exceeds 128 MiB is rejected
 * with FP4IDX_EWORKSPACE before anything runs.  The first call on a device
 * looks up the array's device address (with that device current); make that
 * first call before capturing any stream.  All calls on a device share the
 * one array, so calls that may overlap on the GPU (different streams without
 * ordering between them) race and must be serialised by the caller.  Nothing
 * in it needs clearing between calls.  No memory is allocated or freed.
 */
fp4idx_status_t fp4idx_topk_noalloc(const fp4idx_problem_t* problem, const float* w,
                                    int64_t w_row_stride, int32_t k, uint32_t flags,
                                    int32_t* indices, float* values, int32_t* valid_count,
                                    void* stream);

/*
 * Write keys into the MXFP4 cache (SGLang PR 42861: the benchmark fills the
 * cache with store_fp4_index_k_cache(keys, table, slots, page_size, rne=True);
 * "Modifications": the quantizer clamps E8M0 exponents to 1..254 and the
 * E2M1 level set is [0, 0.5, 1, 1.5, 2, 3, 4, 6]).  The pages do not print
 * the scale rule; this call uses the OCP microscaling one:
 *   per group of 32 values of one (token, K head) row:
 *     code  = clamp(floor(log2(max |x|)) - 2 + 127, 1, 254)   (1 for all zeros)
 *     scale = 2^(code - 127)
 *     each value: x / scale rounded to the nearest E2M1 level, ties to the
 *     even level (round-to-nearest-even on the E2M1 grid), saturating at 6;
 *     sign bit set only for a non-zero level.
 *   keys      [N][Hkv][128] bfloat16 (raw 16-bit words), device; key_row_stride
 *             = elements between consecutive tokens (>= Hkv * 128).  Finite.
 *   slots     [N] int32, device: token i is written at page slots[i] / page_size,
 *             offset slots[i] % page_size of every K head; a negative slot is
 *             skipped; a slot >= num_pages * page_size is skipped and sets
 *             FP4IDX_ERR_PAGE_RANGE.
 *   k, k_scale  the cache of fp4idx_problem_t with format FP4IDX_MXFP4:
 *             [num_pages][Hkv][page_size][64] and [num_pages][Hkv][page_size][4].
 * Graph-capturable, no workspace.  EINVAL on NULL pointers, sizes or
 * misalignment (keys 16-byte aligned with key_row_stride a multiple of 8;
 * k 16-byte aligned), EUNSUPPORTED for page_size other than 64 or 128.
 */
fp4idx_status_t fp4idx_store_k(const uint16_t* keys, int64_t key_row_stride, int32_t num_tokens,
                               int32_t num_kv_heads, const int32_t* slots, int32_t page_size,
                               int64_t num_pages, uint8_t* k, uint8_t* k_scale, void* stream);

/*
 * The MXFP4 K-cache writer of fp4idx_store_k into the fused layout
 * (FP4IDX_KV_FUSED): table is [num_pages][num_kv_heads][page_size * 68] bytes,
 * 16-byte aligned; token i of K head h lands at page slots[i] / page_size,
 * offset o = slots[i] % page_size: its 64 code bytes at o*64 and its 4 scale
 * bytes at page_size*64 + o*4 of the (page, h) block (SGLang PR 42861: its
 * benchmark's writer fills such a table).  Codes, scales, slot rules and errors
 * are those of fp4idx_store_k.
 */
fp4idx_status_t fp4idx_store_k_fused(const uint16_t* keys, int64_t key_row_stride, int32_t num_tokens,
                                     int32_t num_kv_heads, const int32_t* slots, int32_t page_size,
                                     int64_t num_pages, uint8_t* table, void* stream);

/*
 * Quantise bf16 queries to the MXFP4 query operand of fp4idx_problem_t
 * (format FP4IDX_MXFP4).  SGLang PR 42861's fp4_index_logits_paged takes
 * bf16 queries and multiplies them with the dequantised keys; this library
 * runs every contraction on the FP4 tensor cores, so bf16 queries are first
 * quantised here, group by group, by the rule of fp4idx_store_k (E8M0 code
 * clamp(floor(log2 max|x|) - 2 + 127, 1, 254) per 32 values, each value
 * rounded to the nearest E2M1 level, ties to even, saturating at 6).  The
 * scores then differ from the bf16-query ones by at most
 * sum_h |w[t,h]| * sum_d |q - Q(q)|_d * |k_d| (ReLU is 1-Lipschitz).
 *   q        [num_rows][num_heads][128] bfloat16 words, device; q_row_stride =
 *            elements between rows (>= num_heads * 128, a multiple of 8);
 *            16-byte aligned.  Finite.
 *   q_codes  [num_rows][num_heads][64] uint8, device, 16-byte aligned: the
 *            problem's q (two E2M1 codes per byte, low nibble first).
 *   q_scale  [num_rows][num_heads][4] uint8, device: the problem's q_scale.
 * Graph-capturable, no workspace; one launch (none for num_rows == 0).
 * EINVAL on NULL pointers, sizes, strides or misalignment.
 */
fp4idx_status_t fp4idx_quantize_q(const uint16_t* q, int64_t q_row_stride, int32_t num_rows, int32_t num_heads,
                                  uint8_t* q_codes, uint8_t* q_scale, void* stream);

/*
 * This ABI's request metadata from a per-token slot table (SGLang PR 42861,
 * fp4_index_logits_paged's req / req_table arguments):
 *   req        [num_rows] int32, device: the request of each query row; the
 *              rows of a request must be contiguous, requests non-decreasing.
 *   req_table  [num_reqs][req_stride] int32, device: the cache slot (page *
 *              page_size + offset) of every logical position, < 0 for none.
 * Writes, on the device:
 *   cu_seqlens_q  [num_reqs + 1]: rows per request, from req.
 *   cu_seqlens_k  [num_reqs + 1]: keys per request = 1 + the last position
 *              with a slot >= 0 (in a table that passes the checks below).
 *   block_table   [num_reqs][ceil(req_stride / page_size)]: logical page j of
 *              request b is cache page req_table[b][j*page_size] / page_size
 *              when the slots of its positions below the request's key count
 *              are that page's offsets in order (the layout the benchmark's
 *              writer produces); otherwise -1, and FP4IDX_ERR_TOKEN_TABLE is
 *              set (the scorer then treats that page's keys as absent and sets
 *              FP4IDX_ERR_PAGE_RANGE).  Also -1 for a page with no slot.
 *              A position without a slot (< 0) followed, in the same request,
 *              by one with a slot sets FP4IDX_ERR_TOKEN_TABLE as well; with a
 *              reported table the key count is that of one of its pages.
 * A problem with these arrays, table_stride = ceil(req_stride / page_size),
 * max_seqlen_k = req_stride, and the rows' lens as visible_len scores what
 * fp4_index_logits_paged scores.  Graph-capturable; no workspace; two
 * launches.  EINVAL for NULL pointers or non-positive sizes, EUNSUPPORTED for
 * page_size not 64/128, more than 2^31 table entries or more than 524,280
 * pages per request.
 */
fp4idx_status_t fp4idx_pages_from_token_table(const int32_t* req, int32_t num_rows, const int32_t* req_table,
                                              int32_t num_reqs, int64_t req_stride, int32_t page_size,
                                              int64_t num_pages, int32_t* cu_seqlens_q, int32_t* cu_seqlens_k,
                                              int32_t* block_table, void* stream);

/*
 * Physical cache slots of selected positions, for a sparse-attention consumer
 * that gathers K/V rows by slot (vLLM QSA page, _qsa_physical_slots_kernel:
 * each logical token of a row goes through its request's page table once,
 * becoming page << offset_bits | page offset; masked entries and the padding
 * past the selection become -1).
 *   indices   [T][k] int32, device: logical positions of each row (e.g. the
 *             output of fp4idx_topk), -1 for none.
 *   slots     [T][ncols] int32, device: for c < k and s = indices[t][c] with
 *             0 <= s < the key count of t's request and a physical page
 *             p = table(request, s / page_size) in [0, num_pages):
 *                 (p << offset_bits) | (s % page_size);
 *             -1 otherwise, and for every k <= c < ncols.
 *   offset_bits = max(1, bit length of page_size - 1) (6 for 64-key pages, 7
 *             for 128), returned through *offset_bits when not NULL.
 * Requires ncols >= k >= 1, num_pages << offset_bits < 2^31 and at most 65,535
 * rows (EUNSUPPORTED otherwise).  Device metadata is read on the device only; graph-capturable.
 */
fp4idx_status_t fp4idx_topk_slots(const fp4idx_problem_t* problem, const int32_t* indices,
                                  int32_t k, int32_t* slots, int32_t ncols,
                                  int32_t* offset_bits, void* stream);

/*
 * Device error word of the current device (FP4IDX_ERR_* bits).  Synchronises
 * `stream` first; when clear != 0 the word is reset to 0 afterwards.
 */
fp4idx_status_t fp4idx_get_error(uint32_t* bits, int32_t clear, void* stream);

/* Static description of a status code. */
const char* fp4idx_status_string(fp4idx_status_t status);

/* Detail of the last non-OK status returned on this thread ("" if none). */
const char* fp4idx_last_error_message(void);

#ifdef __cplusplus
}
#endif
#endif /* FP4IDX_H */
