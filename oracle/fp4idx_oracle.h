/*
 * fp4idx_oracle.h -- plain CPU oracle for the FP4 lightning-indexer scorer.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may include, link or
 * call this file; only the tests, the package's smoke check and the bench's
 * CPU-baseline arm use it.  It shares no code, header, table or helper with
 * the CUDA library.
 *
 * What it computes (every value in fp64, rounded once to fp32 at the end):
 *   - E2M1 nibble decode through the level set {0,.5,1,1.5,2,3,4,6} with bit 3
 *     as the sign (CURRENT_ISSUE_FROM_OUTSIDE_CONSULTANT.md, "Why it's wrong"
 *     and "Fix (interim)"); the low nibble of a byte is the even element
 *     (M3-indexer README, "输入 shape 和类型": two E2M1 per byte).
 *   - E8M0 scale = 2^(code-127) for the stored codes 1..254 (SGLang PR 42861,
 *     "Modifications" / "Accuracy Tests"); codes 0 and 255 follow that page's
 *     scorer: 0 and +inf.
 *   - E4M3 ("fn") scale per 16 values for NVFP4, no global scale
 *     (M3-indexer README, "FP4 和 scale layout").
 *   - dot(t,h,s) = sum_d Q_real[t,h,d] * K_real[s,hk,d]   (M3-indexer README,
 *     "数学语义"), hk = h / (Hq/Hkv).
 *   - logit(t,s) = sum_h w[t,h] * max(dot(t,h,s), 0) for s < vis(t), else -inf
 *     (CURRENT_ISSUE..., "TL;DR": I[t,s] = sum_h w_h ReLU(q.K)).
 *   - block score = max over visible keys of a 128-key block of dot, -inf when
 *     the block has none (M3-indexer README, "数学语义" / "输出 shape 和类型").
 *   - top-k = full sort of the visible positions by (value desc, index asc),
 *     first k kept, -1 padded; a position whose logit is NaN has no rank and
 *     is not selected.
 *   - SGLang PR 42861's input variants (its benchmark script): the fused K
 *     table of PAGE_SIZE * (64 + G) bytes per page (order inside a page not
 *     printed; read as the page's codes, then its scales), the per-token
 *     slot table req_table[req[t]][s], the optional candidate mask (a
 *     position it clears is not a candidate: -inf, never selected), and
 *     bf16 queries (Q_real = the bf16 value, no block scale).
 *
 * Parity pins: see tests/test_oracle_pins.py (exhaustive decodes, closed forms,
 * library-routine cross-checks, brute-force top-k, invariants).
 */
#ifndef FP4IDX_ORACLE_H
#define FP4IDX_ORACLE_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct orc_problem {
  int32_t format;          /* 0: MXFP4 (E8M0 per 32 values), 1: NVFP4 (E4M3 per 16) */
  int32_t num_seqs;        /* B */
  int32_t num_rows;        /* T (total query rows) */
  int32_t num_heads;       /* Hq */
  int32_t num_kv_heads;    /* Hkv, Hq % Hkv == 0 */
  int32_t page_size;       /* tokens per physical page */
  int64_t num_pages;       /* physical pages in the cache */
  int64_t table_stride;    /* int32 entries per block-table row */
  const uint8_t* q;        /* [T][Hq][64] packed E2M1, row stride q_row_stride bytes */
  const uint8_t* q_scale;  /* [T][Hq][G], row stride q_scale_row_stride bytes */
  int64_t q_row_stride;
  int64_t q_scale_row_stride;
  const uint8_t* k;        /* [P][Hkv][page][64] */
  const uint8_t* k_scale;  /* [P][Hkv][page][G] */
  const int32_t* cu_seqlens_q;  /* [B+1] */
  const int32_t* cu_seqlens_k;  /* [B+1] */
  const int32_t* block_table;   /* logical page j of request b at block_table[base(b)+j] */
  const int32_t* page_offsets;  /* [B] base(b), or NULL for base(b) = b*table_stride */
  const int32_t* visible_len;   /* [T] or NULL */
  int32_t causal;
  const int32_t* qo_offset;     /* [B] or NULL */
  /* SGLang PR 42861's variants of the inputs ("bench_fp4_index_scorer.py":
   * the K table of PAGE_SIZE * 68 bytes per page, req / req_table / lens,
   * the candidate-mask argument, bf16 q). */
  int32_t kv_layout;            /* 0: k and k_scale arrays; 1: fused pages, k only:
                                   [P][Hkv][page*64 code bytes, then page*G scale bytes] */
  const uint8_t* cand_mask;     /* [T][mask_ld] or NULL: position s of row t is a
                                   candidate only when cand_mask[t][s] != 0 */
  int64_t mask_ld;
  const int32_t* req;           /* [T] request of each row, or NULL (cu_seqlens_q rule) */
  const int32_t* req_table;     /* [B][req_stride] cache slot of each logical position
                                   (slot = page*page_size + offset; < 0: no key); with it,
                                   block_table / page_offsets / cu_seqlens_k are unused and
                                   vis(t) = clamp(visible_len[t], 0, req_stride) */
  int64_t req_stride;
  int32_t q_dtype;              /* 0: FP4 codes + scales; 1: bf16 words [T][Hq][128]
                                   (row stride q_row_stride bytes; q_scale unused) */
} orc_problem;

/* element decodes */
double orc_e2m1(uint32_t nibble);
double orc_e8m0(uint32_t code);
double orc_e4m3(uint32_t code);

/* request that owns query row t, and the number of keys that row can see */
int32_t orc_request_of_row(const orc_problem* p, int32_t t);
int64_t orc_visible(const orc_problem* p, int32_t t);

/* One unweighted dot.  abs_sum (nullable) receives sum_d |Q_real*K_real|;
 * safe (nullable) receives 1 when every partial sum of the 128 products, in any
 * order, is exactly representable in fp32. */
double orc_dot(const orc_problem* p, int32_t t, int32_t hq, int64_t s, double* abs_sum, int32_t* safe);

/* Weighted-ReLU logits for the listed rows at the listed positions.
 * out[i*npos+j] = logit(rows[i], pos[j]) (fp32, -inf when invisible).
 * bound (nullable): 1e-5 * sum_h |w| * sum_d |Q*K| (0 for invisible).
 * safe  (nullable): 1 when the result is exact in fp32 under any summation order. */
void orc_logits(const orc_problem* p, const float* w, int64_t w_row_stride,
                const int32_t* rows, int32_t nrows, const int64_t* pos, int64_t npos,
                float* out, double* bound, uint8_t* safe);

/* Full logit rows: out[i*ncols + s] for s in [0, ncols). */
void orc_logits_rows(const orc_problem* p, const float* w, int64_t w_row_stride,
                     const int32_t* rows, int32_t nrows, int64_t ncols,
                     float* out, double* bound, uint8_t* safe);

/* Block max scores for the listed rows, every head and every 128-key block
 * kb < ktiles: out[(h*ktiles + kb)*nrows + i]. */
void orc_block_scores(const orc_problem* p, int32_t ktiles, const int32_t* rows, int32_t nrows,
                      float* out, double* bound, uint8_t* safe);

/* Top-k for the listed rows: idx[i*k+j] (-1 padded), val[i*k+j] (-inf padded,
 * nullable), count[i] = min(k, visible positions with a non-NaN logit)
 * (nullable). */
void orc_topk(const orc_problem* p, const float* w, int64_t w_row_stride, int32_t k,
              const int32_t* rows, int32_t nrows, int32_t* idx, float* val, int32_t* count);

/* Top-k blocks of every (head, row) column of block scores [H][Kt][T]
 * (M3-indexer README, "输出 shape 和类型": a caller that needs a top-k takes it
 * along Ktiles).  A block is a candidate when its score is neither -inf (no
 * visible key) nor NaN; order (score desc, block asc).  idx / val [H][T][k]
 * (-1 / -inf padded; val nullable), count [H][T] = min(k, candidates)
 * (nullable). */
void orc_block_topk(const float* scores, int32_t num_heads, int32_t ktiles, int32_t num_rows, int32_t k,
                    int32_t* idx, float* val, int32_t* count);

/* Physical cache slots of logical positions (vLLM QSA page,
 * _qsa_physical_slots_kernel): for c < k and s = indices[t][c] with
 * 0 <= s < the key count of t's request and page = table(request, s / page)
 * in [0, num_pages): (page << bits) | (s % page_size), bits = max(1, bit
 * length of page_size - 1); -1 otherwise and for k <= c < ncols. */
void orc_topk_slots(const orc_problem* p, const int32_t* indices, int32_t k, int32_t ncols, int32_t* slots);

/* MXFP4 K-cache writer (SGLang PR 42861: store_fp4_index_k_cache with
 * round-to-nearest-even; E8M0 codes clamped to 1..254; the scale rule is the
 * OCP microscaling one, a reading): per 32-value group of a (token, head)
 * row, code = clamp(floor(log2 max|x|) - 2 + 127, 1, 254) (1 for zeros), each
 * value the nearest E2M1 level of |x| / 2^(code-127), ties to the even
 * level, saturating at 6, sign only on a non-zero level.  keys [N][Hkv][128]
 * bf16 words with token stride key_row_stride; token i goes to slot
 * slots[i] (page slot / page_size, offset slot % page_size); negative or
 * out-of-range slots are skipped. */
void orc_store_k(const uint16_t* keys, int64_t key_row_stride, int32_t num_tokens, int32_t num_kv_heads,
                 const int32_t* slots, int32_t page_size, int64_t num_pages, uint8_t* k, uint8_t* k_scale);

/* Number of threads the parallel loops use (1 without OpenMP). */
int32_t orc_num_threads(void);

#ifdef __cplusplus
}
#endif
#endif
