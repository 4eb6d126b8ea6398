/*
 * fp4idx_oracle.c -- plain, slow, obviously correct CPU oracle (fp64).
 *
 * TEST INFRASTRUCTURE ONLY: used by tests/, the package smoke check and the
 * bench's CPU-baseline arm; never by the product path.  No blocking, fusion
 * or reordering beyond the definitions cited in fp4idx_oracle.h.
 */
#include "fp4idx_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define HEAD_DIM 128
#define BLOCK_KEYS 128

/* E2M1 level set, indexed by the three magnitude bits (CURRENT_ISSUE...,
 * "Why it's wrong": [0, 0.5, 1, 1.5, 2, 3, 4, 6]). */
static const double kE2M1Levels[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};

double orc_e2m1(uint32_t nibble) {
  double mag = kE2M1Levels[nibble & 7u];
  return (nibble & 8u) ? -mag : mag;
}

/* SGLang PR 42861, "Modifications": stored codes 1..254 are 2^(code-127);
 * the scorer decodes code 0 to 0 and code 255 to inf ("Accuracy Tests"). */
double orc_e8m0(uint32_t code) {
  code &= 0xFFu;
  if (code == 0u) return 0.0;
  if (code == 255u) return INFINITY;
  return ldexp(1.0, (int)code - 127);
}

/* E4M3 "fn": 1 sign, 4 exponent (bias 7), 3 mantissa bits; exponent 0 is
 * subnormal (m/8 * 2^-6); S.1111.111 is NaN; no infinities. */
double orc_e4m3(uint32_t code) {
  code &= 0xFFu;
  uint32_t sign = code >> 7, e = (code >> 3) & 15u, m = code & 7u;
  double v;
  if (e == 15u && m == 7u) return NAN;
  if (e == 0u)
    v = ldexp((double)m / 8.0, -6);
  else
    v = ldexp(1.0 + (double)m / 8.0, (int)e - 7);
  return sign ? -v : v;
}

static int group_size(const orc_problem* p) { return p->format == 0 ? 32 : 16; }
static int num_groups(const orc_problem* p) { return HEAD_DIM / group_size(p); }
static double scale_value(const orc_problem* p, uint8_t code) {
  return p->format == 0 ? orc_e8m0(code) : orc_e4m3(code);
}

int32_t orc_request_of_row(const orc_problem* p, int32_t t) {
  if (p->req) {  /* per-token table: the row's request is given */
    int32_t b = p->req[t];
    return (b >= 0 && b < p->num_seqs) ? b : -1;
  }
  for (int32_t b = 0; b < p->num_seqs; ++b)
    if (t >= p->cu_seqlens_q[b] && t < p->cu_seqlens_q[b + 1]) return b;
  return -1;
}

/* Visible key count of row t (M3-indexer README "数学语义": bottom-right causal
 * alignment, offset = k_len - q_len unless qo_offset is given; SGLang PR
 * 42861: a per-row visible length).  Positions [0, vis) are visible. */
int64_t orc_visible(const orc_problem* p, int32_t t) {
  int32_t b = orc_request_of_row(p, t);
  if (b < 0) return 0;
  if (p->req_table) {  /* per-token table: lens, clipped to the table width */
    int64_t v = p->visible_len ? p->visible_len[t] : p->req_stride;
    if (v < 0) v = 0;
    if (v > p->req_stride) v = p->req_stride;
    return v;
  }
  int64_t q_len = p->cu_seqlens_q[b + 1] - p->cu_seqlens_q[b];
  int64_t k_len = p->cu_seqlens_k[b + 1] - p->cu_seqlens_k[b];
  int64_t q_local = t - p->cu_seqlens_q[b];
  int64_t vis;
  if (p->visible_len) {
    vis = p->visible_len[t];
  } else if (p->causal) {
    int64_t off = p->qo_offset ? p->qo_offset[b] : k_len - q_len;
    vis = q_local + off + 1;
  } else {
    vis = k_len;
  }
  if (vis < 0) vis = 0;
  if (vis > k_len) vis = k_len;
  return vis;
}

/* Largest power of two dividing the nonzero double x. */
static double lsb_weight(double x) {
  int e;
  double m = frexp(fabs(x), &e);
  uint64_t mant = (uint64_t)ldexp(m, 53);
  int tz = 0;
  while (((mant >> tz) & 1u) == 0u) ++tz;
  return ldexp(1.0, e - 53 + tz);
}

/* A sum of exact terms is exact in fp32 under every order when all terms are
 * multiples of the smallest term granularity g and sum|terms| < 2^24 * g. */
typedef struct {
  double abs_sum;
  double min_lsb;
  int all_finite;
} exact_tracker;

static void tracker_init(exact_tracker* tr) {
  tr->abs_sum = 0.0;
  tr->min_lsb = INFINITY;
  tr->all_finite = 1;
}
static void tracker_add(exact_tracker* tr, double term) {
  if (!isfinite(term)) {
    tr->all_finite = 0;
    return;
  }
  if (term == 0.0) return;
  tr->abs_sum += fabs(term);
  double g = lsb_weight(term);
  if (g < tr->min_lsb) tr->min_lsb = g;
}
static int tracker_safe(const exact_tracker* tr) {
  if (!tr->all_finite) return 0;
  if (tr->abs_sum == 0.0) return 1;
  return tr->abs_sum < ldexp(tr->min_lsb, 24);
}

/* value of a bfloat16 word from its fields: (-1)^s 2^(e-127) (1 + m/128), or
 * (-1)^s 2^-126 m/128 for e = 0 */
static double bf16_value(uint16_t w) {
  const int s = w >> 15, e = (w >> 7) & 0xFF, m = w & 0x7F;
  double v;
  if (e == 0) v = ldexp((double)m / 128.0, -126);
  else if (e == 255) v = m ? NAN : INFINITY;
  else v = ldexp(1.0 + (double)m / 128.0, e - 127);
  return s ? -v : v;
}

/* Codes and scales of key s (request b, kv head hk) inside the paged cache;
 * 0 when position s has no key (a per-token table entry < 0 or a page
 * outside the cache). */
static int key_addr(const orc_problem* p, int32_t b, int32_t hk, int64_t s, const uint8_t** codes,
                    const uint8_t** scales) {
  const int G = num_groups(p);
  int64_t page, token;
  if (p->req_table) {
    int64_t slot = p->req_table[(int64_t)b * p->req_stride + s];
    if (slot < 0) return 0;
    page = slot / p->page_size;
    token = slot % p->page_size;
  } else {
    int64_t base = p->page_offsets ? (int64_t)p->page_offsets[b] : (int64_t)b * p->table_stride;
    page = p->block_table[base + s / p->page_size];
    token = s % p->page_size;
  }
  if (page < 0 || page >= p->num_pages) return 0;
  int64_t block = page * p->num_kv_heads + hk;  /* one (page, K head) */
  if (p->kv_layout == 1) {
    const uint8_t* pg = p->k + block * (int64_t)p->page_size * (64 + G);
    *codes = pg + token * 64;
    *scales = pg + (int64_t)p->page_size * 64 + token * G;
  } else {
    int64_t row = block * p->page_size + token;
    *codes = p->k + row * 64;
    *scales = p->k_scale + row * G;
  }
  return 1;
}

/* Whether position s of row t holds a key the row may select: visible, in
 * the cache, and not cleared by the candidate mask. */
static int is_candidate(const orc_problem* p, int32_t t, int64_t s, int64_t vis) {
  if (s >= vis) return 0;
  if (p->cand_mask && p->cand_mask[(int64_t)t * p->mask_ld + s] == 0) return 0;
  const uint8_t *c, *sc;
  return key_addr(p, orc_request_of_row(p, t), 0, s, &c, &sc);
}


double orc_dot(const orc_problem* p, int32_t t, int32_t hq, int64_t s, double* abs_sum, int32_t* safe) {
  const int G = num_groups(p), S = group_size(p);
  int32_t b = orc_request_of_row(p, t);
  int32_t hk = hq / (p->num_heads / p->num_kv_heads);
  const uint8_t *kc = NULL, *ks = NULL;
  if (b < 0 || !key_addr(p, b, hk, s, &kc, &ks)) {  /* no key at s */
    if (abs_sum) *abs_sum = 0.0;
    if (safe) *safe = 1;
    return NAN;
  }
  const uint8_t* qc = p->q + (int64_t)t * p->q_row_stride + (int64_t)hq * (p->q_dtype == 1 ? 256 : 64);
  const uint8_t* qs = p->q_dtype == 1 ? NULL : p->q_scale + (int64_t)t * p->q_scale_row_stride + (int64_t)hq * G;
  exact_tracker tr;
  tracker_init(&tr);
  double sum = 0.0, asum = 0.0;
  for (int d = 0; d < HEAD_DIM; ++d) {
    uint32_t qn = (d & 1) ? (qc[d >> 1] >> 4) : (qc[d >> 1] & 15u);
    uint32_t kn = (d & 1) ? (kc[d >> 1] >> 4) : (kc[d >> 1] & 15u);
    double qr;
    if (p->q_dtype == 1) {
      uint16_t wq;
      memcpy(&wq, qc + 2 * d, sizeof(wq));
      qr = bf16_value(wq);
    } else {
      qr = orc_e2m1(qn) * scale_value(p, qs[d / S]);
    }
    double kr = orc_e2m1(kn) * scale_value(p, ks[d / S]);
    double prod = qr * kr;
    sum += prod;
    asum += fabs(prod);
    tracker_add(&tr, prod);
  }
  if (abs_sum) *abs_sum = asum;
  if (safe) *safe = tracker_safe(&tr);
  return sum;
}

/* One weighted-ReLU logit in fp64 with its bound and exactness flag. */
static float logit_one(const orc_problem* p, const float* w, int64_t w_row_stride, int32_t t,
                       int64_t s, int64_t vis, double* bound, uint8_t* safe) {
  if (!is_candidate(p, t, s, vis)) {
    if (bound) *bound = 0.0;
    if (safe) *safe = 1;
    return -INFINITY;
  }
  exact_tracker tr;
  tracker_init(&tr);
  int all_dots_safe = 1;
  double acc = 0.0, bnd = 0.0;
  for (int32_t h = 0; h < p->num_heads; ++h) {
    double asum;
    int32_t dsafe;
    double dot = orc_dot(p, t, h, s, &asum, &dsafe);
    double wh = (double)w[(int64_t)t * w_row_stride + h];
    /* ReLU; a NaN dot stays NaN. */
    double relu = dot > 0.0 ? dot : 0.0;
    if (isnan(dot)) relu = dot;
    double term = wh * relu;
    acc += term;
    bnd += fabs(wh) * asum;
    all_dots_safe &= dsafe;
    tracker_add(&tr, term);
  }
  if (bound) *bound = 1e-5 * bnd;
  if (safe) *safe = (uint8_t)(all_dots_safe && tracker_safe(&tr));
  return (float)acc;
}

void orc_logits(const orc_problem* p, const float* w, int64_t w_row_stride, const int32_t* rows,
                int32_t nrows, const int64_t* pos, int64_t npos, float* out, double* bound,
                uint8_t* safe) {
  for (int32_t i = 0; i < nrows; ++i) {
    int32_t t = rows[i];
    int64_t vis = orc_visible(p, t);
#pragma omp parallel for schedule(dynamic, 64)
    for (int64_t j = 0; j < npos; ++j) {
      int64_t o = (int64_t)i * npos + j;
      out[o] = logit_one(p, w, w_row_stride, t, pos[j], vis, bound ? &bound[o] : NULL,
                         safe ? &safe[o] : NULL);
    }
  }
}

void orc_logits_rows(const orc_problem* p, const float* w, int64_t w_row_stride,
                     const int32_t* rows, int32_t nrows, int64_t ncols, float* out, double* bound,
                     uint8_t* safe) {
  for (int32_t i = 0; i < nrows; ++i) {
    int32_t t = rows[i];
    int64_t vis = orc_visible(p, t);
#pragma omp parallel for schedule(dynamic, 64)
    for (int64_t s = 0; s < ncols; ++s) {
      int64_t o = (int64_t)i * ncols + s;
      out[o] = logit_one(p, w, w_row_stride, t, s, vis, bound ? &bound[o] : NULL,
                         safe ? &safe[o] : NULL);
    }
  }
}

void orc_block_scores(const orc_problem* p, int32_t ktiles, const int32_t* rows, int32_t nrows,
                      float* out, double* bound, uint8_t* safe) {
  const int32_t H = p->num_heads;
#pragma omp parallel for collapse(2) schedule(dynamic, 4)
  for (int32_t i = 0; i < nrows; ++i) {
    for (int32_t h = 0; h < H; ++h) {
      int32_t t = rows[i];
      int64_t vis = orc_visible(p, t);
      for (int32_t kb = 0; kb < ktiles; ++kb) {
        double best = -INFINITY, bnd = 0.0;
        int found = 0, all_safe = 1;
        for (int64_t s = (int64_t)kb * BLOCK_KEYS; s < (int64_t)(kb + 1) * BLOCK_KEYS && s < vis; ++s) {
          const uint8_t *kc, *ks;
          if (!key_addr(p, orc_request_of_row(p, t), h / (H / p->num_kv_heads), s, &kc, &ks)) continue;
          double asum;
          int32_t dsafe;
          double dot = orc_dot(p, t, h, s, &asum, &dsafe);
          /* NaN propagates through the max, as through the ReLU. */
          if (!isnan(best) && (!found || isnan(dot) || dot > best)) best = dot;
          found = 1;
          if (asum > bnd) bnd = asum;
          all_safe &= dsafe;
        }
        int64_t o = ((int64_t)h * ktiles + kb) * nrows + i;
        out[o] = (float)best;
        if (bound) bound[o] = 1e-5 * bnd;
        if (safe) safe[o] = (uint8_t)all_safe;
      }
    }
  }
}

/* Total order of the selection: value descending (with -0 == +0), then
 * logical index ascending. */
typedef struct {
  float value;
  int64_t index;
} scored_pos;

static int cmp_scored(const void* a, const void* b) {
  const scored_pos* x = (const scored_pos*)a;
  const scored_pos* y = (const scored_pos*)b;
  if (x->value > y->value) return -1;
  if (x->value < y->value) return 1;
  if (x->index < y->index) return -1;
  if (x->index > y->index) return 1;
  return 0;
}

void orc_topk(const orc_problem* p, const float* w, int64_t w_row_stride, int32_t k,
              const int32_t* rows, int32_t nrows, int32_t* idx, float* val, int32_t* count) {
  for (int32_t i = 0; i < nrows; ++i) {
    int32_t t = rows[i];
    int64_t vis = orc_visible(p, t);
    scored_pos* all = (scored_pos*)malloc(sizeof(scored_pos) * (size_t)(vis > 0 ? vis : 1));
#pragma omp parallel for schedule(dynamic, 64)
    for (int64_t s = 0; s < vis; ++s) {
      all[s].value = logit_one(p, w, w_row_stride, t, s, vis, NULL, NULL);
      all[s].index = s;
    }
    /* A NaN logit has no place in the order: such positions are not selected;
     * neither are positions that are not candidates (no key, or cleared by
     * the candidate mask: their logit is -inf by definition, not a value). */
    int64_t m = 0;
    for (int64_t s = 0; s < vis; ++s)
      if (!isnan(all[s].value) && is_candidate(p, t, s, vis)) all[m++] = all[s];
    qsort(all, (size_t)m, sizeof(scored_pos), cmp_scored);
    int64_t n = m < k ? m : k;
    for (int64_t j = 0; j < k; ++j) {
      idx[(int64_t)i * k + j] = j < n ? (int32_t)all[j].index : -1;
      if (val) val[(int64_t)i * k + j] = j < n ? all[j].value : -INFINITY;
    }
    if (count) count[i] = (int32_t)n;
    free(all);
  }
}

void orc_block_topk(const float* scores, int32_t num_heads, int32_t ktiles, int32_t num_rows, int32_t k,
                    int32_t* idx, float* val, int32_t* count) {
  const int64_t cols = (int64_t)num_heads * num_rows;
#pragma omp parallel
  {
    unsigned char* taken = (unsigned char*)malloc((size_t)ktiles);
#pragma omp for schedule(dynamic, 64)
    for (int64_t c = 0; c < cols; ++c) {
      const int64_t h = c / num_rows, t = c % num_rows;
      memset(taken, 0, (size_t)ktiles);
      int32_t n = 0;
      /* k rounds of "the best remaining candidate": the largest score, the
       * lowest block among equal scores; -inf and NaN are not candidates */
      for (int32_t r = 0; r < k; ++r) {
        int32_t best = -1;
        float bv = 0.0f;
        for (int32_t b = 0; b < ktiles; ++b) {
          const float v = scores[(h * ktiles + b) * num_rows + t];
          if (taken[b] || isnan(v) || v == -INFINITY) continue;
          if (best < 0 || v > bv) {
            best = b;
            bv = v;
          }
        }
        idx[c * k + r] = best;
        if (val) val[c * k + r] = best >= 0 ? bv : -INFINITY;
        if (best >= 0) {
          taken[best] = 1;
          ++n;
        }
      }
      if (count) count[c] = n;
    }
    free(taken);
  }
}

void orc_topk_slots(const orc_problem* p, const int32_t* indices, int32_t k, int32_t ncols, int32_t* slots) {
  int32_t bits = 1;
  while ((1 << bits) < p->page_size) ++bits;
  for (int32_t t = 0; t < p->num_rows; ++t) {
    const int32_t b = orc_request_of_row(p, t);
    const int64_t k_len = (int64_t)p->cu_seqlens_k[b + 1] - p->cu_seqlens_k[b];
    for (int32_t c = 0; c < ncols; ++c) {
      int32_t slot = -1;
      if (c < k) {
        const int64_t s = indices[(int64_t)t * k + c];
        if (s >= 0 && s < k_len) {
          const int64_t base = p->page_offsets ? (int64_t)p->page_offsets[b] : (int64_t)b * p->table_stride;
          const int64_t page = p->block_table[base + s / p->page_size];
          if (page >= 0 && page < p->num_pages) slot = (int32_t)((page << bits) | (s % p->page_size));
        }
      }
      slots[(int64_t)t * ncols + c] = slot;
    }
  }
}


void orc_store_k(const uint16_t* keys, int64_t key_row_stride, int32_t num_tokens, int32_t num_kv_heads,
                 const int32_t* slots, int32_t page_size, int64_t num_pages, uint8_t* k, uint8_t* k_scale) {
  for (int32_t i = 0; i < num_tokens; ++i) {
    const int64_t slot = slots[i];
    if (slot < 0 || slot >= num_pages * page_size) continue;
    for (int32_t h = 0; h < num_kv_heads; ++h) {
      const int64_t crow = ((slot / page_size) * num_kv_heads + h) * page_size + slot % page_size;
      for (int g = 0; g < 4; ++g) {
        double x[32], amax = 0.0;
        for (int j = 0; j < 32; ++j) {
          x[j] = bf16_value(keys[i * key_row_stride + h * 128 + g * 32 + j]);
          if (fabs(x[j]) > amax) amax = fabs(x[j]);
        }
        /* shared exponent: floor(log2(amax)) minus E2M1's largest exponent (2) */
        int code = 1;
        if (amax > 0.0) {
          int ex;
          frexp(amax, &ex); /* amax = f 2^ex, f in [0.5, 1): floor(log2 amax) = ex - 1 */
          code = ex - 1 - 2 + 127;
          if (code < 1) code = 1;
          if (code > 254) code = 254;
        }
        const double scale = ldexp(1.0, code - 127);
        k_scale[crow * 4 + g] = (uint8_t)code;
        for (int j = 0; j < 32; j += 2) {
          uint8_t byte = 0;
          for (int u = 0; u < 2; ++u) {
            const double y = fabs(x[j + u]) / scale;
            /* nearest E2M1 level; on a tie the level with the even index */
            int best = 0;
            for (int l = 1; l < 8; ++l) {
              const double d = fabs(y - kE2M1Levels[l]), db = fabs(y - kE2M1Levels[best]);
              if (d < db || (d == db && (l & 1) == 0)) best = l;
            }
            const int nib = best | ((x[j + u] < 0.0 && best != 0) ? 8 : 0);
            byte |= (uint8_t)(nib << (4 * u));
          }
          k[crow * 64 + g * 16 + j / 2] = byte;
        }
      }
    }
  }
}

int32_t orc_num_threads(void) {
#ifdef _OPENMP
  return (int32_t)omp_get_max_threads();
#else
  return 1;
#endif
}
