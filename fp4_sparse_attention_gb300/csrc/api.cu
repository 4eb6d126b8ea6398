// api.cu -- the C ABI of include/fp4idx.h: host-side argument checks, TMA
// tensor-map construction, launch planning and kernel launches.  Nothing here
// reads device memory or synchronises (except fp4idx_get_error).
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "fp4idx.h"
#include "internal.h"

namespace fp4idx {
namespace {

thread_local char g_msg[512] = "";

fp4idx_status_t fail(fp4idx_status_t s, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_msg, sizeof(g_msg), fmt, ap);
  va_end(ap);
  return s;
}

fp4idx_status_t cuda_fail(cudaError_t e, const char* what) {
  return fail(FP4IDX_ECUDA, "%s: %s", what, cudaGetErrorString(e));
}

// Device error word: one per device that loads this library.
__device__ uint32_t g_device_error;

struct DeviceInfo {
  bool ready = false;
  int major = 0, minor = 0, sms = 0;
  uint32_t* err = nullptr;
};
constexpr int kMaxDevices = 64;
DeviceInfo g_dev[kMaxDevices];
std::mutex g_dev_mutex;

fp4idx_status_t device_info(DeviceInfo** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return fail(FP4IDX_EDEVICE, "device ordinal %d out of range", dev);
  std::lock_guard<std::mutex> lock(g_dev_mutex);
  DeviceInfo& d = g_dev[dev];
  if (!d.ready) {
    if ((e = cudaDeviceGetAttribute(&d.major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&d.minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
      return cuda_fail(e, "cudaDeviceGetAttribute");
    if (d.major != 10 || d.minor != 3)
      return fail(FP4IDX_EDEVICE, "device %d is sm_%d%d; this library is built for sm_103a", dev, d.major,
                  d.minor);
    void* ptr = nullptr;
    if ((e = cudaGetSymbolAddress(&ptr, g_device_error)) != cudaSuccess)
      return cuda_fail(e, "cudaGetSymbolAddress(error word)");
    d.err = static_cast<uint32_t*>(ptr);
    d.ready = true;
  }
  *out = &d;
  return FP4IDX_OK;
}

// cuTensorMapEncodeTiled through the runtime's driver entry point.
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

fp4idx_status_t encode_fn(EncodeTiledFn* out) {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  static cudaError_t err = cudaSuccess;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    err = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q);
    if (err == cudaSuccess && q == cudaDriverEntryPointSuccess) fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  if (!fn) return fail(FP4IDX_ECUDA, "cuTensorMapEncodeTiled unavailable (%s)", cudaGetErrorString(err));
  *out = fn;
  return FP4IDX_OK;
}

fp4idx_status_t make_tmap(CUtensorMap* m, const void* base, int rank, const cuuint64_t* dims,
                          const cuuint64_t* strides, const cuuint32_t* box) {
  EncodeTiledFn fn;
  fp4idx_status_t s = encode_fn(&fn);
  if (s != FP4IDX_OK) return s;
  cuuint32_t elem[4] = {1, 1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, rank, const_cast<void*>(base), dims, strides, box, elem,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(FP4IDX_EINVAL, "cuTensorMapEncodeTiled failed (%d)", static_cast<int>(r));
  return FP4IDX_OK;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int groups_of(int format) { return format == FP4IDX_MXFP4 ? 4 : 8; }

// Checks shared by every entry point.
fp4idx_status_t check_problem(const fp4idx_problem_t* p) {
  if (!p) return fail(FP4IDX_EINVAL, "problem is NULL");
  if (p->format != FP4IDX_MXFP4 && p->format != FP4IDX_NVFP4)
    return fail(FP4IDX_EINVAL, "format %d is neither MXFP4 (0) nor NVFP4 (1)", p->format);
  if (p->num_seqs < 1) return fail(FP4IDX_EINVAL, "num_seqs must be >= 1 (got %d)", p->num_seqs);
  if (p->num_rows < 0) return fail(FP4IDX_EINVAL, "num_rows must be >= 0");
  if (p->num_heads < 1 || p->num_kv_heads < 1 || p->num_heads % p->num_kv_heads != 0)
    return fail(FP4IDX_EINVAL, "num_heads (%d) must be a positive multiple of num_kv_heads (%d)", p->num_heads,
                p->num_kv_heads);
  if (p->page_size != 64 && p->page_size != 128)
    return fail(FP4IDX_EUNSUPPORTED, "page_size %d: only 64 and 128 are supported", p->page_size);
  if (p->num_pages < 1) return fail(FP4IDX_EINVAL, "num_pages must be >= 1");
  if (p->num_pages * p->num_kv_heads * p->page_size > INT32_MAX)
    return fail(FP4IDX_EUNSUPPORTED, "cache rows exceed 2^31");
  if (p->max_seqlen_q < 1) return fail(FP4IDX_EINVAL, "max_seqlen_q must be >= 1");
  if (p->max_seqlen_k < 0) return fail(FP4IDX_EINVAL, "max_seqlen_k must be >= 0");
  if (p->kv_layout != FP4IDX_KV_SPLIT && p->kv_layout != FP4IDX_KV_FUSED)
    return fail(FP4IDX_EINVAL, "kv_layout %d is neither split (0) nor fused (1)", p->kv_layout);
  const bool fused = p->kv_layout == FP4IDX_KV_FUSED;
  if (!p->q || !p->q_scale || !p->k || (!fused && !p->k_scale) || !p->cu_seqlens_q || !p->cu_seqlens_k ||
      !p->block_table)
    return fail(FP4IDX_EINVAL, "q, q_scale, k, k_scale (split layout), cu_seqlens_q, cu_seqlens_k and block_table "
                               "are required");
  if (!aligned(p->q, 128) || !aligned(p->k, 128))
    return fail(FP4IDX_EINVAL, "q and k must be 128-byte aligned");
  if (!aligned(p->q_scale, 16) || (!fused && !aligned(p->k_scale, 16)))
    return fail(FP4IDX_EINVAL, "q_scale and k_scale must be 16-byte aligned");
  if (p->cand_mask && p->mask_ld < p->max_seqlen_k)
    return fail(FP4IDX_EINVAL, "mask_ld %lld < max_seqlen_k %d", static_cast<long long>(p->mask_ld),
                p->max_seqlen_k);
  const int G = groups_of(p->format);
  if (p->q_row_stride < static_cast<int64_t>(p->num_heads) * 64 || p->q_row_stride % 16 != 0)
    return fail(FP4IDX_EINVAL, "q_row_stride %lld must be a multiple of 16 and >= num_heads*64",
                static_cast<long long>(p->q_row_stride));
  if (p->q_scale_row_stride < static_cast<int64_t>(p->num_heads) * G || p->q_scale_row_stride % 8 != 0)
    return fail(FP4IDX_EINVAL, "q_scale_row_stride %lld must be a multiple of 8 and >= num_heads*%d",
                static_cast<long long>(p->q_scale_row_stride), G);
  if (!p->page_offsets) {
    const int64_t need = (static_cast<int64_t>(p->max_seqlen_k) + p->page_size - 1) / p->page_size;
    if (p->table_stride < need)
      return fail(FP4IDX_EINVAL, "table_stride %lld < pages of max_seqlen_k (%lld)",
                  static_cast<long long>(p->table_stride), static_cast<long long>(need));
  }
  if (p->qo_offset && !p->causal) return fail(FP4IDX_EINVAL, "qo_offset is only allowed with causal != 0");
  return FP4IDX_OK;
}

// Shapes the weighted-ReLU kernels (logits, top-k) implement.
fp4idx_status_t check_weighted_shape(const fp4idx_problem_t* p) {
  if (p->num_kv_heads != 1)
    return fail(FP4IDX_EUNSUPPORTED, "weighted-ReLU scoring supports one K head (num_kv_heads = %d)",
                p->num_kv_heads);
  if (p->num_heads != 8 && p->num_heads != 16 && p->num_heads != 32 && p->num_heads != 64)
    return fail(FP4IDX_EUNSUPPORTED, "num_heads %d: supported 8, 16, 32, 64", p->num_heads);
  return FP4IDX_OK;
}

// Checks of the weighted-ReLU paths (logits, top-k) including the weights.
fp4idx_status_t check_weighted(const fp4idx_problem_t* p, const float* w, int64_t w_row_stride) {
  fp4idx_status_t s = check_weighted_shape(p);
  if (s != FP4IDX_OK) return s;
  if (!w) return fail(FP4IDX_EINVAL, "w is NULL");
  if (!aligned(w, 4)) return fail(FP4IDX_EINVAL, "w must be 4-byte aligned");
  if (w_row_stride < p->num_heads) return fail(FP4IDX_EINVAL, "w_row_stride must be >= num_heads");
  return FP4IDX_OK;
}

// TMA map of the K codes -- 3D {64 B, page, num_pages*Hkv blocks}, one box
// per (page, K head) block -- and where each block's scales start, for
// either cache layout.
fp4idx_status_t k_access(const fp4idx_problem_t* pr, CUtensorMap* tmap, const uint8_t** kscale_base,
                         int64_t* kscale_block_stride) {
  const int G = groups_of(pr->format);
  const int64_t page = pr->page_size;
  const bool fused = pr->kv_layout == FP4IDX_KV_FUSED;
  const int64_t block_bytes = fused ? page * (64 + G) : page * 64;
  cuuint64_t dims[3] = {64, static_cast<cuuint64_t>(page), static_cast<cuuint64_t>(pr->num_pages) * pr->num_kv_heads};
  cuuint64_t strides[2] = {64, static_cast<cuuint64_t>(block_bytes)};
  cuuint32_t box[3] = {64, static_cast<cuuint32_t>(page), 1};
  fp4idx_status_t s = make_tmap(tmap, pr->k, 3, dims, strides, box);
  if (s != FP4IDX_OK) return s;
  *kscale_base = fused ? pr->k + page * 64 : pr->k_scale;
  *kscale_block_stride = fused ? block_bytes : page * G;
  return FP4IDX_OK;
}

// Common part of the scorer parameters.
fp4idx_status_t fill_score_params(const fp4idx_problem_t* pr, const float* w, int64_t w_row_stride,
                                  ScoreParams* sp, int rows_per_cta, uint32_t* err) {
  std::memset(sp, 0, sizeof(*sp));
  const int G = groups_of(pr->format);
  {
    // codes and scales of each (page, K head) block, either cache layout
    const int64_t page = pr->page_size;
    const bool fused = pr->kv_layout == FP4IDX_KV_FUSED;
    sp->kcode_base = pr->k;
    sp->kcode_block_stride = fused ? page * (64 + G) : page * 64;
    sp->kscale_base = fused ? pr->k + page * 64 : pr->k_scale;
    sp->kscale_block_stride = fused ? page * (64 + G) : page * G;
  }
  {
    cuuint64_t dims[3] = {64, static_cast<cuuint64_t>(pr->num_heads), static_cast<cuuint64_t>(pr->num_rows)};
    cuuint64_t strides[2] = {64, static_cast<cuuint64_t>(pr->q_row_stride)};
    cuuint32_t box[3] = {64, static_cast<cuuint32_t>(pr->num_heads), static_cast<cuuint32_t>(rows_per_cta)};
    fp4idx_status_t s = make_tmap(&sp->tmap_q, pr->q, 3, dims, strides, box);
    if (s != FP4IDX_OK) return s;
  }
  sp->cand_mask = pr->cand_mask;
  sp->mask_ld = pr->mask_ld;
  sp->q_scale = pr->q_scale;
  sp->q_scale_row_stride = pr->q_scale_row_stride;
  sp->cu_seqlens_q = pr->cu_seqlens_q;
  sp->cu_seqlens_k = pr->cu_seqlens_k;
  sp->block_table = pr->block_table;
  sp->page_offsets = pr->page_offsets;
  sp->table_stride = pr->table_stride;
  sp->visible_len = pr->visible_len;
  sp->qo_offset = pr->qo_offset;
  sp->causal = pr->causal;
  sp->page_size = pr->page_size;
  sp->page_shift = pr->page_size == 128 ? 7 : 6;
  sp->num_pages = pr->num_pages;
  sp->num_rows = pr->num_rows;
  sp->num_heads = pr->num_heads;
  sp->num_seqs = pr->num_seqs;
  sp->row_groups = (pr->max_seqlen_q + rows_per_cta - 1) / rows_per_cta;
  sp->max_seqlen_k = pr->max_seqlen_k;
  sp->uniform_items = 0;
  sp->w = w;
  sp->w_row_stride = w_row_stride;
  sp->err = err;
  return FP4IDX_OK;
}

// Scorer CTAs for top-k: one per SM, fewer when there are fewer tiles.
int topk_ctas(const fp4idx_problem_t* p, int sms) {
  const int R = score_rows_per_cta(p->num_heads);
  const int64_t items = static_cast<int64_t>(p->num_seqs) * ((p->max_seqlen_q + R - 1) / R);
  const int64_t tiles = items * ((static_cast<int64_t>(p->max_seqlen_k) + kTileKeys - 1) / kTileKeys);
  int64_t c = tiles < sms ? tiles : sms;
  return c < 1 ? 1 : static_cast<int>(c);
}

struct TopkWorkspace {
  size_t keys_off, count_off, cand_off, start_off, pool_off, pool_bytes, bytes;
};

// Whether the streaming top-k pools its bucket counts across CTAs: rows
// scored by four-row CTAs (their keys spread over many CTAs), few enough
// rows that the counts (8 KB a row) are cheap to clear.
bool use_pool(const fp4idx_problem_t* p) {
  return score_rows_per_cta(p->num_heads) == 4 && p->num_rows <= kPoolMaxRows;
}

// Short-context plan of fp4idx_topk: logits into the workspace, then a
// per-row selection.  Decided from host scalars only.
int64_t logits_plan_ld(const fp4idx_problem_t* p) { return (static_cast<int64_t>(p->max_seqlen_k) + 3) / 4 * 4; }
bool use_logits_plan(const fp4idx_problem_t* p) {
  return p->max_seqlen_k <= 16384 && static_cast<int64_t>(p->num_rows) * logits_plan_ld(p) <= (int64_t(1) << 24);
}

// Workspace of the top-k path: per-CTA partial lists, their counts, and each
// scorer CTA's per-row streaming candidate buffers.
TopkWorkspace topk_workspace(const fp4idx_problem_t* p, int32_t k, int sms) {
  const int R = score_rows_per_cta(p->num_heads);
  const int ctas = topk_ctas(p, sms);
  const int64_t items = static_cast<int64_t>(p->num_seqs) * ((p->max_seqlen_q + R - 1) / R);
  const int64_t slots = (ctas + items) * R;
  auto up = [](size_t x) { return (x + 255) / 256 * 256; };
  TopkWorkspace ws;
  ws.keys_off = 0;
  ws.count_off = up(static_cast<size_t>(slots) * topk_part_capacity(k) * 8);
  ws.cand_off = ws.count_off + up(static_cast<size_t>(slots) * 4);
  ws.start_off = ws.cand_off + up(static_cast<size_t>(ctas) * R * topk_cand_capacity(k) * 8);
  ws.pool_off = ws.start_off + up(static_cast<size_t>(items + 1) * 4);
  ws.pool_bytes = use_pool(p) ? up(static_cast<size_t>(p->num_rows) * (kPoolBins + 1) * 4) : 0;
  ws.bytes = ws.pool_off + ws.pool_bytes;
  // the short-context plan keeps the logits [T][ld] at offset 0 instead
  if (use_logits_plan(p)) {
    const size_t lb = up(static_cast<size_t>(p->num_rows) * logits_plan_ld(p) * 4);
    if (lb > ws.bytes) ws.bytes = lb;
  }
  return ws;
}

}  // namespace

void set_last_error(const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_msg, sizeof(g_msg), fmt, ap);
  va_end(ap);
}

}  // namespace fp4idx

using namespace fp4idx;

extern "C" {

const char* fp4idx_status_string(fp4idx_status_t s) {
  switch (s) {
    case FP4IDX_OK: return "ok";
    case FP4IDX_EINVAL: return "invalid argument";
    case FP4IDX_EUNSUPPORTED: return "unsupported configuration";
    case FP4IDX_EWORKSPACE: return "workspace too small";
    case FP4IDX_ECUDA: return "CUDA error";
    case FP4IDX_EDEVICE: return "unsupported device";
  }
  return "unknown status";
}

const char* fp4idx_last_error_message(void) { return g_msg; }

fp4idx_status_t fp4idx_logits(const fp4idx_problem_t* problem, const float* w, int64_t w_row_stride,
                              float* logits, int64_t ld, void* stream) {
  g_msg[0] = 0;
  fp4idx_status_t s = check_problem(problem);
  if (s != FP4IDX_OK) return s;
  if ((s = check_weighted(problem, w, w_row_stride)) != FP4IDX_OK) return s;
  if (!logits) return fail(FP4IDX_EINVAL, "logits is NULL");
  if (ld < 1 || ld % 4 != 0) return fail(FP4IDX_EINVAL, "ld must be a positive multiple of 4");
  if (!aligned(logits, 16)) return fail(FP4IDX_EINVAL, "logits must be 16-byte aligned");
  if (problem->num_rows == 0) return FP4IDX_OK;
  DeviceInfo* dev;
  if ((s = device_info(&dev)) != FP4IDX_OK) return s;
  const int R = score_rows_per_cta(problem->num_heads);
  ScoreParams sp;
  if ((s = fill_score_params(problem, w, w_row_stride, &sp, R, dev->err)) != FP4IDX_OK) return s;
  sp.total_tiles = static_cast<int32_t>((ld + kTileKeys - 1) / kTileKeys);
  // one request whose row count fills every row group: each item holds
  // total_tiles tiles, so the CTAs need not read the metadata to plan
  sp.uniform_items = problem->num_seqs == 1 && sp.row_groups == (problem->num_rows + R - 1) / R ? 1 : 0;
  sp.logits = logits;
  sp.ld = ld;
  sp.k = 1;
  const int64_t items = static_cast<int64_t>(problem->num_seqs) * sp.row_groups;
  const int64_t tiles = items * sp.total_tiles;
  const int ctas = static_cast<int>(tiles < dev->sms ? tiles : dev->sms);
  sp.score_ctas = ctas;
  cudaError_t e = launch_score(sp, problem->format, kModeLogits, problem->num_heads, dim3(ctas),
                               static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "scorer launch");
  return FP4IDX_OK;
}

size_t fp4idx_topk_workspace_bytes(const fp4idx_problem_t* problem, int32_t k) {
  if (check_problem(problem) != FP4IDX_OK || k < 1 || k > 2048) return 0;
  DeviceInfo* dev;
  if (device_info(&dev) != FP4IDX_OK) return 0;
  return topk_workspace(problem, k, dev->sms).bytes;
}

}  // extern "C"

namespace fp4idx {
namespace {

// Validation and parameters common to both top-k phases.
fp4idx_status_t topk_prepare(const fp4idx_problem_t* problem, const float* w, int64_t w_row_stride, int32_t k,
                             void* workspace, size_t workspace_bytes, bool need_w, ScoreParams* sp,
                             int* ctas) {
  fp4idx_status_t s = check_problem(problem);
  if (s != FP4IDX_OK) return s;
  s = need_w ? check_weighted(problem, w, w_row_stride) : check_weighted_shape(problem);
  if (s != FP4IDX_OK) return s;
  if (k < 1 || k > 2048) return fail(FP4IDX_EUNSUPPORTED, "k = %d: supported 1..2048", k);
  DeviceInfo* dev;
  if ((s = device_info(&dev)) != FP4IDX_OK) return s;
  const TopkWorkspace ws = topk_workspace(problem, k, dev->sms);
  if (!workspace || workspace_bytes < ws.bytes)
    return fail(FP4IDX_EWORKSPACE, "workspace needs %zu bytes (got %zu)", ws.bytes, workspace_bytes);
  if (!aligned(workspace, 256)) return fail(FP4IDX_EINVAL, "workspace must be 256-byte aligned");
  const int R = score_rows_per_cta(problem->num_heads);
  if ((s = fill_score_params(problem, w, w_row_stride, sp, R, dev->err)) != FP4IDX_OK) return s;
  sp->total_tiles = (problem->max_seqlen_k + kTileKeys - 1) / kTileKeys;
  sp->k = k;
  sp->part_keys = reinterpret_cast<uint64_t*>(static_cast<uint8_t*>(workspace) + ws.keys_off);
  sp->part_count = reinterpret_cast<int32_t*>(static_cast<uint8_t*>(workspace) + ws.count_off);
  sp->cand = reinterpret_cast<uint64_t*>(static_cast<uint8_t*>(workspace) + ws.cand_off);
  sp->item_start = reinterpret_cast<int32_t*>(static_cast<uint8_t*>(workspace) + ws.start_off);
  sp->item_overhead = kTopkItemOverhead;
  if (ws.pool_bytes) {
    sp->pool_hist = reinterpret_cast<uint32_t*>(static_cast<uint8_t*>(workspace) + ws.pool_off);
    sp->pool_top = sp->pool_hist + static_cast<size_t>(problem->num_rows) * kPoolBins;
  }
  *ctas = topk_ctas(problem, dev->sms);
  if (*ctas >= kMaxMergeSlots) return fail(FP4IDX_EUNSUPPORTED, "more than %d SMs", kMaxMergeSlots - 1);
  sp->score_ctas = *ctas;
  return FP4IDX_OK;
}

}  // namespace
}  // namespace fp4idx

extern "C" {

fp4idx_status_t fp4idx_topk_score(const fp4idx_problem_t* problem, const float* w, int64_t w_row_stride,
                                  int32_t k, void* workspace, size_t workspace_bytes, void* stream) {
  g_msg[0] = 0;
  if (problem && problem->num_rows == 0 && check_problem(problem) == FP4IDX_OK) return FP4IDX_OK;
  ScoreParams sp;
  int ctas = 0;
  fp4idx_status_t s = topk_prepare(problem, w, w_row_stride, k, workspace, workspace_bytes, true, &sp, &ctas);
  if (s != FP4IDX_OK) return s;
  if (sp.pool_hist) {
    const size_t bytes = static_cast<size_t>(problem->num_rows) * (kPoolBins + 1) * 4;
    cudaError_t e = cudaMemsetAsync(sp.pool_hist, 0, bytes, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "pooled-count clear");
  }
  cudaError_t e = launch_score(sp, problem->format, kModeTopk, problem->num_heads, dim3(ctas),
                               static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "scorer launch");
  return FP4IDX_OK;
}

fp4idx_status_t fp4idx_topk_merge(const fp4idx_problem_t* problem, int32_t k, uint32_t flags, int32_t* indices,
                                  float* values, int32_t* valid_count, void* workspace, size_t workspace_bytes,
                                  void* stream) {
  g_msg[0] = 0;
  if (flags & ~static_cast<uint32_t>(FP4IDX_TOPK_SORTED)) return fail(FP4IDX_EINVAL, "unknown flags 0x%x", flags);
  if (!indices) return fail(FP4IDX_EINVAL, "indices is NULL");
  if (problem && problem->num_rows == 0 && check_problem(problem) == FP4IDX_OK) return FP4IDX_OK;
  ScoreParams sp;
  int ctas = 0;
  fp4idx_status_t s = topk_prepare(problem, nullptr, 0, k, workspace, workspace_bytes, false, &sp, &ctas);
  if (s != FP4IDX_OK) return s;
  MergeParams mp;
  mp.sp = sp;
  mp.rows_per_cta = score_rows_per_cta(problem->num_heads);
  mp.flags = flags;
  mp.indices = indices;
  mp.values = values;
  mp.valid_count = valid_count;
  DeviceInfo* dev;
  if ((s = device_info(&dev)) != FP4IDX_OK) return s;
  cudaError_t e = launch_topk_merge(mp, problem->num_rows, problem->num_rows > 4 * dev->sms,
                                    static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "merge launch");
  return FP4IDX_OK;
}

}  // extern "C"

namespace fp4idx {
namespace {

// Logits of every row into `logits` [T][ld], then each row's top-k from them.
fp4idx_status_t logits_then_select(const fp4idx_problem_t* problem, const float* w, int64_t w_row_stride,
                                   float* logits, int64_t ld, int32_t k, uint32_t flags, int32_t* indices,
                                   float* values, int32_t* valid_count, void* stream) {
  fp4idx_status_t s = fp4idx_logits(problem, w, w_row_stride, logits, ld, stream);
  if (s != FP4IDX_OK) return s;
  if (problem->num_rows == 0) return FP4IDX_OK;
  DeviceInfo* dev;
  if ((s = device_info(&dev)) != FP4IDX_OK) return s;
  MergeParams mp;
  std::memset(&mp, 0, sizeof(mp));
  const int R = score_rows_per_cta(problem->num_heads);
  if ((s = fill_score_params(problem, w, w_row_stride, &mp.sp, R, dev->err)) != FP4IDX_OK) return s;
  mp.sp.logits = logits;
  mp.sp.ld = ld;
  mp.sp.k = k;
  mp.rows_per_cta = R;
  mp.flags = flags & FP4IDX_TOPK_SORTED;
  mp.indices = indices;
  mp.values = values;
  mp.valid_count = valid_count;
  cudaError_t e = launch_topk_select(mp, problem->num_rows, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "select launch");
  return FP4IDX_OK;
}

}  // namespace
}  // namespace fp4idx

extern "C" {

fp4idx_status_t fp4idx_topk(const fp4idx_problem_t* problem, const float* w, int64_t w_row_stride, int32_t k,
                            uint32_t flags, int32_t* indices, float* values, int32_t* valid_count,
                            void* workspace, size_t workspace_bytes, void* stream) {
  g_msg[0] = 0;
  if (flags & ~static_cast<uint32_t>(FP4IDX_TOPK_SORTED | FP4IDX_TOPK_STREAMING))
    return fail(FP4IDX_EINVAL, "unknown flags 0x%x", flags);
  if (!indices) return fail(FP4IDX_EINVAL, "indices is NULL");
  if (!(flags & FP4IDX_TOPK_STREAMING) && problem && check_problem(problem) == FP4IDX_OK &&
      use_logits_plan(problem)) {
    // same validation and workspace contract as the streaming plan
    ScoreParams sp;
    int ctas = 0;
    fp4idx_status_t s = topk_prepare(problem, w, w_row_stride, k, workspace, workspace_bytes, true, &sp, &ctas);
    if (s != FP4IDX_OK) return s;
    if (!aligned(workspace, 16)) return fail(FP4IDX_EINVAL, "workspace must be 16-byte aligned");
    return logits_then_select(problem, w, w_row_stride, static_cast<float*>(workspace), logits_plan_ld(problem), k,
                              flags, indices, values, valid_count, stream);
  }
  fp4idx_status_t s = fp4idx_topk_score(problem, w, w_row_stride, k, workspace, workspace_bytes, stream);
  if (s != FP4IDX_OK) return s;
  return fp4idx_topk_merge(problem, k, flags & FP4IDX_TOPK_SORTED, indices, values, valid_count, workspace,
                           workspace_bytes, stream);
}

fp4idx_status_t fp4idx_logits_topk(const fp4idx_problem_t* problem, const float* w, int64_t w_row_stride,
                                   float* logits, int64_t ld, int32_t k, uint32_t flags, int32_t* indices,
                                   float* values, int32_t* valid_count, void* stream) {
  g_msg[0] = 0;
  if (flags & ~static_cast<uint32_t>(FP4IDX_TOPK_SORTED)) return fail(FP4IDX_EINVAL, "unknown flags 0x%x", flags);
  if (!indices) return fail(FP4IDX_EINVAL, "indices is NULL");
  fp4idx_status_t s = check_problem(problem);
  if (s != FP4IDX_OK) return s;
  if ((s = check_weighted(problem, w, w_row_stride)) != FP4IDX_OK) return s;
  if (k < 1 || k > 2048) return fail(FP4IDX_EUNSUPPORTED, "k = %d: supported 1..2048", k);
  if (ld < problem->max_seqlen_k) return fail(FP4IDX_EINVAL, "ld must be >= max_seqlen_k");
  return logits_then_select(problem, w, w_row_stride, logits, ld, k, flags, indices, values, valid_count, stream);
}

}  // extern "C"

namespace fp4idx {
namespace {

// Both layouts of the K-cache writer (k_scale == nullptr: the fused table).
fp4idx_status_t store_k_any(const uint16_t* keys, int64_t key_row_stride, int32_t num_tokens,
                            int32_t num_kv_heads, const int32_t* slots, int32_t page_size, int64_t num_pages,
                            uint8_t* k, uint8_t* k_scale, void* stream) {
  g_msg[0] = 0;
  if (!keys || !slots || !k) return fail(FP4IDX_EINVAL, "keys, slots or the cache is NULL");
  if (num_tokens < 0 || num_kv_heads < 1 || num_pages < 1)
    return fail(FP4IDX_EINVAL, "num_tokens >= 0, num_kv_heads >= 1 and num_pages >= 1 required");
  if (page_size != 64 && page_size != 128) return fail(FP4IDX_EUNSUPPORTED, "page_size %d: 64 or 128", page_size);
  if (key_row_stride < static_cast<int64_t>(num_kv_heads) * 128 || key_row_stride % 8 != 0)
    return fail(FP4IDX_EINVAL, "key_row_stride must be >= num_kv_heads * 128 and a multiple of 8");
  if (!aligned(keys, 16) || !aligned(k, 16) || !aligned(slots, 4))
    return fail(FP4IDX_EINVAL, "keys and k must be 16-byte aligned, slots 4-byte aligned");
  if (num_tokens == 0) return FP4IDX_OK;
  DeviceInfo* dev;
  fp4idx_status_t s;
  if ((s = device_info(&dev)) != FP4IDX_OK) return s;
  StoreParams sp;
  std::memset(&sp, 0, sizeof(sp));
  sp.keys = keys;
  sp.key_row_stride = key_row_stride;
  sp.slots = slots;
  sp.k = k;
  sp.k_scale = k_scale;
  sp.fused = k_scale ? 0 : 1;
  sp.num_pages = num_pages;
  sp.num_tokens = num_tokens;
  sp.num_kv_heads = num_kv_heads;
  sp.page_size = page_size;
  sp.err = dev->err;
  cudaError_t e = launch_store_k(sp, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "store launch");
  return FP4IDX_OK;
}

}  // namespace
}  // namespace fp4idx

extern "C" {

fp4idx_status_t fp4idx_store_k(const uint16_t* keys, int64_t key_row_stride, int32_t num_tokens,
                               int32_t num_kv_heads, const int32_t* slots, int32_t page_size, int64_t num_pages,
                               uint8_t* k, uint8_t* k_scale, void* stream) {
  if (!k_scale) {
    g_msg[0] = 0;
    return fail(FP4IDX_EINVAL, "k_scale is NULL");
  }
  return store_k_any(keys, key_row_stride, num_tokens, num_kv_heads, slots, page_size, num_pages, k, k_scale,
                     stream);
}

fp4idx_status_t fp4idx_store_k_fused(const uint16_t* keys, int64_t key_row_stride, int32_t num_tokens,
                                     int32_t num_kv_heads, const int32_t* slots, int32_t page_size,
                                     int64_t num_pages, uint8_t* table, void* stream) {
  return store_k_any(keys, key_row_stride, num_tokens, num_kv_heads, slots, page_size, num_pages, table, nullptr,
                     stream);
}

fp4idx_status_t fp4idx_quantize_q(const uint16_t* q, int64_t q_row_stride, int32_t num_rows, int32_t num_heads,
                                  uint8_t* q_codes, uint8_t* q_scale, void* stream) {
  g_msg[0] = 0;
  if (!q || !q_codes || !q_scale) return fail(FP4IDX_EINVAL, "q, q_codes or q_scale is NULL");
  if (num_rows < 0 || num_heads < 1) return fail(FP4IDX_EINVAL, "num_rows >= 0 and num_heads >= 1 required");
  if (q_row_stride < static_cast<int64_t>(num_heads) * 128 || q_row_stride % 8 != 0)
    return fail(FP4IDX_EINVAL, "q_row_stride must be >= num_heads * 128 and a multiple of 8");
  if (!aligned(q, 16) || !aligned(q_codes, 16)) return fail(FP4IDX_EINVAL, "q and q_codes must be 16-byte aligned");
  if (num_rows == 0) return FP4IDX_OK;
  DeviceInfo* dev;
  fp4idx_status_t s;
  if ((s = device_info(&dev)) != FP4IDX_OK) return s;
  // each query row is a token on a one-token page of its own: the cache
  // arrays [rows][heads][1][64] / [rows][heads][1][4] are the query layout
  StoreParams sp;
  std::memset(&sp, 0, sizeof(sp));
  sp.keys = q;
  sp.key_row_stride = q_row_stride;
  sp.slots = nullptr;
  sp.k = q_codes;
  sp.k_scale = q_scale;
  sp.fused = 0;
  sp.num_pages = num_rows;
  sp.num_tokens = num_rows;
  sp.num_kv_heads = num_heads;
  sp.page_size = 1;
  sp.err = dev->err;
  cudaError_t e = launch_store_k(sp, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "quantize launch");
  return FP4IDX_OK;
}

fp4idx_status_t fp4idx_pages_from_token_table(const int32_t* req, int32_t num_rows, const int32_t* req_table,
                                              int32_t num_reqs, int64_t req_stride, int32_t page_size,
                                              int64_t num_pages, int32_t* cu_seqlens_q, int32_t* cu_seqlens_k,
                                              int32_t* block_table, void* stream) {
  g_msg[0] = 0;
  if (!req || !req_table || !cu_seqlens_q || !cu_seqlens_k || !block_table)
    return fail(FP4IDX_EINVAL, "req, req_table, cu_seqlens_q, cu_seqlens_k and block_table are required");
  if (num_rows < 0 || num_reqs < 1 || req_stride < 1 || num_pages < 1)
    return fail(FP4IDX_EINVAL, "num_rows >= 0, num_reqs >= 1, req_stride >= 1 and num_pages >= 1 required");
  if (page_size != 64 && page_size != 128) return fail(FP4IDX_EUNSUPPORTED, "page_size %d: 64 or 128", page_size);
  if (req_stride > INT32_MAX || static_cast<int64_t>(num_reqs) * req_stride > INT32_MAX)
    return fail(FP4IDX_EUNSUPPORTED, "more than 2^31 table entries");
  if ((req_stride + page_size - 1) / page_size > 65535 * 8)
    return fail(FP4IDX_EUNSUPPORTED, "more than 524,280 pages per request");  // grid.y of the page pass
  DeviceInfo* dev;
  fp4idx_status_t s;
  if ((s = device_info(&dev)) != FP4IDX_OK) return s;
  TokenTableParams tp;
  std::memset(&tp, 0, sizeof(tp));
  tp.req = req;
  tp.req_table = req_table;
  tp.req_stride = req_stride;
  tp.num_rows = num_rows;
  tp.num_reqs = num_reqs;
  tp.page_size = page_size;
  tp.num_pages = num_pages;
  tp.cu_seqlens_q = cu_seqlens_q;
  tp.cu_seqlens_k = cu_seqlens_k;
  tp.block_table = block_table;
  tp.table_pages = static_cast<int32_t>((req_stride + page_size - 1) / page_size);
  tp.err = dev->err;
  cudaError_t e = launch_token_table(tp, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "token-table launch");
  return FP4IDX_OK;
}

fp4idx_status_t fp4idx_topk_slots(const fp4idx_problem_t* problem, const int32_t* indices, int32_t k,
                                  int32_t* slots, int32_t ncols, int32_t* offset_bits, void* stream) {
  g_msg[0] = 0;
  fp4idx_status_t s = check_problem(problem);
  if (s != FP4IDX_OK) return s;
  if (!indices || !slots) return fail(FP4IDX_EINVAL, "indices or slots is NULL");
  if (k < 1 || ncols < k) return fail(FP4IDX_EINVAL, "need ncols >= k >= 1 (k = %d, ncols = %d)", k, ncols);
  if (!aligned(indices, 4) || !aligned(slots, 4)) return fail(FP4IDX_EINVAL, "indices and slots must be 4-byte aligned");
  int bits = 1;
  while ((1 << bits) < problem->page_size) ++bits;  // bit length of page_size - 1, at least 1
  if (static_cast<int64_t>(problem->num_pages) << bits >= (int64_t(1) << 31))
    return fail(FP4IDX_EUNSUPPORTED, "num_pages << %d does not fit in 31 bits", bits);
  if (offset_bits) *offset_bits = bits;
  if (problem->num_rows == 0) return FP4IDX_OK;
  if (problem->num_rows > 65535) return fail(FP4IDX_EUNSUPPORTED, "more than 65,535 rows");  // grid.y
  SlotParams sp;
  std::memset(&sp, 0, sizeof(sp));
  sp.indices = indices;
  sp.slots = slots;
  sp.cu_seqlens_q = problem->cu_seqlens_q;
  sp.cu_seqlens_k = problem->cu_seqlens_k;
  sp.block_table = problem->block_table;
  sp.page_offsets = problem->page_offsets;
  sp.table_stride = problem->table_stride;
  sp.num_seqs = problem->num_seqs;
  sp.num_pages = static_cast<int32_t>(problem->num_pages);
  sp.page_size = problem->page_size;
  sp.page_shift = problem->page_size == 128 ? 7 : 6;
  sp.offset_bits = bits;
  sp.k = k;
  sp.ncols = ncols;
  cudaError_t e = launch_topk_slots(sp, problem->num_rows, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "slot launch");
  return FP4IDX_OK;
}

fp4idx_status_t fp4idx_block_topk(const float* scores, int32_t num_heads, int32_t ktiles, int32_t num_rows,
                                  int32_t k, int32_t* indices, float* values, int32_t* valid_count, void* stream) {
  g_msg[0] = 0;
  if (!scores) return fail(FP4IDX_EINVAL, "scores is NULL");
  if (!indices) return fail(FP4IDX_EINVAL, "indices is NULL");
  if (num_heads < 1 || ktiles < 1 || num_rows < 1 || k < 1)
    return fail(FP4IDX_EINVAL, "num_heads, ktiles, num_rows and k must be positive");
  if (k > 128) return fail(FP4IDX_EUNSUPPORTED, "k = %d: supported 1..128", k);
  if (k > 32 && ktiles > 1024) return fail(FP4IDX_EUNSUPPORTED, "k = %d > 32 needs ktiles <= 1024 (got %d)", k, ktiles);
  if (!aligned(scores, 4) || !aligned(indices, 4) || (values && !aligned(values, 4)) ||
      (valid_count && !aligned(valid_count, 4)))
    return fail(FP4IDX_EINVAL, "scores, indices, values and valid_count must be 4-byte aligned");
  if (static_cast<int64_t>(num_heads) * num_rows >= (int64_t(1) << 38))  // grid.x < 2^31 blocks of 256
    return fail(FP4IDX_EUNSUPPORTED, "too many columns");
  DeviceInfo* dev;
  fp4idx_status_t s;
  if ((s = device_info(&dev)) != FP4IDX_OK) return s;
  cudaError_t e = launch_block_topk(scores, num_heads, ktiles, num_rows, k, indices, values, valid_count, dev->sms,
                                    static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "block top-k launch");
  return FP4IDX_OK;
}

fp4idx_status_t fp4idx_block_scores(const fp4idx_problem_t* problem, float* scores, void* stream) {
  g_msg[0] = 0;
  fp4idx_status_t s = check_problem(problem);
  if (s != FP4IDX_OK) return s;
  if (!scores) return fail(FP4IDX_EINVAL, "scores is NULL");
  if (!aligned(scores, 4)) return fail(FP4IDX_EINVAL, "scores must be 4-byte aligned");
  const int g = problem->num_heads / problem->num_kv_heads;
  if (g > 128 || (g & (g - 1)) != 0)
    return fail(FP4IDX_EUNSUPPORTED, "num_heads / num_kv_heads = %d: supported powers of two up to 128", g);
  const int64_t ktiles = (static_cast<int64_t>(problem->max_seqlen_k) + kTileKeys - 1) / kTileKeys;
  if (problem->num_rows == 0 || ktiles == 0) return FP4IDX_OK;  // nothing to write
  int group_shift = 0;
  while ((1 << group_shift) < g) ++group_shift;
  const int rt_shift = 7 - group_shift;
  const int64_t row_tiles = (static_cast<int64_t>(problem->max_seqlen_q) + (1 << rt_shift) - 1) >> rt_shift;
  const int64_t items = static_cast<int64_t>(problem->num_seqs) * problem->num_kv_heads * row_tiles;
  if (items * ktiles > INT32_MAX) return fail(FP4IDX_EUNSUPPORTED, "more than 2^31 block tiles");
  DeviceInfo* dev;
  if ((s = device_info(&dev)) != FP4IDX_OK) return s;
  BlockParams bp;
  std::memset(&bp, 0, sizeof(bp));
  if ((s = k_access(problem, &bp.tmap_k, &bp.kscale_base, &bp.kscale_block_stride)) != FP4IDX_OK) return s;
  {
    // rows (t) before heads (h) in the box: MMA row m = h_local * RT + t_local
    cuuint64_t dims[3] = {64, static_cast<cuuint64_t>(problem->num_rows), static_cast<cuuint64_t>(problem->num_heads)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(problem->q_row_stride), 64};
    cuuint32_t box[3] = {64, static_cast<cuuint32_t>(1 << rt_shift), static_cast<cuuint32_t>(g)};
    if ((s = make_tmap(&bp.tmap_q, problem->q, 3, dims, strides, box)) != FP4IDX_OK) return s;
  }

  bp.q_scale = problem->q_scale;
  bp.q_scale_row_stride = problem->q_scale_row_stride;
  bp.cu_seqlens_q = problem->cu_seqlens_q;
  bp.cu_seqlens_k = problem->cu_seqlens_k;
  bp.block_table = problem->block_table;
  bp.page_offsets = problem->page_offsets;
  bp.table_stride = problem->table_stride;
  bp.visible_len = problem->visible_len;
  bp.qo_offset = problem->qo_offset;
  bp.causal = problem->causal;
  bp.page_size = problem->page_size;
  bp.page_shift = problem->page_size == 128 ? 7 : 6;
  bp.num_pages = problem->num_pages;
  bp.num_rows = problem->num_rows;
  bp.num_heads = problem->num_heads;
  bp.num_kv_heads = problem->num_kv_heads;
  bp.num_seqs = problem->num_seqs;
  bp.group_shift = group_shift;
  bp.rt_shift = rt_shift;
  bp.row_tiles = static_cast<int32_t>(row_tiles);
  bp.ktiles = static_cast<int32_t>(ktiles);
  bp.scores = scores;
  bp.err = dev->err;
  const int64_t tiles = items * ktiles;
  const int ctas = static_cast<int>(tiles < dev->sms ? tiles : dev->sms);
  cudaError_t e = launch_block_scores(bp, problem->format, dim3(ctas), static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "block-score launch");
  return FP4IDX_OK;
}

fp4idx_status_t fp4idx_get_error(uint32_t* bits, int32_t clear, void* stream) {
  g_msg[0] = 0;
  if (!bits) return fail(FP4IDX_EINVAL, "bits is NULL");
  DeviceInfo* dev;
  fp4idx_status_t s = device_info(&dev);
  if (s != FP4IDX_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  if ((e = cudaMemcpy(bits, dev->err, sizeof(uint32_t), cudaMemcpyDeviceToHost)) != cudaSuccess)
    return cuda_fail(e, "read error word");
  if (clear && (e = cudaMemset(dev->err, 0, sizeof(uint32_t))) != cudaSuccess)
    return cuda_fail(e, "clear error word");
  return FP4IDX_OK;
}

}  // extern "C"
