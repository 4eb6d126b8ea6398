// topk_noalloc.cu -- fp4idx_topk_noalloc: the top-k path for callers that
// cannot allocate device memory.
//
// Some callers cannot call cudaMalloc: an engine that reserved the GPU's
// memory up front for its own pool (a further cudaMalloc fails or fragments
// that pool), or a latency-critical loop where the synchronisation that
// cudaMalloc/cudaFree imply is not acceptable.  For them this entry point
// runs exactly fp4idx_topk, with the workspace taken from a fixed array in
// the library's own device memory instead of from the caller.
//
// The array is a file-scope __device__ variable, so every GPU that loads
// the library holds kScratchBytes of it until the process exits.  Its
// device address is looked up once per device (cudaGetSymbolAddress, with
// that device current) on the first call made on that device; make that
// first call before capturing any stream.  All calls on a device share the
// array: calls that overlap on the GPU (different streams, no ordering
// between them) race on it and must be serialised by the caller.  The
// top-k workspace needs no initial contents, so nothing is cleared between
// calls.  No cudaMalloc, cudaFree or allocating library routine is called.
#include <mutex>

#include "fp4idx.h"
#include "internal.h"

namespace fp4idx {
namespace {

constexpr size_t kScratchBytes = 128u << 20;  // 128 MiB

static __device__ __align__(256) unsigned char g_topk_scratch[kScratchBytes];

constexpr int kMaxScratchDevices = 64;
void* g_scratch_ptr[kMaxScratchDevices] = {};
std::mutex g_scratch_mutex;

// Device address of g_topk_scratch on the current device (set-up on first use).
fp4idx_status_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    set_last_error("cudaGetDevice: %s", cudaGetErrorString(e));
    return FP4IDX_ECUDA;
  }
  if (dev < 0 || dev >= kMaxScratchDevices) {
    set_last_error("device ordinal %d out of range", dev);
    return FP4IDX_EDEVICE;
  }
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (!g_scratch_ptr[dev]) {
    void* ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_topk_scratch);
    if (e != cudaSuccess || !ptr) {
      set_last_error("cudaGetSymbolAddress(top-k scratch): %s", cudaGetErrorString(e));
      return FP4IDX_ECUDA;
    }
    g_scratch_ptr[dev] = ptr;
  }
  *out = g_scratch_ptr[dev];
  return FP4IDX_OK;
}

}  // namespace
}  // namespace fp4idx

extern "C" {

fp4idx_status_t fp4idx_topk_noalloc(const fp4idx_problem_t* problem, const float* w, int64_t w_row_stride,
                                    int32_t k, uint32_t flags, int32_t* indices, float* values,
                                    int32_t* valid_count, void* stream) {
  // A size of 0 means an invalid or unsupported problem or k: fp4idx_topk
  // below then reports the same status it would give any caller.
  const size_t need = fp4idx_topk_workspace_bytes(problem, k);
  if (need > fp4idx::kScratchBytes) {
    fp4idx::set_last_error("top-k needs %zu bytes of scratch; the static scratch holds %zu (use fp4idx_topk)",
                           need, fp4idx::kScratchBytes);
    return FP4IDX_EWORKSPACE;
  }
  void* scratch = nullptr;
  fp4idx_status_t s = fp4idx::scratch_address(&scratch);
  if (s != FP4IDX_OK) return s;
  return fp4idx_topk(problem, w, w_row_stride, k, flags, indices, values, valid_count, scratch,
                     fp4idx::kScratchBytes, stream);
}

}  // extern "C"
