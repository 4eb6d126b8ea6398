// score_nv.cu -- NVFP4 (E4M3 per 16 values) instantiations of the scorer.
#include "score_kernel.cuh"

namespace fp4idx {
cudaError_t launch_score_nv(const ScoreParams& p, int mode, int heads, dim3 grid, cudaStream_t stream) {
  return launch_score_fmt<1>(p, mode, heads, grid, stream);
}
}  // namespace fp4idx

#ifdef FP4IDX_STAMPS
// Profiling builds only: copy out (and clear) this unit's stamp sums.
extern "C" int fp4idx_stamps_read_nv(unsigned long long* out, int clear) {
  if (cudaMemcpyFromSymbol(out, fp4idx::fp4idx_stamps, sizeof(fp4idx::fp4idx_stamps)) != cudaSuccess) return -1;
  if (clear) {
    static const unsigned long long zero[4 * fp4idx::kStampCats] = {};
    if (cudaMemcpyToSymbol(fp4idx::fp4idx_stamps, zero, sizeof(zero)) != cudaSuccess) return -1;
  }
  return 0;
}
#endif
