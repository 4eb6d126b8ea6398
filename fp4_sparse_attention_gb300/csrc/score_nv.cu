// score_nv.cu -- NVFP4 (E4M3 per 16 values) instantiations of the scorer.
#include "score_kernel.cuh"

namespace fp4idx {
cudaError_t launch_score_nv(const ScoreParams& p, int mode, int heads, dim3 grid, cudaStream_t stream) {
  return launch_score_fmt<1>(p, mode, heads, grid, stream);
}
}  // namespace fp4idx
