// score_mx.cu -- MXFP4 (E8M0 per 32 values) instantiations of the scorer.
#include "score_kernel.cuh"

namespace fp4idx {
cudaError_t launch_score_mx(const ScoreParams& p, int mode, int heads, dim3 grid, cudaStream_t stream) {
  return launch_score_fmt<0>(p, mode, heads, grid, stream);
}
}  // namespace fp4idx
