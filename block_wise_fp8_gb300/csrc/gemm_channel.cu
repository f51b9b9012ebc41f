// gemm_channel.cu -- instantiations of the channelwise FP8 GEMM (one scale per
// token and per output channel); same tile forms as the per-tensor GEMM.
#include "gemm_kernel.cuh"

namespace fp8bq {

cudaError_t run_channel_pair(int bn, const GemmArgs &a, const void *q, const void *w,
                             const LaunchShape &sh, int grid, cudaStream_t st, int *status) {
  if (bn == 192) return run<kModeChannel, false, 192, 8, 8, 2, true>(a, q, w, sh, grid, st, status);
  return run<kModeChannel, false, 256, 7, 8, 2, true>(a, q, w, sh, grid, st, status);
}

cudaError_t run_channel_swap(int bn, const GemmArgs &a, const void *q, const void *w,
                             const LaunchShape &sh, int grid, cudaStream_t st, int *status) {
  switch (bn) {
    case 16: return run<kModeChannel, true, 16, 8, 4, 2, false>(a, q, w, sh, grid, st, status);
    case 32: return run<kModeChannel, true, 32, 8, 4, 2, false>(a, q, w, sh, grid, st, status);
    default: return run<kModeChannel, true, 64, 8, 4, 2, false>(a, q, w, sh, grid, st, status);
  }
}

}  // namespace fp8bq
