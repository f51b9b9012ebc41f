// gemm_block.cu -- instantiations of the block-scaled (FP32 128x128 / 1x128
// scales) FP8 GEMM: the prefill tile and the swapped decode tiles.
#include "gemm_kernel.cuh"

namespace fp8bq {

cudaError_t run_block_normal(const GemmArgs &a, const void *q, const void *w,
                             const LaunchShape &sh, int grid, cudaStream_t st, int *status) {
  return run<kModeBlock, false, 256, 4, 8>(a, q, w, sh, grid, st, status);
}

cudaError_t run_block_swap(int bn, const GemmArgs &a, const void *q, const void *w,
                           const LaunchShape &sh, int grid, cudaStream_t st, int *status) {
  switch (bn) {
    case 16: return run<kModeBlock, true, 16, 8, 4>(a, q, w, sh, grid, st, status);
    case 32: return run<kModeBlock, true, 32, 8, 4>(a, q, w, sh, grid, st, status);
    default: return run<kModeBlock, true, 64, 8, 4>(a, q, w, sh, grid, st, status);
  }
}

}  // namespace fp8bq
