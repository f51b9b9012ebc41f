// gemm_block.cu -- instantiations of the block-scaled (FP32 128x128 / 1x128
// scales) FP8 GEMM: the pair prefill tiles, the swapped decode tiles, and the
// grouped (MoE) forms: 256 x 256 pair tiles and single-CTA 128 x 256 tiles.
#include "gemm_kernel.cuh"

namespace fp8bq {

cudaError_t run_block_pair(int bn, const GemmArgs &a, const void *q, const void *w,
                           const LaunchShape &sh, int grid, cudaStream_t st, int *status) {
  if (bn == 192) return run<kModeBlock, false, 192, 6, 12, 2, true>(a, q, w, sh, grid, st, status);
  return run<kModeBlock, false, 256, 5, 8, 2, true>(a, q, w, sh, grid, st, status);
}

cudaError_t run_block_grouped(bool pair, const GemmArgs &a, const void *q, const void *w,
                              const LaunchShape &sh, int grid, cudaStream_t st, int *status) {
  // single-CTA tiles: three 48 KB stages, with the Y staging boxes, the scale
  // ring and the tile table, fill the 227 KB (a fourth stage in place of the
  // staging, with Y stored row by row, measured no faster)
  if (pair) return run<kModeBlock, false, 256, 5, 8, 2, true, true>(a, q, w, sh, grid, st, status);
  return run<kModeBlock, false, 256, 3, 8, 2, false, true>(a, q, w, sh, grid, st, status);
}

// the decode linear with the activation quantisation fused in: each stage also
// holds the BF16 activation slice (256 B per token), so the deeper tiles keep
// fewer stages
cudaError_t run_block_swap_fused(int bn, const GemmArgs &a, const void *w, const LaunchShape &sh,
                                 int grid, cudaStream_t st, int *status) {
  switch (bn) {
    case 16: return run<kModeBlock, true, 16, 8, 4, 8, false, false, true>(a, nullptr, w, sh, grid, st, status);
    case 32: return run<kModeBlock, true, 32, 7, 4, 8, false, false, true>(a, nullptr, w, sh, grid, st, status);
    default: return run<kModeBlock, true, 64, 5, 4, 8, false, false, true>(a, nullptr, w, sh, grid, st, status);
  }
}

cudaError_t run_block_swap(int bn, const GemmArgs &a, const void *q, const void *w,
                           const LaunchShape &sh, int grid, cudaStream_t st, int *status) {
  switch (bn) {
    case 16: return run<kModeBlock, true, 16, 8, 4, 8, false>(a, q, w, sh, grid, st, status);
    case 32: return run<kModeBlock, true, 32, 8, 4, 8, false>(a, q, w, sh, grid, st, status);
    default: return run<kModeBlock, true, 64, 8, 4, 8, false>(a, q, w, sh, grid, st, status);
  }
}

}  // namespace fp8bq
