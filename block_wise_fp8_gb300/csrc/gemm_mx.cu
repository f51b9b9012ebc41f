// gemm_mx.cu -- instantiation of the MXFP8 block-scaled FP8 GEMM.
#include "gemm_kernel.cuh"

namespace fp8bq {

cudaError_t run_mx_normal(const GemmArgs &a, const void *q, const void *w,
                          const LaunchShape &sh, int grid, cudaStream_t st, int *status) {
  return run<kModeMx, false, 128, 6, 4, 2, false>(a, q, w, sh, grid, st, status);
}

}  // namespace fp8bq
