// gemm_tensor.cu -- instantiations of the per-tensor (static) FP8 GEMM.
#include "gemm_kernel.cuh"

namespace fp8bq {

cudaError_t run_tensor_normal(const GemmArgs &a, const void *q, const void *w,
                              const LaunchShape &sh, int grid, cudaStream_t st, int *status) {
  return run<kModeTensor, false, 256, 4, 8>(a, q, w, sh, grid, st, status);
}

cudaError_t run_tensor_swap(int bn, const GemmArgs &a, const void *q, const void *w,
                            const LaunchShape &sh, int grid, cudaStream_t st, int *status) {
  switch (bn) {
    case 16: return run<kModeTensor, true, 16, 8, 4>(a, q, w, sh, grid, st, status);
    case 32: return run<kModeTensor, true, 32, 8, 4>(a, q, w, sh, grid, st, status);
    default: return run<kModeTensor, true, 64, 8, 4>(a, q, w, sh, grid, st, status);
  }
}

}  // namespace fp8bq
