// gemm_mx.cu -- instantiation of the MXFP8 block-scaled FP8 GEMM.
#include "gemm_kernel.cuh"

namespace fp8bq {

cudaError_t run_mx_normal(const GemmArgs &a, const void *q, const void *w,
                          const LaunchShape &sh, int grid, cudaStream_t st, int *status) {
  return run<kModeMx, false, kMxBN, 4, 4, 2, false>(a, q, w, sh, grid, st, status);
}

cudaError_t run_mx_pair(const GemmArgs &a, const void *q, const void *w, const LaunchShape &sh,
                        int grid, cudaStream_t st, int *status) {
  return run<kModeMx, false, kMxBN, 6, 8, 2, true>(a, q, w, sh, grid, st, status);
}

}  // namespace fp8bq

// ------------------------------------------------------------ scale-factor chunks
namespace fp8bq {
namespace {

struct SfJob {
  const uint8_t *u;  // [rows, G] row-major UE8M0 codes
  uint8_t *out;      // chunks
  int64_t rows;
  int tile_rows;     // rows per tile
  int blocks;        // 512-byte blocks per chunk (32 x 4 codes each)
  int64_t n;         // 16-byte chunk rows to write: tiles * KB * blocks * 32
  int rdiv;          // rows sharing one code row (128 for 128 x 128 weight blocks)
};

// Four codes (K groups 4kb..4kb+3) of one row, little-endian; 0 past the row's end
__device__ __forceinline__ uint32_t sf_codes(const uint8_t *u, int64_t row, int G, int kb,
                                             bool words) {
  const uint8_t *p = u + row * G + 4 * kb;
  if (words) return __ldg(reinterpret_cast<const uint32_t *>(p));
  uint32_t v = 0;
  for (int g = 0; g < 4; ++g)
    if (4 * kb + g < G) v |= static_cast<uint32_t>(__ldg(p + g)) << (8 * g);
  return v;
}

// One thread per 16-byte chunk row: chunk (t, kb), block h, row i holds the codes
// of tile rows i + 32(4h + c), c = 0..3 (code 0 = 2^-127 outside the tile or the
// matrix, where the operand's data are zero-filled).
// g128: the codes are one per 128-wide K block (u[row / rdiv][kb], KB per row),
// each standing for the four 32-groups of its block.
__global__ void __launch_bounds__(256) mx_sf_tile_kernel(SfJob ja, SfJob jb, int G, int KB,
                                                         int words, int g128) {
  griddep_launch_dependents();
  griddep_wait();
  const int64_t total = ja.n + jb.n;
  for (int64_t x = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; x < total;
       x += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const bool is_a = x < ja.n;
    const SfJob &j = is_a ? ja : jb;
    const int64_t y = is_a ? x : x - ja.n;
    const int i = static_cast<int>(y & 31);
    int64_t r = y >> 5;
    const int h = static_cast<int>(r % j.blocks);
    r /= j.blocks;
    const int kb = static_cast<int>(r % KB);
    const int64_t t = r / KB;
    uint32_t v[4];
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const int local = i + 32 * (4 * h + c);
      const int64_t row = t * j.tile_rows + local;
      if (local < j.tile_rows && row < j.rows)
        v[c] = g128 ? __ldg(j.u + (row / j.rdiv) * KB + kb) * 0x01010101u
                    : sf_codes(j.u, row, G, kb, words != 0);
      else
        v[c] = 0u;
    }
    *reinterpret_cast<uint4 *>(j.out + ((t * KB + kb) * j.blocks + h) * 512 + 16 * i) =
        make_uint4(v[0], v[1], v[2], v[3]);
  }
}

}  // namespace

void launch_mx_sf_tiles(const uint8_t *ux, int64_t M, const uint8_t *uw, int64_t N, int64_t K,
                        uint8_t *sfa, uint8_t *sfb, int num_sms, cudaStream_t st) {
  const int G = static_cast<int>(K / 32);
  const int KB = static_cast<int>((K + 127) / 128);
  SfJob ja{ux, sfa, M, 128, 1, (M + 127) / 128 * KB * 32, 1};
  SfJob jb{uw, sfb, N, kMxBN, kMxSfBBlocks, (N + kMxBN - 1) / kMxBN * KB * kMxSfBBlocks * 32, 1};
  const bool words = (G % 4 == 0) && (reinterpret_cast<uintptr_t>(ux) & 3u) == 0 &&
                     (reinterpret_cast<uintptr_t>(uw) & 3u) == 0;
  const int64_t total = ja.n + jb.n;
  int64_t grid = (total + 255) / 256;
  if (grid > 4L * num_sms) grid = 4L * num_sms;
  if (grid < 1) grid = 1;
  launch_pdl(mx_sf_tile_kernel, dim3(static_cast<unsigned>(grid)), dim3(256), 0, st, ja, jb, G,
             KB, words ? 1 : 0, 0);
}

void launch_ue8m0_sf_tiles(const uint8_t *ux, int64_t M, const uint8_t *uw, int64_t N, int64_t K,
                           uint8_t *sfa, uint8_t *sfb, int num_sms, cudaStream_t st) {
  const int KB = static_cast<int>((K + 127) / 128);
  SfJob ja{ux, sfa, M, 128, 1, (M + 127) / 128 * KB * 32, 1};
  SfJob jb{uw, sfb, N, kMxBN, kMxSfBBlocks, (N + kMxBN - 1) / kMxBN * KB * kMxSfBBlocks * 32, 128};
  const int64_t total = ja.n + jb.n;
  int64_t grid = (total + 255) / 256;
  if (grid > 4L * num_sms) grid = 4L * num_sms;
  if (grid < 1) grid = 1;
  launch_pdl(mx_sf_tile_kernel, dim3(static_cast<unsigned>(grid)), dim3(256), 0, st, ja, jb, KB,
             KB, 0, 1);
}

}  // namespace fp8bq
