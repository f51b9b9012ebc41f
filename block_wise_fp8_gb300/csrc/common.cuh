// common.cuh -- shared definitions of the CUDA library (host and device).
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>
#include <utility>

namespace fp8bq {

constexpr int kBlockK = 128;  // K width of one scale block / one pipeline stage
constexpr int kBlockN = 128;  // rows of W sharing one weight scale
constexpr int kMxGroup = 32;  // K elements per UE8M0 scale
constexpr int kMaxParts = 64; // static path: maximum number of output partitions
constexpr int kMxBN = 224;    // weight rows per MXFP8 tile (must match gemm_mx.cu)
constexpr int kMaxExperts = 1024;  // grouped GEMM: most expert segments per call
// grouped GEMM: shared memory of the per-CTA tile table (first m-tile, first
// row and end row of every expert segment, int32)
constexpr int kGroupTableBytes = (3 * kMaxExperts + 1) * 4;

// Status values stored in the workspace status word (same numbers as fp8bq_status).
constexpr uint32_t kStatusTimeout = 8;
constexpr uint32_t kStatusBounds = 9;  // a debug build's bounds check caught a write

// Every kernel of the library is launched with programmatic stream
// serialization: it may start while the preceding kernel of the stream is
// finishing, and it executes griddepcontrol.wait before it reads or writes any
// global memory that another kernel may produce or consume (the GEMMs only
// prefetch weight tiles into L2 before that point).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t st, Args &&...args) {
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// ---------------------------------------------------------------- quant kernels

void launch_quant_group(const void *x, int64_t M, int64_t K, int64_t ldx, void *q, float *s,
                        int s_layout, int num_sms, cudaStream_t st);
void launch_quant_mx(const void *x, int64_t M, int64_t K, int64_t ldx, void *q, uint8_t *s,
                     int num_sms, cudaStream_t st);
void launch_quant_static(const void *x, int64_t M, int64_t K, int64_t ldx, const float *s,
                         void *q, int num_sms, cudaStream_t st);
// Group-128 quantisation with power-of-two (UE8M0) scales, u[M][ceil(K/128)].
void launch_quant_group_ue8m0(const void *x, int64_t M, int64_t K, int64_t ldx, void *q,
                              uint8_t *u, int num_sms, cudaStream_t st);
// FP32 128x128 weight block scales -> UE8M0 (rounded up), codes re-encoded.
void launch_requant_ue8m0(const void *q, const float *s, int64_t N, int64_t K, void *q2, uint8_t *u,
                          cudaStream_t st);
// One scale per row: s[i] = max(amax_i, 1e-10) / 448, q = RNE_sat(x / s[i]).
void launch_quant_token(const void *x, int64_t M, int64_t K, int64_t ldx, void *q, float *s,
                        int num_sms, cudaStream_t st);
// Residual add + RMSNorm, then (q != null) group-128 quantisation (s_x == null)
// or static quantisation with the scale s_x[0].  res, r_out, y may be null.
cudaError_t launch_add_rmsnorm(const void *x, int64_t ldx, const void *res, int64_t ldr,
                               void *r_out, const void *g, float eps, int64_t M, int64_t K,
                               void *y, void *q, float *s, int s_layout, const float *s_x,
                               int num_sms, cudaStream_t st);
void launch_quant_weight_block(const void *w, int64_t N, int64_t K, int64_t ldw, void *q,
                               float *s, cudaStream_t st);
void launch_absmax_scale(const void *x, int64_t rows, int64_t K, int64_t ldx, float *s,
                         int num_sms, cudaStream_t st);
// Counts unusable FP32 scales (out[0] the sentinel -FLT_MAX, out[1] NaN / inf,
// out[2] other values <= 0) and the smallest bad index (out[3]; above every
// index when there is none).  `out` is device memory of 4 words.
void launch_check_scales(const float *s, int64_t n, unsigned long long *out, int num_sms,
                         cudaStream_t st);
// codes[i] = the quantisers' binary32 -> E4M3 conversion of bit pattern first + i
// (i < n); `codes` 8-byte aligned.
void launch_e4m3_bits(uint32_t first, int64_t n, uint8_t *codes, int num_sms, cudaStream_t st);

// ---------------------------------------------------------------- GEMM

// kModeChannel: one FP32 scale per token (activation row) and per output
// channel (weight row), applied after the full-K sum like kModeTensor's
enum GemmMode : int { kModeBlock = 0, kModeTensor = 1, kModeMx = 2, kModeChannel = 3 };

// Everything a GEMM launch needs besides the two tensor maps.
struct GemmArgs {
  int mode;
  int M, N, K;
  // block path; the channel path uses sx [M] (per token) and sw [N] (per
  // output channel)
  const float *sx;
  int sx_layout;  // 0 row-major [M][KB], 1 column-major [KB][ldsx]
  int ldsx;       // KB for row-major, round_up(M,4) for column-major
  const float *sw;
  int sc_tma;     // set by the launcher: s_x and s_w reach the epilogue through TMA
  // static path
  const float *sx_scalar;
  const float *sw_part;
  int n_parts;
  int part_end[kMaxParts];
  // MX path
  const uint8_t *ux;
  const uint8_t *uw;
  // epilogue
  const void *bias;
  void *y;
  int y_tma;  // set by the launcher: Y is written with TMA stores
  // grouped (MoE) form, g_experts > 0: A and Y rows are split into one segment
  // per expert (contiguous: rows g_offsets[e] .. g_offsets[e+1]-1; masked: the
  // first g_masked[e] of the g_max_m rows from e * g_max_m), B is [E * N, K]
  // (expert e's weight at rows e * N) and s_w [E * ceil(N/128)][KB]
  int g_experts;
  const int *g_offsets;
  const int *g_masked;
  int g_max_m;
  int g_tile_cap;  // most m-tiles the segments can hold (set by the launcher)
  // workspace
  uint32_t *status;
  uint32_t *counters;
  float *partials;
  int64_t partials_bytes;  // room behind `partials` (0: no split tail tiles)
  uint64_t wait_limit_ns;
  // fault injection for the timeout tests (0 in normal use): CTA 0 issues no
  // copy for its first K block, so the waits on that stage run out
  int fault_skip_first_load;
  // fused decode linear: the BF16 activations [M, K] (pitch ldxq elements)
  // that the GEMM quantises itself; nullptr otherwise
  const void *xq;
  int64_t ldxq;
  // decode tiles: token rows of the B operand each stage copies (set by the
  // launcher: M rounded up to 8, at most the tile's width)
  int b_box_rows;
};

struct DeviceInfo {
  int num_sms;
  int cc_major, cc_minor;
  size_t max_smem_optin;
};

// Workspace layout (byte offsets), shared by the host entry points.
struct WorkspaceLayout {
  size_t status, counters, partials, q, s, sfa, sfb, total;
};

// MXFP8 scale-factor chunks, the form the MX GEMM loads with each operand stage:
// per row tile and 128-wide K block, 32 rows of 16 bytes per 32 x 4 block of
// codes (word c of row i = the four codes of tile row i + 32c).  Activations:
// 128-row tiles, one 512-byte block; weights: kMxBN-row tiles, kMxSfBBlocks.
constexpr int kMxSfBBlocks = (kMxBN / 32 + 3) / 4;
inline int64_t mx_sfa_bytes(int64_t M, int64_t K) { return (M + 127) / 128 * ((K + 127) / 128) * 512; }
inline int64_t mx_sfb_bytes(int64_t N, int64_t K) {
  return (N + kMxBN - 1) / kMxBN * ((K + 127) / 128) * 512 * kMxSfBBlocks;
}
// Rearranges s_x [M, K/32] and s_w [N, K/32] (row-major UE8M0) into chunks.
void launch_mx_sf_tiles(const uint8_t *ux, int64_t M, const uint8_t *uw, int64_t N, int64_t K,
                        uint8_t *sfa, uint8_t *sfb, int num_sms, cudaStream_t st);
// The same chunks from 128-wide block codes: s_x [M][ceil(K/128)] and s_w
// [ceil(N/128)][ceil(K/128)], each code standing for four 32-groups (and for
// the 128 weight rows of its block).
void launch_ue8m0_sf_tiles(const uint8_t *ux, int64_t M, const uint8_t *uw, int64_t N, int64_t K,
                           uint8_t *sfa, uint8_t *sfb, int num_sms, cudaStream_t st);
// Block pair tiles whose K range is split (the last wave's tiles): each split
// publishes its CTA's promoted 128 x 256 FP32 accumulators (128 KB).  At most
// kMaxTailItems splits per launch (more than the clusters a GB300 holds).
constexpr int kMaxTailItems = 80;
constexpr int64_t kTailItemBytes = 2 * 128 * 256 * 4;  // both CTAs of a pair
// `tail`: reserve the split-tail partials (block GEMM and linear, M > 64)
WorkspaceLayout workspace_layout(int op, int64_t M, int64_t N, int64_t K, bool tail = true);

// Work decomposition of one GEMM launch.
struct LaunchShape {
  int units;        // work units (output tiles, times splits in the swapped form)
  int num_a_tiles;  // A-operand row tiles (128 rows; 256 for pair tiles)
  int splits;       // K splits per tile (swapped form only)
  int kps;          // K blocks per split
  int KB;           // ceil(K / 128)
  int sx_stage;     // floats of shared memory staging s_x (swapped block form)
  // block pair tiles: the first full_units units are whole tiles; the tiles
  // after them (the last, partly filled wave) are split over tail_splits K
  // ranges of tail_kps blocks each, one unit per range (full_units = units
  // and tail_splits = 1 when nothing is split)
  int full_units;
  int tail_splits;
  int tail_kps;
};

// K-major E4M3 matrix [rows, K] (pitch K bytes) as a TMA map with a
// [box_rows x 128 B] box and 128-byte swizzling.
bool make_kmajor_map(CUtensorMap *m, const void *base, int64_t rows, int64_t K, int box_rows);
// The same through a small per-process cache of recently encoded maps.
bool cached_kmajor_map(CUtensorMap *m, const void *base, int64_t rows, int64_t K,
                       int box_rows);
// FP32 matrix [rows, cols] (row pitch `pitch` floats, a multiple of 4) as a TMA
// map with a [box_rows x box_cols] box, no swizzle; through a small cache.
bool cached_f32_map(CUtensorMap *m, const void *base, int64_t rows, int64_t cols,
                    int64_t pitch, int box_cols, int box_rows);
// Row-major BF16 matrix [rows, cols] (pitch 2*cols bytes, cols % 8 == 0) as a
// TMA map with a [box_rows x box_cols] box, 128-byte swizzled (box_cols = 64),
// through a small cache like the one above.
bool cached_bf16_rows_map(CUtensorMap *m, const void *base, int64_t rows, int64_t cols,
                          int box_cols, int box_rows);
// BF16 [rows, cols] with a row pitch of `pitch` elements, unswizzled boxes of
// [box_rows x box_cols] (the fused decode linear's activations)
bool cached_bf16_pitched_map(CUtensorMap *m, const void *base, int64_t rows, int64_t cols,
                             int64_t pitch, int box_cols, int box_rows);

// Kernel variants, one translation unit each (instantiated from gemm_kernel.cuh).
// Pair (prefill) forms: `bn` is the weight-row tile, 192 or 256, and `grid` the
// number of CTA pairs.  Swapped (decode) forms: `bn` is the token tile, 16, 32
// or 64, and `grid` the number of CTAs.
cudaError_t run_block_pair(int bn, const GemmArgs &a, const void *q, const void *w,
                           const LaunchShape &sh, int grid, cudaStream_t st, int *status);
// Grouped block GEMM: 256 x 256 pair tiles (`grid` pairs) or single-CTA
// 128 x 256 tiles (`grid` CTAs).
cudaError_t run_block_grouped(bool pair, const GemmArgs &a, const void *q, const void *w,
                              const LaunchShape &sh, int grid, cudaStream_t st, int *status);
cudaError_t run_block_swap_fused(int bn, const GemmArgs &a, const void *w, const LaunchShape &sh,
                                 int grid, cudaStream_t st, int *status);
cudaError_t run_block_swap(int bn, const GemmArgs &a, const void *q, const void *w,
                           const LaunchShape &sh, int grid, cudaStream_t st, int *status);
cudaError_t run_tensor_pair(int bn, const GemmArgs &a, const void *q, const void *w,
                            const LaunchShape &sh, int grid, cudaStream_t st, int *status);
cudaError_t run_tensor_swap(int bn, const GemmArgs &a, const void *q, const void *w,
                            const LaunchShape &sh, int grid, cudaStream_t st, int *status);
cudaError_t run_channel_pair(int bn, const GemmArgs &a, const void *q, const void *w,
                             const LaunchShape &sh, int grid, cudaStream_t st, int *status);
cudaError_t run_channel_swap(int bn, const GemmArgs &a, const void *q, const void *w,
                             const LaunchShape &sh, int grid, cudaStream_t st, int *status);
cudaError_t run_mx_normal(const GemmArgs &a, const void *q, const void *w,
                          const LaunchShape &sh, int grid, cudaStream_t st, int *status);
cudaError_t run_mx_pair(const GemmArgs &a, const void *q, const void *w, const LaunchShape &sh,
                        int grid, cudaStream_t st, int *status);

// Chooses the kernel variant for the shape and launches it.  Returns 0 or an
// fp8bq status; a CUDA error is returned through `cuda_err`.
int launch_gemm(const GemmArgs &a, const void *q_act, const void *w, const DeviceInfo &dev,
                cudaStream_t st, cudaError_t *cuda_err);
// K split of the decode tiles (M <= 64): the number of splits (0 if K is too
// large for them) and, in *kps, the K blocks per split
int decode_splits(int64_t N, int64_t K, int num_sms, int *kps);

}  // namespace fp8bq
