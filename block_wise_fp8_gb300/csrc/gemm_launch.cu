// gemm_launch.cu -- host side of the GEMMs: TMA tensor maps, workspace layout
// and the choice of kernel variant and work decomposition for a shape.
#include <cudaTypedefs.h>

#include <mutex>

#include "common.cuh"

namespace fp8bq {
namespace {

PFN_cuTensorMapEncodeTiled_v12000 get_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

constexpr int kMaxSplits = 8;

}  // namespace

// Decode (M <= 64) tiles: 128 weight rows each, the K blocks split over
// splits CTAs so that tiles x splits fills the SMs (at most kMaxSplits, each
// split at most 64 K blocks, no empty split).  Returns the split count and
// the K blocks per split, or 0 when K needs more than kMaxSplits x 64 blocks.
int decode_splits(int64_t N, int64_t K, int num_sms, int *kps_out) {
  const int KB = static_cast<int>((K + 127) / 128);
  const int tiles = static_cast<int>((N + 127) / 128);
  int splits = num_sms / tiles;
  if (splits < 1) splits = 1;
  if (splits > kMaxSplits) splits = kMaxSplits;
  if (splits > KB) splits = KB;
  int kps = (KB + splits - 1) / splits;
  while (kps > 64 && splits < kMaxSplits) {  // bounds the s_x staging buffer
    ++splits;
    kps = (KB + splits - 1) / splits;
  }
  if (kps > 64) return 0;
  *kps_out = kps;
  return (KB + kps - 1) / kps;  // no empty split
}

bool make_kmajor_map(CUtensorMap *m, const void *base, int64_t rows, int64_t K, int box_rows) {
  auto enc = get_encoder();
  if (!enc) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(K)};
  cuuint32_t box[2] = {128u, static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estr[2] = {1u, 1u};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(base), dims, strides,
                   box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Small cache of encoded tensor maps keyed by (base, rows, K, box rows): repeated
// calls on the same tensors (every forward of a layer) skip the host-side encode.
bool cached_kmajor_map(CUtensorMap *m, const void *base, int64_t rows, int64_t K,
                       int box_rows) {
  struct Entry {
    const void *base;
    int64_t rows, K;
    int box;
    CUtensorMap map;
  };
  constexpr int kEntries = 32;
  static Entry cache[kEntries];
  static int used = 0, next = 0;
  static std::mutex mu;
  {
    std::lock_guard<std::mutex> g(mu);
    for (int i = 0; i < used; ++i)
      if (cache[i].base == base && cache[i].rows == rows && cache[i].K == K &&
          cache[i].box == box_rows) {
        *m = cache[i].map;
        return true;
      }
  }
  if (!make_kmajor_map(m, base, rows, K, box_rows)) return false;
  std::lock_guard<std::mutex> g(mu);
  Entry &e = cache[next];
  e.base = base;
  e.rows = rows;
  e.K = K;
  e.box = box_rows;
  e.map = *m;
  next = (next + 1) % kEntries;
  if (used < kEntries) ++used;
  return true;
}

bool cached_f32_map(CUtensorMap *m, const void *base, int64_t rows, int64_t cols,
                    int64_t pitch, int box_cols, int box_rows) {
  struct Entry {
    const void *base;
    int64_t rows, cols, pitch;
    int bc, br;
    CUtensorMap map;
  };
  constexpr int kEntries = 16;
  static Entry cache[kEntries];
  static int used = 0, next = 0;
  static std::mutex mu;
  {
    std::lock_guard<std::mutex> g(mu);
    for (int i = 0; i < used; ++i)
      if (cache[i].base == base && cache[i].rows == rows && cache[i].cols == cols &&
          cache[i].pitch == pitch && cache[i].bc == box_cols && cache[i].br == box_rows) {
        *m = cache[i].map;
        return true;
      }
  }
  auto enc = get_encoder();
  if (!enc) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(pitch) * 4};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(box_cols), static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estr[2] = {1u, 1u};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void *>(base), dims, strides,
                   box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                   CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return false;
  std::lock_guard<std::mutex> g(mu);
  Entry &e = cache[next];
  e.base = base;
  e.rows = rows;
  e.cols = cols;
  e.pitch = pitch;
  e.bc = box_cols;
  e.br = box_rows;
  e.map = *m;
  next = (next + 1) % kEntries;
  if (used < kEntries) ++used;
  return true;
}

bool cached_bf16_rows_map(CUtensorMap *m, const void *base, int64_t rows, int64_t cols,
                          int box_cols, int box_rows) {
  struct Entry {
    const void *base;
    int64_t rows, cols;
    int bc, br;
    CUtensorMap map;
  };
  constexpr int kEntries = 16;
  static Entry cache[kEntries];
  static int used = 0, next = 0;
  static std::mutex mu;
  {
    std::lock_guard<std::mutex> g(mu);
    for (int i = 0; i < used; ++i)
      if (cache[i].base == base && cache[i].rows == rows && cache[i].cols == cols &&
          cache[i].bc == box_cols && cache[i].br == box_rows) {
        *m = cache[i].map;
        return true;
      }
  }
  auto enc = get_encoder();
  if (!enc) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * 2};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(box_cols), static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estr[2] = {1u, 1u};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims,
                   strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return false;
  std::lock_guard<std::mutex> g(mu);
  Entry &e = cache[next];
  e.base = base;
  e.rows = rows;
  e.cols = cols;
  e.bc = box_cols;
  e.br = box_rows;
  e.map = *m;
  next = (next + 1) % kEntries;
  if (used < kEntries) ++used;
  return true;
}

bool cached_bf16_pitched_map(CUtensorMap *m, const void *base, int64_t rows, int64_t cols,
                             int64_t pitch, int box_cols, int box_rows) {
  struct Entry {
    const void *base;
    int64_t rows, cols, pitch;
    int bc, br;
    CUtensorMap map;
  };
  constexpr int kEntries = 16;
  static Entry cache[kEntries];
  static int used = 0, next = 0;
  static std::mutex mu;
  {
    std::lock_guard<std::mutex> g(mu);
    for (int i = 0; i < used; ++i)
      if (cache[i].base == base && cache[i].rows == rows && cache[i].cols == cols &&
          cache[i].pitch == pitch && cache[i].bc == box_cols && cache[i].br == box_rows) {
        *m = cache[i].map;
        return true;
      }
  }
  auto enc = get_encoder();
  if (!enc) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(pitch) * 2};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(box_cols), static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estr[2] = {1u, 1u};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims,
                   strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return false;
  std::lock_guard<std::mutex> g(mu);
  Entry &e = cache[next];
  e.base = base;
  e.rows = rows;
  e.cols = cols;
  e.pitch = pitch;
  e.bc = box_cols;
  e.br = box_rows;
  e.map = *m;
  next = (next + 1) % kEntries;
  if (used < kEntries) ++used;
  return true;
}

// [status word | split-K tile counters | split-K FP32 partials | fused: Q | fused: scales |
//  MX: activation and weight scale-factor chunks]
WorkspaceLayout workspace_layout(int op, int64_t M, int64_t N, int64_t K, bool tail) {
  auto up = [](size_t v) { return (v + 255) / 256 * 256; };
  WorkspaceLayout L{};
  const int64_t KB = (K + 127) / 128;
  const int64_t NT = (N + 127) / 128;
  L.status = 0;
  L.counters = 256;
  // one counter per 128 output columns (split-K decode tiles), and two per
  // split tail tile of the block pair form
  size_t off = L.counters + up(static_cast<size_t>(NT > 2 * kMaxTailItems ? NT : 2 * kMaxTailItems) * 4);
  L.partials = off;
  const bool mx = (op == 2 || op == 3 || op == 8 || op == 9);  // MX GEMM (UE8M0 views too)
  const bool grouped = (op == 10);  // pair tiles at every M: no split-K partials
  const bool block = (op == 0 || op == 1);
  if (M <= 64 && !mx && !grouped) {
    // decode split-K partials, one FP32 slot per split, token and weight row
    // (room for the token count rounded up to 4)
    off += up(static_cast<size_t>(kMaxSplits) * ((M + 3) / 4 * 4) * N * 4);
  } else if (block && tail) {
    // split tail tiles: at most 4 K ranges per pair tile (256 rows by at least
    // 192 weight rows, the narrowest pair tile), and kMaxTailItems
    const int64_t tiles = (M + 255) / 256 * ((N + 191) / 192);
    const int64_t items = 4 * tiles < kMaxTailItems ? 4 * tiles : kMaxTailItems;
    off += up(static_cast<size_t>(items * kTailItemBytes));
  }
  L.q = off;
  const bool fused = (op == 1 || op == 3 || op == 5 || op == 7 || op == 9);
  if (fused) off += up(static_cast<size_t>(M) * K);
  L.s = off;
  if (op == 1) off += up(static_cast<size_t>(M) * KB * 4);
  if (op == 3) off += up(static_cast<size_t>(M) * (K / 32));
  if (op == 7) off += up(static_cast<size_t>(M) * 4);  // one FP32 scale per token
  if (op == 9) off += up(static_cast<size_t>(M) * KB);  // one UE8M0 code per 128-group
  L.sfa = off;
  if (mx) off += up(static_cast<size_t>(mx_sfa_bytes(M, K)));
  L.sfb = off;
  if (mx) off += up(static_cast<size_t>(mx_sfb_bytes(N, K)));
  L.total = off;
  return L;
}

int launch_gemm(const GemmArgs &a, const void *q_act, const void *w, const DeviceInfo &dev,
                cudaStream_t st, cudaError_t *cuda_err) {
  *cuda_err = cudaSuccess;
  int status = 0;
  LaunchShape sh{};
  sh.KB = (a.K + 127) / 128;
  if (a.g_experts > 0) {
    // grouped (MoE) form: block tiles over the table each CTA builds from the
    // segment bounds, weight tiles fastest (the tiles of one m-tile run side by
    // side and share its activation rows in L2).  Each segment rounds up to whole
    // m-tiles, so with few rows per expert the padding decides the tensor
    // work: 128-row single-CTA tiles while the mean segment is at most 512 rows
    // (and always for the masked layout, whose slots are mostly unfilled),
    // 256-row pair tiles above.  The host knows only a bound on the tile
    // count, so the persistent grid covers that bound and CTAs without work
    // leave at once.
    if (a.mode != kModeBlock || a.g_experts > kMaxExperts) return 4;
    const bool masked = a.g_offsets == nullptr;
    const bool pair = !masked && a.M > 512L * a.g_experts;
    const int rows = pair ? 256 : 128;
    GemmArgs g = a;
    // each segment has at most one ragged tile
    g.g_tile_cap = masked ? a.g_experts * ((a.g_max_m + rows - 1) / rows)
                          : a.g_experts + (a.M + rows - 1) / rows;
    const int slots = pair ? dev.num_sms / 2 : dev.num_sms;
    const long units_cap = static_cast<long>(g.g_tile_cap) * ((a.N + 255) / 256);
    sh.num_a_tiles = 0;
    sh.units = 0;
    sh.splits = 1;
    sh.kps = sh.KB;
    sh.sx_stage = 3 * a.g_experts + 1;  // the table, in 4-byte words
    const int grid = static_cast<int>(units_cap < slots ? units_cap : slots);
    if (grid == 0) return 0;
    *cuda_err = run_block_grouped(pair, g, q_act, w, sh, grid, st, &status);
    return status;
  }
  const bool swap = (a.mode != kModeMx) && a.M <= 64;
  if (swap) {
    // decode: weight rows on the MMA's M side, tokens on its N side, K split so
    // that tiles x splits fills the SMs; split 0 of each tile sums the partials
    const int tiles = (a.N + 127) / 128;
    int kps = 0;
    const int splits = decode_splits(a.N, a.K, dev.num_sms, &kps);
    if (splits == 0) return 4;  // FP8BQ_ERR_UNSUPPORTED: K too large for the decode tile
    sh.splits = splits;
    sh.kps = kps;
    sh.num_a_tiles = tiles;
    sh.units = tiles * splits;
    const int bn = a.M <= 16 ? 16 : a.M <= 32 ? 32 : 64;
    sh.sx_stage = (a.mode == kModeBlock) ? bn * kps : 0;
    if (a.xq) {
      // fused decode linear: the GEMM quantises the activations itself
      if (a.mode != kModeBlock) return 4;
      *cuda_err = run_block_swap_fused(bn, a, w, sh, sh.units, st, &status);
      return status;
    }
    *cuda_err = (a.mode == kModeBlock)     ? run_block_swap(bn, a, q_act, w, sh, sh.units, st, &status)
                : (a.mode == kModeChannel) ? run_channel_swap(bn, a, q_act, w, sh, sh.units, st, &status)
                                           : run_tensor_swap(bn, a, q_act, w, sh, sh.units, st, &status);
    return status;
  }
  if (a.mode == kModeMx) {
    // MXFP8: 224-wide weight tiles, persistent CTAs, M fastest.  224 is the
    // widest UMMA N for which two accumulators and the scale-factor slots fit
    // in the 512 TMEM columns (2 x 224 + 64), so the epilogue of one tile
    // overlaps the MMAs of the next.  Above 128 tokens, CTA pairs take 256 x 224
    // tiles (each CTA loads half the weight tile); otherwise single CTAs take
    // 128 x 224 tiles.
    const bool pair = a.M > 128;
    const int rows = pair ? 256 : 128;
    sh.num_a_tiles = (a.M + rows - 1) / rows;
    sh.splits = 1;
    sh.kps = sh.KB;
    sh.units = sh.num_a_tiles * ((a.N + kMxBN - 1) / kMxBN);
    sh.sx_stage = 0;
    const int slots = pair ? dev.num_sms / 2 : dev.num_sms;
    const int grid = sh.units < slots ? sh.units : slots;
    *cuda_err = pair ? run_mx_pair(a, q_act, w, sh, grid, st, &status)
                     : run_mx_normal(a, q_act, w, sh, grid, st, &status);
    return status;
  }
  // prefill: CTA pairs over 256 x bn tiles, persistent clusters, M fastest.  The
  // weight tile width bn is the one with the least (waves x bn x time per
  // column), i.e. the smallest tail when the tiles are dealt to the pairs; a
  // 256-wide tile takes about 20 % less time per column than a 192-wide one
  // (measured on GB300: channel scaling 4096 x 24576 x 6144 in 345 us against
  // 406 us).
  const int pairs = dev.num_sms / 2;
  sh.num_a_tiles = (a.M + 255) / 256;
  int best_bn = 256;
  long best_cost = -1;
  for (int bn : {256, 192}) {
    const long units = static_cast<long>(sh.num_a_tiles) * ((a.N + bn - 1) / bn);
    const long per_col = bn == 256 ? 80 : 100;
    const long cost = (units + pairs - 1) / pairs * bn * per_col;
    if (best_cost < 0 || cost < best_cost) {
      best_cost = cost;
      best_bn = bn;
    }
  }
  sh.splits = 1;
  sh.kps = sh.KB;
  sh.units = sh.num_a_tiles * ((a.N + best_bn - 1) / best_bn);
  sh.sx_stage = 0;
  sh.full_units = sh.units;
  sh.tail_splits = 1;
  sh.tail_kps = sh.KB;
  const int grid = sh.units < pairs ? sh.units : pairs;
  *cuda_err = (a.mode == kModeBlock)     ? run_block_pair(best_bn, a, q_act, w, sh, grid, st, &status)
              : (a.mode == kModeChannel) ? run_channel_pair(best_bn, a, q_act, w, sh, grid, st, &status)
                                         : run_tensor_pair(best_bn, a, q_act, w, sh, grid, st, &status);
  return status;
}

}  // namespace fp8bq
