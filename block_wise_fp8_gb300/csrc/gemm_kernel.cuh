// gemm_kernel.cuh -- FP8 GEMMs on the 5th-generation tensor cores (tcgen05 + TMEM + TMA).
//
// One warp-specialised kernel template covers the three scalings of the pages
// ("SGLang 源码完全拆解(十九)", §一条 GEMM 的三种缩放组合):
//
//   kModeBlock   y = sum_b P_b * s_x[i][b] * s_w[j/128][b]   (128x128 weight blocks,
//                1x128 activation groups).  The tensor core produces P_b, the FP32
//                sum over one 128-wide K block, into TMEM; the epilogue warps read
//                it back and promote it into FP32 registers with one FMA per
//                element and K block (paired FP32 FMAs, two elements per
//                instruction) -- the per-128-K promotion of "GLM-5.3 推理全链路
//                (十七)", DeepSeek-V3 Fig. 7 paragraph.  TMEM holds ACCB partial
//                buffers so the MMA runs up to ACCB K blocks ahead of the promotion.
//   kModeTensor  y = (sum_k q w) * s_x * s_w[p(j)]: full-K accumulation in TMEM,
//                one scale product per column in the epilogue.
//   kModeChannel y = (sum_k q w) * s_x[i] * s_w[j]: as kModeTensor, with one
//                scale per token and per output channel ("SGLang 源码完全拆解
//                (十九)", §一条 GEMM 的三种缩放组合, the M x N outer product).
//   kModeMx      y = sum_g P_g * 2^(ua-127) * 2^(uw-127) with the block-scaled MMA
//                (kind::mxf8f6f4, one UE8M0 scale per 32 K).  The codes arrive
//                pre-arranged (one chunk per row tile and K block) with each
//                operand stage; the MMA thread copies them into TMEM
//                (tcgen05.cp) ahead of its MMAs, so no dequantisation runs in
//                software ("GLM-5.3 推理全链路(十七)", §第7站).
//
// Roles (warp index):
//   0            TMA producer: A and B tiles, 128 K per stage, 128B-swizzled.
//   1            TMEM allocator and single-thread MMA issuer.
//   2 ..         further MMA issuers taking alternate K blocks: block tiles
//                (two; four for the 16- and 32-token decode tiles) and the
//                per-tensor / channel decode tiles (four; two at 64 tokens),
//                whose issuers each accumulate into their own TMEM columns.
//   then         epilogue: TMEM -> registers -> promotion -> BF16 -> global.
//   then         (fused decode linear) the activation quantiser warps.
//
// Tile forms:
//   pair    (prefill) a cluster of two CTAs on two SMs computes a 256 x BN tile
//           with the pair MMA (tcgen05 cta_group::2): each CTA TMA-loads its own
//           128 token rows and half of the BN weight rows, the even CTA issues the
//           MMAs, each CTA's TMEM receives its 128 rows of the result and its own
//           epilogue promotes and stores them.  Persistent clusters walk the tiles
//           M-fastest so concurrent clusters share weight tiles in L2.  Block
//           tiles of a last, partly filled wave are split into K ranges on idle
//           clusters; the last range to finish sums the promoted partials in
//           range order (split_tail_tiles).
//   normal  the same with one CTA: UMMA M = 128 tokens, UMMA N = BN weight rows.
//   swap    UMMA M = 128 weight rows, UMMA N = BN tokens (decode, M <= 64), with
//           split-K across CTAs: split 0 of each weight tile polls the other
//           splits' partials (no counter, no election) and sums them in
//           ascending split order (deterministic).
//   grouped (GROUPED instances, block pair or normal) the MoE form: A and Y rows
//           are split into per-expert segments whose bounds the kernel reads
//           from the device; every CTA builds the m-tile table in shared
//           memory, tiles stop at their segment's end, and B / s_w are the
//           expert's slices of [E * N, K] and [E * ceil(N/128), KB]
//           ("SGLang 源码完全拆解(十九)", §MoE:专家权重多一个维度).
//
// Every wait is bounded (see ptx.cuh); a CTA that gives up records a timeout in
// the workspace status word, lets its in-flight copies and MMAs land, frees its
// TMEM and exits.
#pragma once
#include <cuda_bf16.h>

#include <cstring>
#include <mutex>

#include "common.cuh"
#include "ptx.cuh"
#include "quant_math.cuh"

namespace fp8bq {
namespace {

constexpr int kBM = 128;           // UMMA M
constexpr int kAbytes = kBM * 128; // one A stage (128 rows x 128 B)

constexpr uint32_t pow2_at_least(uint32_t v) {
  uint32_t p = 32;
  while (p < v) p <<= 1;
  return p;
}

template <int MODE, bool SWAP, int BN, int STAGES, int EPI_WARPS, int ACCB, bool PAIR,
          bool GROUPED = false, bool FUSEQ = false>
struct Cfg {
  static constexpr int kMmaM = PAIR ? 256 : 128;     // rows of the MMA (both CTAs)
  static constexpr int kBrows = PAIR ? BN / 2 : BN;  // weight rows loaded by this CTA
  // MX: the UE8M0 codes arrive pre-arranged (one chunk per row tile and K
  // block, written by the scale-factor tiling kernel) with each operand stage;
  // the MMA thread copies them into a TMEM slot (tcgen05.cp) ahead of its MMAs
  static constexpr int kSfSlots = 4;             // TMEM slots, used round-robin
  static constexpr int kSfColsB = (MODE == kModeMx) ? BN / 32 : 4;
  static constexpr int kSfSlotCols = 16;         // A at +0, B at +8
  static constexpr int kSfColsBPad = (kSfColsB + 3) / 4 * 4;
  // per stage: [A: 32 rows x 16 B][B: kSfColsBPad/4 blocks of 32 rows x 16 B];
  // word c of row i holds the four codes of tile row i + 32c
  static constexpr int kSfBBytes = 128 * kSfColsBPad;
  static constexpr int kSfStageBytes = (MODE == kModeMx) ? 512 + kSfBBytes : 0;
  // block tiles: two MMA-issuing warps take alternate K blocks (disjoint TMEM
  // partial buffers), so one issues while the other waits on its barriers.
  // The decode tiles with 16 or 32 tokens issue from four warps: their MMAs
  // are so short that one MMA instruction's issue latency, not its work, sets
  // the pace (measured 10.4 -> 9.1 us at 1 x 6144 x 6144; the 64-token tile
  // measured slower with four)
  // The per-tensor and channel decode tiles (full-K accumulation) issue from
  // four warps too (two for the 64-token tile), each into its own TMEM
  // accumulator over its K blocks; the epilogue adds them in a fixed order
  static constexpr int kIssuers = (MODE == kModeBlock) ? ((SWAP && BN <= 32) ? 4 : 2)
                                  : (SWAP && MODE != kModeMx) ? (BN <= 32 ? 4 : 2) : 1;
  static constexpr int kSubAcc = (MODE != kModeBlock) ? kIssuers : 1;  // accumulators per tile buffer
  // block pair and normal tiles keep the promoted FP32 accumulators in the
  // epilogue warps' registers: warpgroup 0 (producer, the two issuers and one
  // idle warp) hands registers to the epilogue warpgroups with setmaxnreg
  static constexpr bool kRegSplit = (MODE == kModeBlock) && !SWAP;
  static constexpr int kEpiBase = kRegSplit ? 4 : 1 + kIssuers;  // first epilogue warp
  // fused decode linear (FUSEQ): more warps quantise each stage's BF16
  // activation slice into the stage's E4M3 operand -- eight for the 16- and
  // 32-token tiles, so that groups of them take the stages in turn
  // (measured 11.3 -> 9.9 us at 1 x 6144 x 6144, 12.0 -> 11.3 us at 16
  // tokens); four for the 64-token tile, whose registers would spill with eight
  static constexpr bool kFuseQ = FUSEQ;
  static constexpr int kQWarps = FUSEQ ? (BN <= 32 ? 8 : 4) : 0;
  static constexpr int kQBase = kEpiBase + EPI_WARPS;          // first quantiser warp
  static constexpr int kThreads = 32 * (kEpiBase + EPI_WARPS + kQWarps);
  // register budget: warps are dealt round-robin to the SM's four schedulers,
  // each with a quarter of the register file, so the bound counts whole
  // groups of four warps
  static constexpr int kBoundThreads = (kThreads + 127) / 128 * 128;
  static constexpr int kLaunchRegs = (65536 / kBoundThreads) / 8 * 8 < 248 ? (65536 / kBoundThreads) / 8 * 8 : 248;
  // warpgroup 0 after the split (grouped launches: the producer and the
  // issuers also walk the expert table)
  static constexpr int kLowRegs = GROUPED ? 48 : 32;
  static constexpr int kHighRegsRaw =
      (kLaunchRegs * kBoundThreads - 128 * kLowRegs) / (kBoundThreads > 128 ? kBoundThreads - 128 : 1) / 8 * 8;
  static constexpr int kHighRegs = kHighRegsRaw < 248 ? kHighRegsRaw : 248;  // epilogue warpgroups
  static constexpr int kEpiThreads = 32 * EPI_WARPS;
  static constexpr int kColGroups = EPI_WARPS / 4;
  static constexpr int kCPT = BN / kColGroups;   // columns per epilogue thread
  // tcgen05.ld chunk width: 16 columns where a large FP32 accumulator lives in
  // registers without the register split, otherwise 32
  static constexpr int kCW = kRegSplit ? 32
                             : (MODE == kModeBlock && !SWAP && kCPT > 64) ? 16
                             : (kCPT % 32 == 0) ? 32 : 16;
  // columns loaded per tcgen05.wait::ld in the block-tile promotion
  static constexpr int kLD = kRegSplit ? (kCPT < 64 ? kCPT : 64) : kCW;
  // block pair and normal tiles write Y with TMA stores from a per-warp
  // staging area (32 rows x 64 BF16 columns per box, 128-byte swizzled)
  static constexpr bool kTmaStoreY = (MODE == kModeBlock) && !SWAP;
  static constexpr int kYBoxCols = 64;
  static constexpr int kYBoxBytes = 32 * kYBoxCols * 2;
  // one box per epilogue warp; a thread's columns beyond one box go out in
  // further rounds through the same box
  static constexpr int kYStageBytes = kTmaStoreY ? EPI_WARPS * kYBoxBytes : 0;
  // B slot of a stage: the E4M3 operand (kBrows x 128 B, 128-byte swizzled);
  // fused: followed by the BF16 activation slice it is quantised from
  // (kBrows x 128 values, 256 B per row, unswizzled)
  static constexpr int kXbytes = FUSEQ ? kBrows * 256 : 0;
  static constexpr int kBbytes = kBrows * 128 + kXbytes;
  static constexpr int kStageBytes = kAbytes + kBbytes;
  // bytes that land on a stage's full barrier
  // block pair and normal tiles: promotion factors come through a shared-memory
  // ring filled by the TMA producer, kScQuad K blocks per slot: s_x of this
  // CTA's 128 rows and s_w of the tile's (at most two) 128-row weight blocks
  static constexpr bool kScRing = (MODE == kModeBlock) && !SWAP;
  static constexpr int kScQuad = 4;
  static constexpr int kScSlots = kScRing ? 4 : 0;
  static constexpr int kScDiv = kScSlots > 0 ? kScSlots : 1;  // ring index divisor
  static constexpr int kScXBytes = kBM * kScQuad * 4;           // 2 KB
  static constexpr int kScWBytes = 2 * kScQuad * 4;             // 32 B
  static constexpr int kScSlotBytes = kScXBytes + 128;          // s_w at +kScXBytes
  static constexpr int kScBytes = kScSlots * kScSlotBytes;
  static constexpr int kAccCols = ACCB * BN * kSubAcc;  // accumulators / partials
  static constexpr int kSfBase = kAccCols;
  static constexpr uint32_t kTmemCols =
      pow2_at_least(kAccCols + (MODE == kModeMx ? kSfSlots * kSfSlotCols : 0));
  static constexpr int kBarBytes = 512;
  // dynamic shared memory: [align slack][A stages][B stages][barriers][sx stage]
  static constexpr size_t kFixedSmem = 1024 + size_t(STAGES) * (kStageBytes + kSfStageBytes) +
                                       kYStageBytes + kScBytes + kBarBytes;

  static_assert(EPI_WARPS % 4 == 0, "epilogue warps must cover the 4 TMEM lane quarters");
  static_assert(BN % 16 == 0 && BN >= 16 && BN <= 256, "UMMA N for M = 128");
  static_assert(kCPT % kCW == 0 && kCPT % 2 == 0, "chunking");
  static_assert(kTmemCols <= 512, "TMEM columns");
  static_assert(STAGES <= 8 && ACCB <= 8, "barrier arrays");
  static_assert(MODE != kModeMx || (!SWAP && BN % 32 == 0 && kSfColsB <= 8 && BN == kMxBN &&
                                    kSfBBytes == 512 * kMxSfBBlocks),
                "MX tiles match the scale-factor chunks");
  static_assert(!PAIR || (!SWAP && kBrows % 8 == 0), "pair tiles");
  static_assert(MODE != kModeBlock || SWAP || (128 % kCPT == 0 && BN % kCPT == 0),
                "block tiles: each thread's columns lie in one 128-row weight block");
  static_assert(!SWAP || (kCPT <= 64 && EPI_WARPS == 4),
                "swapped tiles keep all token columns of a weight row in one thread");
  static_assert(!FUSEQ || (SWAP && MODE == kModeBlock && !PAIR && !GROUPED &&
                           (kBrows * 128) % 1024 == 0 && kBbytes % 1024 == 0),
                "fused quantisation: decode block tiles, swizzle atoms aligned");
  static_assert(!kRegSplit || (kThreads % 128 == 0 && kHighRegs >= kLowRegs &&
                               128 * kLowRegs + (kThreads - 128) * kHighRegs <=
                                   kLaunchRegs * kThreads),
                "register split fits in the registers the block is launched with");
  static_assert(kCPT % kLD == 0 && kLD % kCW == 0, "promotion load groups");
  static_assert(!kTmaStoreY || (kCPT % kYBoxCols == 0 && kStageBytes % 1024 == 0),
                "TMA-stored Y boxes");
};

struct SmemBarriers {
  uint64_t full[8], empty[8];
  uint64_t tfull[8], tempty[8];
  uint64_t sc_full[4], sc_empty[4];
  uint64_t qfull[8];  // fused quantisation: a stage's E4M3 operand is written
  uint64_t drain;
  uint32_t tmem_base;
  uint32_t abort;
  uint32_t is_last;
};

__device__ __forceinline__ float bf16_bits_to_float(uint16_t b) {
  return __uint_as_float(static_cast<uint32_t>(b) << 16);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
  __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t *>(&h);
}

// (c0, c1) = (a0 * b0 + c0, a1 * b1 + c1): one paired FP32 FMA, each lane an
// IEEE round-to-nearest fused multiply-add.
__device__ __forceinline__ void ffma2(float &c0, float &c1, float a0, float a1, float b0,
                                      float b1) {
  asm("{\n\t.reg .b64 ra, rb, rc;\n\t"
      "mov.b64 ra, {%2, %3};\n\t"
      "mov.b64 rb, {%4, %5};\n\t"
      "mov.b64 rc, {%0, %1};\n\t"
      "fma.rn.f32x2 rc, ra, rb, rc;\n\t"
      "mov.b64 {%0, %1}, rc;\n\t}"
      : "+f"(c0), "+f"(c1)
      : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}

__device__ __forceinline__ void fmul2(float &a0, float &a1, float b0, float b1) {
  asm("{\n\t.reg .b64 ra, rb;\n\t"
      "mov.b64 ra, {%0, %1};\n\t"
      "mov.b64 rb, {%2, %3};\n\t"
      "mul.rn.f32x2 ra, ra, rb;\n\t"
      "mov.b64 {%0, %1}, ra;\n\t}"
      : "+f"(a0), "+f"(a1)
      : "f"(b0), "f"(b1));
}

__device__ __forceinline__ void record_timeout(const GemmArgs &a) {
  if (a.status) atomicExch(a.status, kStatusTimeout);
}

// Debug builds (FP8BQ_DEBUG_CHECKS defined): every global write of the
// epilogues is checked against the buffer it belongs to (Y rows and columns,
// the workspace's partial region); a write outside is skipped and recorded as
// FP8BQ_ERR_BOUNDS in the workspace status word.  Release builds compile the
// checks away.
#ifdef FP8BQ_DEBUG_CHECKS
constexpr bool kDebugChecks = true;
#else
constexpr bool kDebugChecks = false;
#endif
__device__ __forceinline__ bool write_ok(const GemmArgs &a, bool in_bounds) {
  if (!kDebugChecks || in_bounds) return true;
  if (a.status) atomicExch(a.status, kStatusBounds);
  return false;
}

// every lane waits; the warp proceeds only if all lanes saw the phase complete
__device__ __forceinline__ bool warp_wait(uint64_t *bar, uint32_t parity, volatile uint32_t *ab,
                                          uint64_t limit) {
  const bool ok = mbar_wait(bar, parity, ab, limit);
  return __all_sync(0xffffffffu, ok);
}

template <int CW>
__device__ __forceinline__ void tmem_ld_chunk(uint32_t taddr, uint32_t *r) {
  if (CW == 32) tmem_ld32(taddr, r);
  else tmem_ld16(taddr, r);
}

// Work unit -> (row0 of A, row0 of B, kb range, split, tile id for counters).
struct Unit {
  int a_row0;       // first A row of this CTA (tokens, or weight rows when swapped)
  int b_row0;       // first B row of the tile (the epilogue's first weight column)
  int b_load_row0;  // first B row this CTA loads (pair tiles: its half)
  int kb0, kb1, split, tile;
  int row_end;      // rows of A at or past this one are not the tile's (M, or the segment end)
  int expert;       // grouped form: the tile's expert (0 otherwise)
  int sw_row0;      // row of the tile's first 128-row weight block in s_w
};

// Grouped form: the m-tile table of one launch, built by every CTA in shared
// memory as three int arrays back to back: start [E+1], begin [E], end [E].
// Expert e owns m-tiles start[e] .. start[e+1]-1 and rows begin[e] .. end[e]-1.
// experts == 0 for plain GEMMs.
struct GroupTable {
  const int *start;
  int experts;
};

template <bool SWAP, bool PAIR, bool GROUPED>
__device__ __forceinline__ Unit decode_unit(int u, int num_a_tiles, int splits, int kps, int KB,
                                            int bn, uint32_t rank, int M, int N,
                                            const GroupTable &gt, const LaunchShape &sh) {
  Unit r;
  r.row_end = M;
  r.expert = 0;
  if (!SWAP && !GROUPED && sh.tail_splits > 1 && u >= sh.full_units) {
    // a K range of a split tail tile: `tile` numbers the split tiles (their
    // counters), `split` the range
    const int v = u - sh.full_units;
    const int ti = v / sh.tail_splits;
    const int t = sh.full_units + ti;
    const int mt = t % num_a_tiles, nt = t / num_a_tiles;
    constexpr int kTileRows = PAIR ? 2 * kBM : kBM;
    r.tile = ti;
    r.split = v - ti * sh.tail_splits;
    r.a_row0 = mt * kTileRows + static_cast<int>(rank) * kBM;
    r.b_row0 = nt * bn;
    r.b_load_row0 = r.b_row0 + (PAIR ? static_cast<int>(rank) * (bn / 2) : 0);
    r.sw_row0 = r.b_row0 / kBlockN;
    r.kb0 = r.split * sh.tail_kps;
    r.kb1 = min(KB, r.kb0 + sh.tail_kps);
    return r;
  }
  if (!SWAP) {
    // A = tokens (256 per pair tile, 128 per CTA), B = bn weight rows (pair
    // tiles: bn/2 per CTA).  Plain GEMMs walk M fastest, so concurrently
    // running tiles share the (large) weight tiles in L2.  Grouped GEMMs walk
    // the weight tiles fastest: a wave then covers all weight tiles of a few
    // m-tiles, so each m-tile's activation rows and the weight tiles of an
    // expert's consecutive m-tiles are shared by tiles running side by side,
    // rather than re-read from DRAM every wave as the weight stream evicts
    // them
    constexpr int kTileRows = PAIR ? 2 * kBM : kBM;
    const int n_tiles = (N + bn - 1) / bn;
    const int mt = GROUPED ? u / n_tiles : u % num_a_tiles;
    const int nt = GROUPED ? u - mt * n_tiles : u / num_a_tiles;
    r.tile = u;
    r.split = 0;
    int row0 = mt * kTileRows;
    if (GROUPED) {
      // the expert e with start[e] <= mt < start[e+1] (it has at least one tile)
      int lo = 0, hi = gt.experts;
      while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (gt.start[mid] <= mt) lo = mid;
        else hi = mid;
      }
      r.expert = lo;
      const int *begin = gt.start + gt.experts + 1;
      row0 = begin[lo] + (mt - gt.start[lo]) * kTileRows;
      r.row_end = begin[gt.experts + lo];
    }
    r.a_row0 = row0 + static_cast<int>(rank) * kBM;
    r.b_row0 = nt * bn;
    r.b_load_row0 = r.expert * N + r.b_row0 + (PAIR ? static_cast<int>(rank) * (bn / 2) : 0);
    r.sw_row0 = r.expert * ((N + kBlockN - 1) / kBlockN) + r.b_row0 / kBlockN;
    r.kb0 = 0;
    r.kb1 = KB;
    return r;
  }
  // swapped: A = weight rows (128 per tile), B = all tokens; units = tiles x splits
  r.tile = u / splits;
  r.split = u - r.tile * splits;
  r.a_row0 = r.tile * kBM;
  r.b_row0 = 0;
  r.b_load_row0 = 0;
  r.sw_row0 = 0;
  r.kb0 = r.split * kps;
  r.kb1 = min(KB, r.kb0 + kps);
  return r;
}

// Split-K partials of one split for one weight row: v[j] = the slot of token j
// (j < M, rows `stride` apart) once every one of them is non-zero, i.e. written
// (slots j >= M read as 1, the encoding of 0.0).  Polls with a short sleep;
// gives up, setting `abort`, after `limit_ns` or when another wait of the CTA
// has given up.
template <int CNT>
__device__ __forceinline__ bool poll_partials(const uint32_t *src, int64_t stride, int M,
                                              uint32_t (&v)[CNT], volatile uint32_t *abort,
                                              uint64_t limit_ns) {
  uint64_t t0 = 0;
  while (true) {
    bool all = true;
#pragma unroll
    for (int j = 0; j < CNT; ++j) {
      v[j] = j < M ? ld_relaxed_gpu(src + static_cast<int64_t>(j) * stride) : 1u;
      all = all && v[j] != 0u;
    }
    if (all) return true;
    if (*abort) return false;
    const uint64_t now = global_timer_ns();
    if (t0 == 0) {
      t0 = now;
    } else if (now - t0 > limit_ns) {
      *abort = 1u;
      return false;
    }
    __nanosleep(64);
  }
}

// Fused decode linear: quantiser warps that quantise one stage -- the token
// rows below M at eight threads each, rounded up to whole warps (at most
// QWARPS; a power of two, so the warps split into QWARPS / it groups).
template <int BN, int QWARPS>
__device__ __forceinline__ int fused_quant_warps_per_stage(int M) {
  const int need = (min(M, BN) * 8 + 31) / 32;
  int w = 1;
  while (w < need && w < QWARPS) w <<= 1;
  return w;
}

// The same with the slots in 16-byte groups of four tokens: group q of this
// thread's row at src + q * gstride (gstride = 4 N, so that a warp's 32 rows
// read 512 contiguous bytes per group): v[j] for j < M, 1 (the encoding of
// 0.0) beyond.
template <int CNT>
__device__ __forceinline__ bool poll_partials_quads(const uint32_t *src, int64_t gstride, int M,
                                                    uint32_t (&v)[CNT], volatile uint32_t *abort,
                                                    uint64_t limit_ns) {
  uint64_t t0 = 0;
  while (true) {
    bool all = true;
#pragma unroll
    for (int q = 0; q < CNT / 4; ++q) {
      const uint4 x = 4 * q < M ? ld_relaxed_gpu_v4(src + q * gstride) : make_uint4(1u, 1u, 1u, 1u);
      v[4 * q] = x.x;
      v[4 * q + 1] = 4 * q + 1 < M ? x.y : 1u;
      v[4 * q + 2] = 4 * q + 2 < M ? x.z : 1u;
      v[4 * q + 3] = 4 * q + 3 < M ? x.w : 1u;
      all = all && v[4 * q] != 0u && v[4 * q + 1] != 0u && v[4 * q + 2] != 0u && v[4 * q + 3] != 0u;
    }
    if (all) return true;
    if (*abort) return false;
    const uint64_t now = global_timer_ns();
    if (t0 == 0) {
      t0 = now;
    } else if (now - t0 > limit_ns) {
      *abort = 1u;
      return false;
    }
    __nanosleep(64);
  }
}

// Store `n` (multiple of 8 unless ragged) BF16 values of row m starting at column c0.
template <int CNT>
__device__ __forceinline__ void store_row(uint16_t *y, const float *v, int m, int c0,
                                          const GemmArgs &a) {
  uint16_t *yr = y + static_cast<int64_t>(m) * a.N;
  if ((a.N & 7) == 0) {
#pragma unroll
    for (int j = 0; j < CNT; j += 8) {
      if (c0 + j < a.N) {
        uint4 q;
        q.x = pack_bf16x2(v[j], v[j + 1]);
        q.y = pack_bf16x2(v[j + 2], v[j + 3]);
        q.z = pack_bf16x2(v[j + 4], v[j + 5]);
        q.w = pack_bf16x2(v[j + 6], v[j + 7]);
        *reinterpret_cast<uint4 *>(yr + c0 + j) = q;
      }
    }
  } else {
#pragma unroll
    for (int j = 0; j < CNT; ++j)
      if (c0 + j < a.N) {
        __nv_bfloat16 h = __float2bfloat16_rn(v[j]);
        yr[c0 + j] = *reinterpret_cast<uint16_t *>(&h);
      }
  }
}

// One CTA per SM.  Registers are split over the SM's four schedulers, so the
// per-thread budget is set by the scheduler holding the most warps.
template <int MODE, bool SWAP, int BN, int STAGES, int EPI_WARPS, int ACCB, bool PAIR, bool GROUPED,
          bool FUSEQ>
__global__ void __launch_bounds__(Cfg<MODE, SWAP, BN, STAGES, EPI_WARPS, ACCB, PAIR, GROUPED, FUSEQ>::kBoundThreads, 1)
    fp8_gemm_kernel(const __grid_constant__ CUtensorMap tmA,
                    const __grid_constant__ CUtensorMap tmB,
                    const __grid_constant__ CUtensorMap tmY,
                    const __grid_constant__ CUtensorMap tmSx,
                    const __grid_constant__ CUtensorMap tmSw,
                    const __grid_constant__ GemmArgs args, const LaunchShape shape) {
  using C = Cfg<MODE, SWAP, BN, STAGES, EPI_WARPS, ACCB, PAIR, GROUPED, FUSEQ>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t *smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
  uint8_t *sA = smem;
  uint8_t *sB = smem + STAGES * kAbytes;
  uint8_t *y_stage = smem + STAGES * C::kStageBytes;  // 1024-byte aligned
  uint8_t *sc_ring = y_stage + C::kYStageBytes;       // 1024-byte aligned
  uint8_t *sSF = sc_ring + C::kScBytes;               // MX: UE8M0 chunks per stage
  SmemBarriers *bars = reinterpret_cast<SmemBarriers *>(sSF + STAGES * C::kSfStageBytes);
  float *sx_stage = reinterpret_cast<float *>(reinterpret_cast<uint8_t *>(bars) + C::kBarBytes);
  volatile uint32_t *abort_flag = &bars->abort;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint64_t limit = args.wait_limit_ns;
  // pair tiles: rank in the CTA pair; work is distributed per cluster
  const uint32_t rank = PAIR ? cluster_ctarank() : 0u;
  const bool leader = rank == 0u;
  const int cl_id = PAIR ? static_cast<int>(blockIdx.x >> 1) : static_cast<int>(blockIdx.x);
  const int cl_num = PAIR ? static_cast<int>(gridDim.x >> 1) : static_cast<int>(gridDim.x);

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&bars->full[s], 1);
      mbar_init(&bars->empty[s], 1);
    }
    for (int b = 0; b < ACCB; ++b) {
      mbar_init(&bars->tfull[b], C::kSubAcc);  // one commit per accumulating issuer
      mbar_init(&bars->tempty[b], PAIR ? 2 * EPI_WARPS : EPI_WARPS);
    }
    for (int s = 0; s < C::kScSlots; ++s) {
      mbar_init(&bars->sc_full[s], 1);
      mbar_init(&bars->sc_empty[s], EPI_WARPS);
    }
    for (int s = 0; s < (C::kFuseQ ? STAGES : 0); ++s)
      mbar_init(&bars->qfull[s], fused_quant_warps_per_stage<BN, C::kQWarps>(args.M));
    mbar_init(&bars->drain, C::kIssuers);
    bars->abort = 0;
    bars->is_last = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    if ((C::kScRing && args.sc_tma) || MODE == kModeMx) {
      tma_prefetch_desc(&tmSx);
      tma_prefetch_desc(&tmSw);
    }
  }
  if (warp == 1) {
    if (PAIR) {
      tmem_alloc_pair(&bars->tmem_base, C::kTmemCols);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(&bars->tmem_base, C::kTmemCols);
      tmem_relinquish();
    }
  }
  tc_fence_before();
  __syncthreads();
  if (PAIR) cluster_sync();  // the peer's barriers are initialised before any use
  tc_fence_after();
  const uint32_t tmem_base = bars->tmem_base;

  // Programmatic dependent launch: the next kernel of the stream may be
  // scheduled now.  Until the preceding kernel has completed (griddepcontrol.wait)
  // this CTA touches no global memory except L2 prefetches of its first weight
  // tiles; L2 is the point of coherence, so a prefetch cannot make a later load
  // see stale data even if the preceding kernel writes those weights.
  griddep_launch_dependents();
  GroupTable gt{nullptr, 0};
  // (grouped launches learn their tiles only from the segment bounds, which the
  // preceding kernel may write: no prefetch)
  if (!GROUPED && warp == 0 && lane == 0 && cl_id < shape.units) {
    const Unit w0 = decode_unit<SWAP, PAIR, GROUPED>(cl_id, shape.num_a_tiles, shape.splits, shape.kps,
                                            shape.KB, BN, rank, args.M, args.N, gt, shape);
    const int npf = min(w0.kb1 - w0.kb0, SWAP ? 64 : 8);
    for (int i = 0; i < npf; ++i) {
      if (SWAP) tma_prefetch_l2_2d(&tmA, (w0.kb0 + i) * 128, w0.a_row0);
      else tma_prefetch_l2_2d(&tmB, (w0.kb0 + i) * 128, w0.b_load_row0);
    }
  }
  griddep_wait();

  int units = shape.units, num_a = shape.num_a_tiles;
  if (GROUPED) {
    // grouped form: every CTA turns the expert segments into its own copy of
    // the m-tile table (256-row pair tiles or 128-row tiles, a segment's last
    // tile ragged).  Bounds
    // are clamped into [0, M], so no copy or store leaves A or Y whatever the
    // offsets hold.
    const int E = args.g_experts;
    int *gs = reinterpret_cast<int *>(sx_stage);
    int *gb = gs + E + 1;
    int *ge = gb + E;
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
      int b, en;
      if (args.g_offsets) {
        b = args.g_offsets[e];
        en = args.g_offsets[e + 1];
      } else {
        b = e * args.g_max_m;
        en = b + min(max(args.g_masked[e], 0), args.g_max_m);
      }
      b = min(max(b, 0), args.M);
      en = min(max(en, b), args.M);
      gb[e] = b;
      ge[e] = en;
      const int len = en - b;
      constexpr int kTileRows = PAIR ? 2 * kBM : kBM;
      gs[e + 1] = len / kTileRows + (len % kTileRows != 0);
    }
    __syncthreads();
    if (warp == 0) {
      // inclusive scan of the tile counts, 32 experts per step
      int carry = 0;
      for (int base = 0; base < E; base += 32) {
        const int e = base + lane;
        int v = e < E ? gs[e + 1] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int t = __shfl_up_sync(0xffffffffu, v, o);
          if (lane >= o) v += t;
        }
        if (e < E) gs[e + 1] = v + carry;
        carry += __shfl_sync(0xffffffffu, v, 31);
      }
      if (lane == 0) gs[0] = 0;
    }
    __syncthreads();
    gt = GroupTable{gs, E};
    // never more tiles than the host sized the grid and the table for
    num_a = min(gs[E], args.g_tile_cap);
    units = num_a * ((args.N + BN - 1) / BN);
  }

  if (C::kRegSplit) {
    if (warp < 4) setmaxnreg_dec<C::kLowRegs>();
    else setmaxnreg_inc<C::kHighRegs>();
  }

  const int KB = shape.KB;

  if (warp < C::kEpiBase) {
    // producer, MMA issuers, MX scale-factor writers
    if (warp == 0) {
      // ------------------------------------------------------------ TMA producer
      if (lane == 0) {
        uint32_t issued = 0, phase_bits = 0;  // per stage: ever issued, last phase
        uint32_t sc_issued = 0, sc_phase_bits = 0;
        uint32_t it = 0, sq = 0;
        bool ok = true;
        const bool sc_tma = C::kScRing && args.sc_tma;
        for (int u = cl_id; ok && u < units; u += cl_num) {
          const Unit w = decode_unit<SWAP, PAIR, GROUPED>(u, num_a, shape.splits, shape.kps, KB, BN, rank, args.M, args.N, gt, shape);
          for (int kb = w.kb0; kb < w.kb1; ++kb, ++it) {
            if (sc_tma && (kb - w.kb0) % C::kScQuad == 0) {
              // promotion factors of K blocks kb .. kb+3: this CTA's s_x rows and
              // the tile's weight-block scales, on this CTA's own barrier
              const uint32_t q = sq % C::kScDiv, qph = (sq / C::kScDiv) & 1u;
              if (!mbar_wait(&bars->sc_empty[q], qph ^ 1u, abort_flag, limit)) {
                ok = false;
                break;
              }
              uint8_t *slot = sc_ring + q * C::kScSlotBytes;
              mbar_arrive_expect_tx(&bars->sc_full[q], C::kScXBytes + C::kScWBytes);
              if (args.sx_layout == 0) tma_load_2d(slot, &tmSx, &bars->sc_full[q], kb, w.a_row0);
              else tma_load_2d(slot, &tmSx, &bars->sc_full[q], w.a_row0, kb);
              tma_load_2d(slot + C::kScXBytes, &tmSw, &bars->sc_full[q], kb, w.sw_row0);
              sc_issued |= 1u << q;
              sc_phase_bits = (sc_phase_bits & ~(1u << q)) | (qph << q);
              ++sq;
            }
            const uint32_t s = it % STAGES, ph = (it / STAGES) & 1u;
            if (!mbar_wait(&bars->empty[s], ph ^ 1u, abort_flag, limit)) {
              ok = false;
              break;
            }
            if (args.fault_skip_first_load && blockIdx.x == 0 && it == 0) continue;
            // MX: this CTA's A-row chunk and the weight tile's chunk of UE8M0
            // codes (256-byte rows: 2 for A, kSfBBytes / 256 for B)
            const int sfa_row = ((w.a_row0 / kBM) * KB + kb) * 2;
            const int sfb_row = ((w.b_row0 / BN) * KB + kb) * (C::kSfBBytes / 256);
            uint8_t *sf = sSF + s * C::kSfStageBytes;
            if (PAIR) {
              // both CTAs' bytes complete on the even CTA's barrier
              if (leader)
                mbar_arrive_expect_tx(&bars->full[s], 2 * (C::kStageBytes + C::kSfStageBytes));
              const uint32_t bar0 = mapa_shared(smem_u32(&bars->full[s]), 0);
              tma_load_2d_pair(sA + s * kAbytes, &tmA, bar0, kb * 128, w.a_row0);
              tma_load_2d_pair(sB + s * C::kBbytes, &tmB, bar0, kb * 128, w.b_load_row0);
              if (MODE == kModeMx) {
                tma_load_2d_pair(sf, &tmSx, bar0, 0, sfa_row);
                tma_load_2d_pair(sf + 512, &tmSw, bar0, 0, sfb_row);
              }
            } else if (C::kFuseQ) {
              // the weight tile and the BF16 activations of K block kb (all
              // tokens; rows >= M and columns >= K read as zero)
              mbar_arrive_expect_tx(&bars->full[s], kAbytes + args.b_box_rows * 256);
              tma_load_2d(sA + s * kAbytes, &tmA, &bars->full[s], kb * 128, w.a_row0);
              tma_load_2d(sB + s * C::kBbytes + C::kBrows * 128, &tmB, &bars->full[s], kb * 128, 0);
            } else {
              // decode tiles copy only the token rows in use (b_box_rows): the
              // other rows of the operand only feed output columns past M
              mbar_arrive_expect_tx(&bars->full[s],
                                    (SWAP ? kAbytes + args.b_box_rows * 128 : C::kStageBytes) +
                                        C::kSfStageBytes);
              tma_load_2d(sA + s * kAbytes, &tmA, &bars->full[s], kb * 128, w.a_row0);
              tma_load_2d(sB + s * C::kBbytes, &tmB, &bars->full[s], kb * 128, w.b_load_row0);
              if (MODE == kModeMx) {
                tma_load_2d(sf, &tmSx, &bars->full[s], 0, sfa_row);
                tma_load_2d(sf + 512, &tmSw, &bars->full[s], 0, sfb_row);
              }
            }
            issued |= 1u << s;
            phase_bits = (phase_bits & ~(1u << s)) | (ph << s);
          }
        }
        if (!ok) {
          record_timeout(args);
          // let every copy issued land before shared memory goes away (pair tiles:
          // the even CTA's barriers count both CTAs' copies; the odd CTA stays
          // resident until the closing cluster barrier)
          for (int s = 0; s < STAGES && (!PAIR || leader); ++s)
            if ((issued >> s) & 1u) {
              uint32_t dummy = 0;
              mbar_wait(&bars->full[s], (phase_bits >> s) & 1u, &dummy, limit);
            }
          for (int q = 0; q < C::kScSlots; ++q)
            if ((sc_issued >> q) & 1u) {
              uint32_t dummy = 0;
              mbar_wait(&bars->sc_full[q], (sc_phase_bits >> q) & 1u, &dummy, limit);
            }
        }
      }
      __syncwarp();
    } else if (warp <= C::kIssuers) {
      // ------------------------------------------------------------ MMA issuers
      // Issuer `me` takes the K blocks with it % kIssuers == me (block tiles; every
      // K block has its own TMEM partial buffer) -- with one issuer, all of them.
      const uint32_t me = static_cast<uint32_t>(warp - 1);
      if (lane == 0 && (!PAIR || leader)) {
        uint32_t it = 0, uit = 0;
        bool ok = true;
        for (int u = cl_id; ok && u < units; u += cl_num, ++uit) {
          const Unit w = decode_unit<SWAP, PAIR, GROUPED>(u, num_a, shape.splits, shape.kps, KB, BN, rank, args.M, args.N, gt, shape);
          const uint32_t it0 = it;  // this unit's first K block
          if (MODE != kModeBlock) {
            const uint32_t b = uit % ACCB, ph = (uit / ACCB) & 1u;
            if (!mbar_wait(&bars->tempty[b], ph ^ 1u, abort_flag, limit)) {
              ok = false;
              break;
            }
            tc_fence_after();
          }
          for (int kb = w.kb0; kb < w.kb1; ++kb, ++it) {
            if (C::kIssuers > 1 && it % C::kIssuers != me) continue;
            uint32_t d_tmem;
            if (MODE == kModeBlock) {
              const uint32_t b = it % ACCB, ph = (it / ACCB) & 1u;
              if (!mbar_wait(&bars->tempty[b], ph ^ 1u, abort_flag, limit)) {
                ok = false;
                break;
              }
              d_tmem = tmem_base + b * BN;
            } else {
              d_tmem = tmem_base + ((uit % ACCB) * C::kSubAcc + (C::kSubAcc > 1 ? me : 0u)) * BN;
            }
            const uint32_t s = it % STAGES, ph = (it / STAGES) & 1u;
            // fused: the quantiser warps have seen the stage land and written its operand
            if (!mbar_wait(C::kFuseQ ? &bars->qfull[s] : &bars->full[s], ph, abort_flag, limit)) {
              ok = false;
              break;
            }
            const uint32_t sfslot = it % C::kSfSlots;
            tc_fence_after();
            if (MODE == kModeMx) {
              // UE8M0 codes of this K block: shared memory -> TMEM slot, ahead of the
              // MMAs that read them (same issuing thread, executed in order)
              const uint32_t sfcol = tmem_base + C::kSfBase + sfslot * C::kSfSlotCols;
              const uint32_t src = smem_u32(sSF + s * C::kSfStageBytes);
  #pragma unroll
              for (int j = 0; j <= C::kSfColsBPad / 4; ++j) {
                // j = 0: A codes to columns +0..3; j >= 1: B codes to +8.., +12..
                const uint32_t col = sfcol + (j == 0 ? 0 : 4 + 4 * j);
                const uint64_t d = sdesc_kmajor_noswizzle(src + 512 * j, 128, 128);
                if (PAIR) tmem_cp_32x128b_warpx4_pair(col, d);
                else tmem_cp_32x128b_warpx4(col, d);
              }
            }
            const uint64_t adesc = sdesc_kmajor_sw128(smem_u32(sA + s * kAbytes));
            const uint64_t bdesc = sdesc_kmajor_sw128(smem_u32(sB + s * C::kBbytes));
  #pragma unroll
            for (int k = 0; k < 4; ++k) {
              // advance 32 K-bytes inside the 128-byte swizzled row: +2 in the >>4 field
              // block tiles: one K block per partial; full-K tiles: accumulate
              // after this accumulator's first K block of the unit
              const uint32_t acc = (MODE == kModeBlock) ? (k > 0)
                                   : ((it - it0) >= static_cast<uint32_t>(C::kSubAcc) || k > 0);
              if (MODE == kModeMx) {
                const uint32_t sfcol = tmem_base + C::kSfBase + sfslot * C::kSfSlotCols;
                if (PAIR)
                  umma_mxf8f6f4_pair(d_tmem, adesc + 2 * k, bdesc + 2 * k,
                                     idesc_mxf8_e4m3(C::kMmaM, BN, k, k), sfcol, sfcol + 8, acc);
                else
                  umma_mxf8f6f4(d_tmem, adesc + 2 * k, bdesc + 2 * k,
                                idesc_mxf8_e4m3(kBM, BN, k, k), sfcol, sfcol + 8, acc);
              } else if (PAIR) {
                umma_f8f6f4_pair(d_tmem, adesc + 2 * k, bdesc + 2 * k,
                                 idesc_f8f6f4_e4m3(C::kMmaM, BN), acc);
              } else {
                umma_f8f6f4(d_tmem, adesc + 2 * k, bdesc + 2 * k, idesc_f8f6f4_e4m3(kBM, BN), acc);
              }
            }
            if (PAIR) umma_commit_pair(&bars->empty[s], 0x3);
            else umma_commit(&bars->empty[s]);
            if (MODE == kModeBlock) {
              if (PAIR) umma_commit_pair(&bars->tfull[it % ACCB], 0x3);
              else umma_commit(&bars->tfull[it % ACCB]);
            }
          }
          if (!ok) break;
          if (MODE != kModeBlock) {
            if (PAIR) umma_commit_pair(&bars->tfull[uit % ACCB], 0x3);
            else umma_commit(&bars->tfull[uit % ACCB]);
          }
        }
        if (!ok) record_timeout(args);
        // every MMA issued by both issuers has completed once `drain` flips
        if (PAIR) umma_commit_pair(&bars->drain, 0x1);
        else umma_commit(&bars->drain);
        uint32_t dummy = 0;
        mbar_wait(&bars->drain, 0, &dummy, limit);
      }
      __syncwarp();
    }
  } else if (warp < C::kQBase) {
    // ------------------------------------------------------------ epilogue
    const int ew = warp - C::kEpiBase;
    const int quarter = warp & 3;
    // tell the MMA issuer (the even CTA for pair tiles) that accumulator b is drained
    auto release_acc = [&](uint32_t b) {
      if (PAIR && !leader) mbar_arrive_cluster(mapa_shared(smem_u32(&bars->tempty[b]), 0));
      else mbar_arrive(&bars->tempty[b]);
    };
    const int cg = ew >> 2;  // column group
    const int et = ew * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>(32 * quarter) << 16;
    const int NBLK = (args.N + kBlockN - 1) / kBlockN;
    uint16_t *y = static_cast<uint16_t *>(args.y);
    const uint16_t *bias = static_cast<const uint16_t *>(args.bias);
    uint32_t kit = 0, uit = 0, sq = 0;
    bool ok = true;
    for (int u = cl_id; u < units; u += cl_num, ++uit) {
      const Unit w = decode_unit<SWAP, PAIR, GROUPED>(u, num_a, shape.splits, shape.kps, KB, BN, rank, args.M, args.N, gt, shape);
      const int d_row = w.a_row0 + 32 * quarter + lane;  // row of D held by this thread
      const int col0 = cg * C::kCPT;                     // first D column of this thread

      if (!SWAP) {
        // ---------------- normal orientation: thread = one token row, kCPT weight columns
        const int m = d_row;
        const int nbase = w.b_row0 + col0;
        if (MODE == kModeBlock) {
          float acc[C::kCPT];
#pragma unroll
          for (int j = 0; j < C::kCPT; ++j) acc[j] = 0.0f;
          const bool row_ok = m < w.row_end;
          // one K block: wait for its partial, read it from TMEM, hand the
          // buffer back to the MMA issuer, promote it with factor f
          auto promote = [&](float f) -> bool {
            const uint32_t b = kit % ACCB, ph = (kit / ACCB) & 1u;
            if (!warp_wait(&bars->tfull[b], ph, abort_flag, limit)) return false;
            tc_fence_after();
            const uint32_t tbase = tmem_base + lane_base + b * BN + col0;
            // kLD columns per wait: with the register split, a thread's whole
            // share of the partial is in flight in one or two rounds
#pragma unroll
            for (int g = 0; g < C::kCPT / C::kLD; ++g) {
              uint32_t r[C::kLD];
#pragma unroll
              for (int c = 0; c < C::kLD / C::kCW; ++c)
                tmem_ld_chunk<C::kCW>(tbase + g * C::kLD + c * C::kCW, r + c * C::kCW);
              tmem_ld_wait();
              if (g == C::kCPT / C::kLD - 1) {
                tc_fence_before();
                __syncwarp();
                if (lane == 0) release_acc(b);
              }
#pragma unroll
              for (int j = 0; j < C::kLD; j += 2)
                ffma2(acc[g * C::kLD + j], acc[g * C::kLD + j + 1], __uint_as_float(r[j]),
                      __uint_as_float(r[j + 1]), f, f);
            }
            ++kit;
            return true;
          };
          // every column of this thread lies in one 128-row weight block (kCPT
          // divides 128 and tiles start on multiples of kCPT), so the promotion
          // factor of a K block is s_x[m][kb] * s_w[nb][kb]
          if (C::kScRing && args.sc_tma) {
            // factors from the shared-memory ring, four K blocks per slot:
            // s_x row-major box [128 rows][4] or column-major box [4][128 rows],
            // s_w box [2 weight blocks][4]
            const int row = 32 * quarter + lane;
            const int nbi = nbase / kBlockN - w.b_row0 / kBlockN;  // 0 or 1
            for (int kq = w.kb0; kq < w.kb1 && ok; kq += C::kScQuad) {
              const uint32_t q = sq % C::kScDiv, qph = (sq / C::kScDiv) & 1u;
              if (!warp_wait(&bars->sc_full[q], qph, abort_flag, limit)) {
                ok = false;
                break;
              }
              const uint8_t *slot = sc_ring + q * C::kScSlotBytes;
              float4 xv;
              if (args.sx_layout == 0) {
                xv = *reinterpret_cast<const float4 *>(slot + row * 16);
              } else {
                const float *xs = reinterpret_cast<const float *>(slot);
                xv = make_float4(xs[row], xs[kBM + row], xs[2 * kBM + row], xs[3 * kBM + row]);
              }
              const float4 wv = *reinterpret_cast<const float4 *>(slot + C::kScXBytes + nbi * 16);
              __syncwarp();
              if (lane == 0) mbar_arrive(&bars->sc_empty[q]);
              ++sq;
              const float fq[4] = {xv.x * wv.x, xv.y * wv.y, xv.z * wv.z, xv.w * wv.w};
#pragma unroll
              for (int u = 0; u < C::kScQuad; ++u) {
                if (kq + u >= w.kb1) break;
                if (!promote(fq[u])) {
                  ok = false;
                  break;
                }
              }
            }
          } else {
            // factors loaded by each thread two K blocks ahead
            const int nb = min(nbase / kBlockN, NBLK - 1);
            const float *swrow = args.sw + (static_cast<int64_t>(w.expert) * NBLK + nb) * KB;
            auto sx_at = [&](int kb) -> float {
              if (!row_ok || kb >= w.kb1) return 0.0f;
              return __ldg(args.sx + (args.sx_layout == 0
                                          ? static_cast<int64_t>(m) * args.ldsx + kb
                                          : static_cast<int64_t>(kb) * args.ldsx + m));
            };
            auto sw_at = [&](int kb) -> float { return kb < w.kb1 ? __ldg(swrow + kb) : 0.0f; };
            float sx_cur = sx_at(w.kb0), sw_cur = sw_at(w.kb0);
            float sx_nxt = sx_at(w.kb0 + 1), sw_nxt = sw_at(w.kb0 + 1);
            for (int kb = w.kb0; kb < w.kb1 && ok; ++kb) {
              const float f = sx_cur * sw_cur;
              sx_cur = sx_nxt;
              sw_cur = sw_nxt;
              sx_nxt = sx_at(kb + 2);
              sw_nxt = sw_at(kb + 2);
              if (!promote(f)) ok = false;
            }
          }
          // all epilogue warps agree on the outcome before anything is stored
          if (named_bar_any(2, C::kEpiThreads, !ok || *abort_flag)) {
            ok = false;
            break;
          }
          if (!GROUPED && shape.tail_splits > 1 && u >= shape.full_units) {
            // a split tail tile: publish this range's promoted accumulators
            // (column-major 256 x 128 per CTA, so a warp's stores are 128
            // contiguous bytes); the last split to arrive sums all ranges in
            // split order (its own from registers) and stores Y.  The barrier
            // orders the stores before the counter's release; the last CTA's
            // acquire on the same counter makes every split's partial visible.
            const int row = 32 * quarter + lane;
            const int64_t blk = 128 * 256;
            float *mine = args.partials + (static_cast<int64_t>(w.tile) * shape.tail_splits + w.split) * 2 * blk +
                          rank * blk;
#pragma unroll
            for (int j = 0; j < C::kCPT; ++j)
              if (write_ok(args, (mine - args.partials) + (col0 + j) * 128 + row <
                                     args.partials_bytes / 4))
                __stcg(mine + (col0 + j) * 128 + row, acc[j]);
            named_bar_sync(2, C::kEpiThreads);
            if (et == 0) {
              const uint32_t prev = atom_add_acq_rel_gpu(args.counters + 2 * w.tile + rank, 1u);
              bars->is_last = (prev == static_cast<uint32_t>(shape.tail_splits - 1)) ? 1u : 0u;
            }
            named_bar_sync(2, C::kEpiThreads);
            if (!bars->is_last) continue;
            const float *base = args.partials + static_cast<int64_t>(w.tile) * shape.tail_splits * 2 * blk +
                                rank * blk + col0 * 128 + row;
#pragma unroll
            for (int c = 0; c < C::kCPT / 32; ++c) {
              float sum[32];
#pragma unroll
              for (int j = 0; j < 32; ++j) sum[j] = 0.0f;
              for (int sp = 0; sp < shape.tail_splits; ++sp) {
                if (sp == w.split) {
#pragma unroll
                  for (int j = 0; j < 32; ++j) sum[j] += acc[c * 32 + j];
                } else {
                  const float *src = base + static_cast<int64_t>(sp) * 2 * blk + (c * 32) * 128;
                  float v[32];
#pragma unroll
                  for (int j = 0; j < 32; ++j) v[j] = __ldcg(src + j * 128);
#pragma unroll
                  for (int j = 0; j < 32; ++j) sum[j] += v[j];
                }
              }
#pragma unroll
              for (int j = 0; j < 32; ++j) acc[c * 32 + j] = sum[j];
            }
            if (et == 0) args.counters[2 * w.tile + rank] = 0u;  // ready for the next call
          }
          if (bias) {
#pragma unroll
            for (int j = 0; j < C::kCPT; ++j)
              if (nbase + j < args.N) acc[j] += bf16_bits_to_float(bias[nbase + j]);
          }
          // a TMA box writes all of its 32 rows that lie inside Y: only where
          // they all belong to the tile (the grouped form's segments end
          // anywhere) does the warp use one
          const int row0 = w.a_row0 + 32 * quarter;
          if (C::kTmaStoreY && args.y_tma && (row0 + 32 <= w.row_end || w.row_end == args.M)) {
            // BF16 rows into this warp's staging box (16-byte chunk c of row r
            // at chunk position c ^ (r % 8): the 128-byte swizzle the tensor map
            // names, and conflict-free), then one TMA store per 64 columns.
            // Before each refill the previous store must have finished reading.
            uint8_t *stg = y_stage + ew * C::kYBoxBytes;
#pragma unroll
            for (int bx = 0; bx < C::kCPT / C::kYBoxCols; ++bx) {
              if (lane == 0) bulk_wait_group_read0();
              __syncwarp();
              uint8_t *rowp = stg + lane * 128;
#pragma unroll
              for (int c = 0; c < 8; ++c) {
                const float *v = acc + bx * C::kYBoxCols + c * 8;
                uint4 q;
                q.x = pack_bf16x2(v[0], v[1]);
                q.y = pack_bf16x2(v[2], v[3]);
                q.z = pack_bf16x2(v[4], v[5]);
                q.w = pack_bf16x2(v[6], v[7]);
                *reinterpret_cast<uint4 *>(rowp + ((c ^ (lane & 7)) << 4)) = q;
              }
              fence_proxy_async_smem();
              __syncwarp();
              if (lane == 0 && row0 < w.row_end && nbase + bx * C::kYBoxCols < args.N &&
                  write_ok(args, row0 >= 0 && w.row_end <= args.M)) {
                tma_store_2d(&tmY, stg, nbase + bx * C::kYBoxCols, row0);
                bulk_commit_group();
              }
            }
          } else if (m < w.row_end && write_ok(args, m >= 0 && m < args.M)) {
            store_row<C::kCPT>(y, acc, m, nbase, args);
          }
        } else {
          // kModeTensor / kModeChannel / kModeMx: one pass over the full-K accumulator
          const uint32_t b = uit % ACCB, ph = (uit / ACCB) & 1u;
          if (!warp_wait(&bars->tfull[b], ph, abort_flag, limit)) ok = false;
          if (named_bar_any(2, C::kEpiThreads, !ok || *abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t tbase = tmem_base + lane_base + b * BN + col0;
          // the activation factor: the per-tensor scale, or this row's token scale
          const float sxs = (MODE == kModeTensor) ? __ldg(args.sx_scalar)
                            : (MODE == kModeChannel) ? (m < w.row_end ? __ldg(args.sx + m) : 0.0f)
                                                     : 1.0f;
#pragma unroll
          for (int c = 0; c < C::kCPT / C::kCW; ++c) {
            uint32_t r[C::kCW];
            tmem_ld_chunk<C::kCW>(tbase + c * C::kCW, r);
            tmem_ld_wait();
            if (c == C::kCPT / C::kCW - 1) {
              tc_fence_before();
              __syncwarp();
              if (lane == 0) release_acc(b);
            }
            float v[C::kCW];
            // per-tensor scales: one output partition covers the whole chunk
            // unless the chunk straddles a partition boundary (then per column)
            const int n0c = nbase + c * C::kCW;
            float fchunk = 1.0f;
            bool uniform = true;
            if (MODE == kModeTensor) {
              int p = 0;
              while (p < args.n_parts - 1 && n0c >= args.part_end[p]) ++p;
              uniform = (p == args.n_parts - 1) || (n0c + C::kCW <= args.part_end[p]);
              fchunk = sxs * __ldg(args.sw_part + p);
            }
#pragma unroll
            for (int j = 0; j < C::kCW; ++j) {
              v[j] = __uint_as_float(r[j]);
              const int n = n0c + j;
              if (MODE == kModeTensor) {
                if (uniform) {
                  v[j] *= fchunk;
                } else {
                  int p = 0;
                  while (p < args.n_parts - 1 && n >= args.part_end[p]) ++p;
                  v[j] *= sxs * __ldg(args.sw_part + p);
                }
              } else if (MODE == kModeChannel) {
                v[j] = (v[j] * sxs) * (n < args.N ? __ldg(args.sw + n) : 0.0f);
              }
              if (bias && n < args.N) v[j] += bf16_bits_to_float(bias[n]);
            }
            if (m < w.row_end && write_ok(args, m >= 0 && m < args.M))
              store_row<C::kCW>(y, v, m, nbase + c * C::kCW, args);
          }
        }
      } else {
        // ---------------- swapped orientation: thread = one weight row, all tokens
        float acc[C::kCPT];
#pragma unroll
        for (int j = 0; j < C::kCPT; ++j) acc[j] = 0.0f;
        if (MODE == kModeBlock) {
          // stage s_x[token][kb] for this unit's K range: sx_stage[(kb-kb0)*BN + token]
          // (fused: the quantiser warps write it as they quantise each K block)
          const int nkb = C::kFuseQ ? 0 : w.kb1 - w.kb0;
          for (int e = et; e < nkb * BN; e += C::kEpiThreads) {
            const int kb = w.kb0 + e / BN, t = e % BN;
            float v = 0.0f;
            if (t < args.M)
              v = __ldg(args.sx + (args.sx_layout == 0
                                       ? static_cast<int64_t>(t) * args.ldsx + kb
                                       : static_cast<int64_t>(kb) * args.ldsx + t));
            sx_stage[e] = v;
          }
          named_bar_sync(1, C::kEpiThreads);
          // lanes are weight rows of one 128-row block: one s_w per K block,
          // fetched one K block ahead
          const float *swrow = args.sw + static_cast<int64_t>(w.a_row0 / kBlockN) * KB;
          float sw_next = __ldg(swrow + w.kb0);
          for (int kb = w.kb0; kb < w.kb1 && ok; ++kb, ++kit) {
            const uint32_t b = kit % ACCB, ph = (kit / ACCB) & 1u;
            const float swv = sw_next;
            if (!warp_wait(&bars->tfull[b], ph, abort_flag, limit)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t tbase = tmem_base + lane_base + b * BN;
            uint32_t r[C::kCPT];
#pragma unroll
            for (int c = 0; c < C::kCPT / C::kCW; ++c)
              tmem_ld_chunk<C::kCW>(tbase + c * C::kCW, r + c * C::kCW);
            tmem_ld_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) release_acc(b);
            if (kb + 1 < w.kb1) sw_next = __ldg(swrow + kb + 1);  // after the release
            const float *sxk = sx_stage + (kb - w.kb0) * BN;
#pragma unroll
            for (int j = 0; j < C::kCPT; j += 2) {
              float f0 = sxk[j], f1 = sxk[j + 1];
              fmul2(f0, f1, swv, swv);
              ffma2(acc[j], acc[j + 1], __uint_as_float(r[j]), __uint_as_float(r[j + 1]), f0,
                    f1);
            }
          }
        } else if (ok) {
          const uint32_t b = uit % ACCB, ph = (uit / ACCB) & 1u;
          if (!warp_wait(&bars->tfull[b], ph, abort_flag, limit)) {
            ok = false;
          } else {
            tc_fence_after();
            // the issuers' accumulators that received K blocks, added in order
            const int nsub = min(C::kSubAcc, w.kb1 - w.kb0);
            uint32_t r[C::kCPT];
            for (int i = 0; i < nsub; ++i) {
              const uint32_t tbase = tmem_base + lane_base + (b * C::kSubAcc + i) * BN;
              uint32_t t[C::kCPT];
#pragma unroll
              for (int c = 0; c < C::kCPT / C::kCW; ++c)
                tmem_ld_chunk<C::kCW>(tbase + c * C::kCW, t + c * C::kCW);
              tmem_ld_wait();
#pragma unroll
              for (int j = 0; j < C::kCPT; ++j)
                r[j] = i == 0 ? t[j] : __float_as_uint(__uint_as_float(r[j]) + __uint_as_float(t[j]));
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) release_acc(b);
            if (MODE == kModeChannel) {
              // lane = one output channel; columns = tokens, each with its scale
              const float fw = d_row < args.N ? __ldg(args.sw + d_row) : 0.0f;
#pragma unroll
              for (int j = 0; j < C::kCPT; ++j)
                acc[j] = (__uint_as_float(r[j]) * (j < args.M ? __ldg(args.sx + j) : 0.0f)) * fw;
            } else {
              // one output partition per lane (weight row)
              int p = 0;
              while (p < args.n_parts - 1 && d_row >= args.part_end[p]) ++p;
              const float f = __ldg(args.sx_scalar) * __ldg(args.sw_part + p);
#pragma unroll
              for (int j = 0; j < C::kCPT; ++j) acc[j] = __uint_as_float(r[j]) * f;
            }
          }
        }

        if (named_bar_any(2, C::kEpiThreads, !ok || *abort_flag)) {
          ok = false;
          break;
        }
        const int n = d_row;
        const bool n_ok = n < args.N;
        const float bv = (bias && n_ok) ? bf16_bits_to_float(bias[n]) : 0.0f;
        if (shape.splits == 1) {
          if (n_ok) {
#pragma unroll
            for (int j = 0; j < C::kCPT; ++j)
              if (j < args.M) {
                __nv_bfloat16 h = __float2bfloat16_rn(acc[j] + bv);
                y[static_cast<int64_t>(j) * args.N + n] = *reinterpret_cast<uint16_t *>(&h);
              }
          }
        } else {
          // split-K: the K range of weight tile w.tile is split over
          // shape.splits CTAs.  Splits 1.. publish their FP32 partials and
          // leave; split 0 sums them into its own in ascending split order and
          // writes Y.  A partial travels as its bits + 1 in a relaxed GPU-scope
          // store, so a slot holding 0 has not been written yet (FP32
          // arithmetic never yields the bits 0xFFFFFFFF, the one value that
          // would wrap to 0): split 0 polls the elements themselves -- no
          // counter, no fence, no election on the path -- and writes 0 back to
          // every slot it consumed, which leaves the workspace ready for the
          // next call.  The polling ends because every CTA of the grid is
          // resident at once (one CTA per SM, tiles x splits <= SMs, and no
          // CTA waits on anything that a later kernel produces); it is bounded
          // all the same.
          uint32_t *part = reinterpret_cast<uint32_t *>(args.partials);
          // The 16- and 64-token tiles keep the slots in 16-byte groups of four
          // tokens (group q of split sp, row n at ((sp Q + q) N + n) 4, Q = M/4
          // rounded up): a quarter of the accesses, still 512 contiguous bytes
          // per warp and group (measured at 6144 x 6144: M = 64 15.7 -> 14.1
          // us, M = 1 9.1 -> 9.0).  The 32-token tile keeps one token per
          // slot, token-major, a warp's 32 rows contiguous (the groups measured
          // 12.1 against 11.5 us there).
          constexpr bool kQuadSlots = C::kCPT == 16 || C::kCPT == 64;
          const int Q = (args.M + 3) >> 2;
          const int64_t gstride = static_cast<int64_t>(args.N) * 4;
          if (kQuadSlots && w.split != 0) {
            if (n_ok) {
              uint32_t *dst = part + (static_cast<int64_t>(w.split) * Q * args.N + n) * 4;
#pragma unroll
              for (int q = 0; q < C::kCPT / 4; ++q)
                if (4 * q < args.M &&
                    write_ok(args, (dst - part) + q * gstride + 3 < args.partials_bytes / 4)) {
                  auto enc = [&](int j) { return j < args.M ? __float_as_uint(acc[j]) + 1u : 1u; };
                  st_relaxed_gpu_v4(dst + q * gstride,
                                    make_uint4(enc(4 * q), enc(4 * q + 1), enc(4 * q + 2), enc(4 * q + 3)));
                }
            }
          } else if (kQuadSlots && n_ok) {
            float sum[C::kCPT];
#pragma unroll
            for (int j = 0; j < C::kCPT; ++j) sum[j] = acc[j];
            bool got = true;
            for (int sp = 1; sp < shape.splits && got; ++sp) {
              const uint32_t *src = part + (static_cast<int64_t>(sp) * Q * args.N + n) * 4;
              uint32_t v[C::kCPT];
              got = poll_partials_quads<C::kCPT>(src, gstride, args.M, v, abort_flag, limit);
              if (got) {
#pragma unroll
                for (int j = 0; j < C::kCPT; ++j) sum[j] += __uint_as_float(v[j] - 1u);
              }
            }
            if (got) {
#pragma unroll
              for (int j = 0; j < C::kCPT; ++j)
                if (j < args.M) {
                  __nv_bfloat16 h = __float2bfloat16_rn(sum[j] + bv);
                  y[static_cast<int64_t>(j) * args.N + n] = *reinterpret_cast<uint16_t *>(&h);
                }
              // consumed: back to "not written" for the next call
              for (int sp = 1; sp < shape.splits; ++sp) {
                uint32_t *src = part + (static_cast<int64_t>(sp) * Q * args.N + n) * 4;
#pragma unroll
                for (int q = 0; q < C::kCPT / 4; ++q)
                  if (4 * q < args.M)
                    *reinterpret_cast<uint4 *>(src + q * gstride) = make_uint4(0u, 0u, 0u, 0u);
              }
            } else {
              record_timeout(args);
            }
          } else if (w.split != 0) {
            if (n_ok) {
              uint32_t *dst = part + static_cast<int64_t>(w.split) * args.M * args.N + n;
#pragma unroll
              for (int j = 0; j < C::kCPT; ++j)
                if (j < args.M &&
                    write_ok(args, (dst - part) + static_cast<int64_t>(j) * args.N <
                                       args.partials_bytes / 4))
                  st_relaxed_gpu(dst + static_cast<int64_t>(j) * args.N, __float_as_uint(acc[j]) + 1u);
            }
          } else if (n_ok) {
            float sum[C::kCPT];
#pragma unroll
            for (int j = 0; j < C::kCPT; ++j) sum[j] = acc[j];
            bool got = true;
            for (int sp = 1; sp < shape.splits && got; ++sp) {
              uint32_t *src = part + static_cast<int64_t>(sp) * args.M * args.N + n;
              uint32_t v[C::kCPT];
              got = poll_partials<C::kCPT>(src, args.N, args.M, v, abort_flag, limit);
              if (got) {
#pragma unroll
                for (int j = 0; j < C::kCPT; ++j) sum[j] += __uint_as_float(v[j] - 1u);
              }
            }
            if (got) {
#pragma unroll
              for (int j = 0; j < C::kCPT; ++j)
                if (j < args.M) {
                  __nv_bfloat16 h = __float2bfloat16_rn(sum[j] + bv);
                  y[static_cast<int64_t>(j) * args.N + n] = *reinterpret_cast<uint16_t *>(&h);
                }
              // consumed: back to "not written" for the next call
              for (int sp = 1; sp < shape.splits; ++sp) {
                uint32_t *src = part + static_cast<int64_t>(sp) * args.M * args.N + n;
#pragma unroll
                for (int j = 0; j < C::kCPT; ++j)
                  if (j < args.M) src[static_cast<int64_t>(j) * args.N] = 0u;
              }
            } else {
              record_timeout(args);
            }
          }
        }
      }
    }
    // the staging boxes stay in use until this warp's TMA stores complete
    if (C::kTmaStoreY && lane == 0) bulk_wait_group0();
    if (!ok && et == 0) record_timeout(args);
  } else if (C::kFuseQ) {
    // ------------------------------------------------------------ fused activation quantiser
    // Per K block: the group-128 quantisation of every token's 128 BF16 values
    // in the stage (one group per token: s = amax / 448 from the scale table,
    // codes = RNE_sat(x / s) from the FMA-corrected quotient -- the arithmetic
    // of the activation quantiser kernel, so the codes and scales are the
    // same bits), codes into the stage's E4M3 operand in the 128-byte swizzled
    // layout the MMA reads, scales into sx_stage for the promotion.  Eight
    // threads per token, 16 values each.
    const int qt = threadIdx.x - 32 * C::kQBase;  // 0 .. 32 * kQWarps - 1
    const int qw = qt >> 5;
    // Token rows >= M only feed output columns that are never stored, so a
    // stage needs only the tasks of rows below M, rounded up to whole warps
    // (every lane of a warp that works runs the shuffles; only rows < M
    // store).  The quantiser warps form groups of `wps` warps that take the
    // stages in turn -- with four tokens or fewer and eight quantiser warps,
    // each warp quantises every eighth stage.  The number of groups divides
    // STAGES, so each group owns
    // fixed stages and its previous wait on a stage was one ring ago: a
    // barrier phase it waits for is never two phases away.
    const int lim = min(BN * 8, (args.M * 8 + 31) / 32 * 32);
    const int wps = fused_quant_warps_per_stage<BN, C::kQWarps>(args.M);  // warps per stage
    int groups = C::kQWarps / wps;  // a power of two
    while (STAGES % groups != 0) groups >>= 1;
    const int grp = qw / wps;                // this warp's group
    const int t0 = (qw % wps) * 32 + lane;   // first task of this thread in a stage
    ScaleTable &table = *reinterpret_cast<ScaleTable *>(sx_stage + shape.sx_stage);
    for (int m = qt; m <= 128; m += 32 * C::kQWarps) {
      const float a = m < 128 ? 1.0f + static_cast<float>(m) * 0.0078125f : kFloor;
      const float sv = __fdiv_rn(a, 448.0f);
      const float2 v = make_float2(sv, __frcp_rn(sv));
      if (m < 128) table.e[m] = v;
      else table.floor_entry = v;
    }
    named_bar_sync(3, 32 * C::kQWarps);
    uint32_t it = 0;
    bool ok = true;
    for (int u = cl_id; ok && u < units; u += cl_num) {
      const Unit w = decode_unit<SWAP, PAIR, GROUPED>(u, num_a, shape.splits, shape.kps, KB, BN, rank, args.M, args.N, gt, shape);
      for (int kb = w.kb0; kb < w.kb1; ++kb, ++it) {
        if (grp >= groups || static_cast<int>(it & (groups - 1)) != grp) continue;
        const uint32_t s = it % STAGES, ph = (it / STAGES) & 1u;
        if (!warp_wait(&bars->full[s], ph, abort_flag, limit)) {
          ok = false;
          break;
        }
        uint8_t *codes = sB + s * C::kBbytes;
        const uint8_t *xs = codes + C::kBrows * 128;
        for (int task = t0; task < lim; task += 32 * wps) {
          const int t = task >> 3, sub = task & 7;
          uint4 v[2];
          v[0] = *reinterpret_cast<const uint4 *>(xs + t * 256 + sub * 32);
          v[1] = *reinterpret_cast<const uint4 *>(xs + t * 256 + sub * 32 + 16);
          float f[16];
          unpack16(v, f);
          float amax = amax16(f);
          amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
          amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
          amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 4));
          const float2 sc = scale_of(table, amax);
          // 16-byte chunk c of row t sits at chunk position c ^ (t % 8)
          const uint4 out = quant16<1>(v, f, sc.x, sc.y);
          if (t < args.M) {
            *reinterpret_cast<uint4 *>(codes + t * 128 + ((sub ^ (t & 7)) << 4)) = out;
            if (sub == 0) sx_stage[(kb - w.kb0) * BN + t] = sc.x;
          }
        }
        // the operand is read by the tensor cores (async proxy)
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->qfull[s]);
      }
    }
    if (!ok && qt == 0) record_timeout(args);
  }

  // ------------------------------------------------------------ teardown
  tc_fence_before();
  __syncthreads();
  if (PAIR) cluster_sync();  // no CTA leaves while its peer may still signal it
  if (warp == 1) {
    tc_fence_after();
    if (PAIR) tmem_dealloc_pair(tmem_base, C::kTmemCols);
    else tmem_dealloc(tmem_base, C::kTmemCols);
  }
}

// The last wave of block pair tiles: the tiles left after the full waves of
// `clusters` (the clusters the device holds at once) occupy only some of them;
// with fewer tiles than clusters, that is every tile.  When they fill at most
// half, each is
// split into up to 4 K ranges (multiples of 4 blocks: the promotion factors
// arrive four K blocks per TMA box) that run on otherwise idle clusters; the
// last range of a tile to finish sums the others' promoted partials in range
// order.  Needs room for the partials in the workspace.
inline void split_tail_tiles(LaunchShape &sh, int clusters, int64_t partials_bytes) {
  const int T = sh.units % clusters;
  if (T == 0 || 2 * T > clusters) return;
  int S = clusters / T;
  if (S > 4) S = 4;
  if (S > sh.KB / 4) S = sh.KB / 4;
  if (S < 2) return;
  const int kps = ((sh.KB + S - 1) / S + 3) / 4 * 4;
  S = (sh.KB + kps - 1) / kps;
  const int64_t items = static_cast<int64_t>(T) * S;
  if (S < 2 || items > kMaxTailItems || items * kTailItemBytes > partials_bytes) return;
  sh.full_units = sh.units - T;
  sh.tail_splits = S;
  sh.tail_kps = kps;
  sh.units = sh.full_units + T * S;
}

// Launches one variant.  `grid` counts CTAs for single-CTA tiles and clusters
// for pair tiles; for pair tiles it is clamped to the clusters the device can
// hold at once, so the persistent grid is a single wave.
template <int MODE, bool SWAP, int BN, int STAGES, int EPI_WARPS, int ACCB, bool PAIR,
          bool GROUPED = false, bool FUSEQ = false>
cudaError_t run(const GemmArgs &a, const void *q_act, const void *w, const LaunchShape &sh,
                int grid, cudaStream_t st, int *status) {
  using C = Cfg<MODE, SWAP, BN, STAGES, EPI_WARPS, ACCB, PAIR, GROUPED, FUSEQ>;
  static_assert(!GROUPED || (MODE == kModeBlock && !SWAP), "grouped: block tiles");
  if (GROUPED != (a.g_experts > 0)) {
    *status = 4;  // FP8BQ_ERR_UNSUPPORTED: grouped arguments to a plain variant or back
    return cudaSuccess;
  }
  CUtensorMap ta, tb, ty, tsx, tsw;
  std::memset(&ty, 0, sizeof ty);
  std::memset(&tsx, 0, sizeof tsx);
  std::memset(&tsw, 0, sizeof tsw);
  GemmArgs args = a;
  // decode tiles: B carries the tokens, and only the first M rows (rounded up
  // to the 8-row swizzle atom) are copied
  args.b_box_rows = SWAP ? ((a.M + 7) / 8 * 8 < C::kBrows ? (a.M + 7) / 8 * 8 : C::kBrows)
                         : C::kBrows;
  args.y_tma = 0;
  args.sc_tma = 0;
  auto al16 = [](const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
  if (C::kTmaStoreY && a.N % 8 == 0 && al16(a.y))
    args.y_tma = cached_bf16_rows_map(&ty, a.y, a.M, a.N, C::kYBoxCols, 32) ? 1 : 0;
  if (C::kScRing) {
    // s_x: row-major [M][KB] in [128 rows x 4 K blocks] boxes, or column-major
    // [KB][ldsx] in [4 K blocks x 128 rows] boxes; s_w [NB][KB] in [2 x 4] boxes
    const int KB = (a.K + 127) / 128, NB = (a.N + kBlockN - 1) / kBlockN;
    // column-major s_x puts the token row on the box's inner coordinate, which
    // must be a multiple of 4 floats: grouped tiles start at any row, so they
    // take the per-thread path there
    const bool sx_ok = al16(a.sx) && a.ldsx % 4 == 0 && (a.sx_layout == 0 || a.g_experts == 0) &&
                       (a.sx_layout == 0
                            ? cached_f32_map(&tsx, a.sx, a.M, KB, a.ldsx, C::kScQuad, kBM)
                            : cached_f32_map(&tsx, a.sx, KB, a.ldsx, a.ldsx, kBM, C::kScQuad));
    const int experts = a.g_experts > 0 ? a.g_experts : 1;
    const bool sw_ok = al16(a.sw) && KB % 4 == 0 &&
                       cached_f32_map(&tsw, a.sw, static_cast<int64_t>(NB) * experts, KB, KB,
                                      C::kScQuad, 2);
    args.sc_tma = (sx_ok && sw_ok) ? 1 : 0;
  }
  if (MODE == kModeMx) {
    // scale-factor chunks as rows of 256 bytes (typed FP32 only to describe the
    // copy): 2 rows per activation chunk, kSfBBytes / 256 per weight chunk
    const int64_t KB = (a.K + 127) / 128;
    const int64_t rows_a = (a.M + kBM - 1) / kBM * KB * 2;
    const int64_t rows_b = (a.N + BN - 1) / BN * KB * (C::kSfBBytes / 256);
    if (!al16(a.ux) || !al16(a.uw) || !cached_f32_map(&tsx, a.ux, rows_a, 64, 64, 64, 2) ||
        !cached_f32_map(&tsw, a.uw, rows_b, 64, 64, 64, C::kSfBBytes / 256)) {
      *status = 4;  // FP8BQ_ERR_UNSUPPORTED: tensor map rejected
      return cudaSuccess;
    }
  }
  const void *a_ptr = SWAP ? w : q_act;
  const void *b_ptr = SWAP ? q_act : w;
  const int64_t a_rows = SWAP ? a.N : a.M;
  // grouped form: all experts' weights as one [E * N, K] operand
  const int64_t b_rows = SWAP ? a.M : static_cast<int64_t>(a.N) * (a.g_experts > 0 ? a.g_experts : 1);
  // fused quantisation: B is the BF16 activation matrix [M, K] (pitch ldxq),
  // loaded unswizzled in [kBrows tokens x 128 values] boxes
  const bool b_ok = FUSEQ ? (a.xq != nullptr && al16(a.xq) &&
                             cached_bf16_pitched_map(&tb, a.xq, a.M, a.K, a.ldxq, 128, args.b_box_rows))
                          : cached_kmajor_map(&tb, b_ptr, b_rows, a.K, args.b_box_rows);
  if (!cached_kmajor_map(&ta, a_ptr, a_rows, a.K, kBM) || !b_ok) {
    *status = 4;  // FP8BQ_ERR_UNSUPPORTED: tensor map rejected
    return cudaSuccess;
  }
  const size_t smem = C::kFixedSmem + static_cast<size_t>(sh.sx_stage) * sizeof(float) +
                      (FUSEQ ? sizeof(ScaleTable) : 0);
  auto kern = fp8_gemm_kernel<MODE, SWAP, BN, STAGES, EPI_WARPS, ACCB, PAIR, GROUPED, FUSEQ>;
  // the opt-in shared-memory limit is raised once per variant to the largest
  // request it can see: the fixed part plus the biggest s_x staging buffer
  // (swapped tiles) or, where it fits in 227 KB, the grouped form's tile table
  // (pair tiles)
  constexpr size_t kSmemCap = 227 * 1024;
  constexpr size_t kTail = SWAP ? size_t(BN) * 64 * sizeof(float) + (FUSEQ ? sizeof(ScaleTable) : 0)
                           : GROUPED ? kGroupTableBytes
                                                                                     : 0;
  static_assert(C::kFixedSmem + kTail <= kSmemCap, "shared memory");
  if (smem > C::kFixedSmem + kTail) {
    *status = 4;  // FP8BQ_ERR_UNSUPPORTED: the variant has no room for this request
    return cudaSuccess;
  }
  static std::once_flag attr_once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(attr_once, [&] {
    attr_err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    static_cast<int>(C::kFixedSmem + kTail));
  });
  cudaError_t e = attr_err;
  if (e != cudaSuccess) return e;
  if (C::kRegSplit) {
    // setmaxnreg.inc waits for registers the block was launched with: refuse
    // to launch unless the compiled register count covers the split
    static std::once_flag regs_once;
    static int regs = 0;
    std::call_once(regs_once, [&] {
      cudaFuncAttributes fa;
      if (cudaFuncGetAttributes(&fa, kern) == cudaSuccess) regs = fa.numRegs;
    });
    if (static_cast<long>(regs) * C::kThreads <
        128L * C::kLowRegs + static_cast<long>(C::kThreads - 128) * C::kHighRegs) {
      *status = 4;  // FP8BQ_ERR_UNSUPPORTED: build does not fit the register split
      return cudaSuccess;
    }
  }
  if (!PAIR) {
    e = launch_pdl(kern, grid, C::kThreads, smem, st, ta, tb, ty, tsx, tsw, args, sh);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
  }
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.blockDim = dim3(C::kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  // clusters the device holds at once, queried once per variant (the library
  // targets one device type); thread-safe like the attribute set-up above
  static std::once_flag occ_once;
  static int max_clusters = 0;
  static cudaError_t occ_err = cudaSuccess;
  std::call_once(occ_once, [&] {
    cudaLaunchConfig_t q = cfg;
    q.gridDim = dim3(2 * grid, 1, 1);
    int n = 0;
    occ_err = cudaOccupancyMaxActiveClusters(&n, kern, &q);
    max_clusters = n > 0 ? n : 1;
  });
  if (occ_err != cudaSuccess) return occ_err;
  // block tiles: the last wave (all of them when there are fewer tiles than
  // the device holds clusters) may be split over idle clusters; the grid then
  // covers the split units
  LaunchShape shx = sh;
  int want = grid;
  if (MODE == kModeBlock && !GROUPED) {
    split_tail_tiles(shx, max_clusters, args.partials_bytes);
    if (shx.units > want) want = shx.units;
  }
  const int clusters = want < max_clusters ? want : max_clusters;
  cfg.gridDim = dim3(2 * clusters, 1, 1);
  e = cudaLaunchKernelEx(&cfg, kern, ta, tb, ty, tsx, tsw, args, shx);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace
}  // namespace fp8bq
