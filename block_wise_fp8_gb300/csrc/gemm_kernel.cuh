// gemm_kernel.cuh -- FP8 GEMMs on the 5th-generation tensor cores (tcgen05 + TMEM + TMA).
//
// One warp-specialised kernel template covers the three scalings of the pages
// ("SGLang 源码完全拆解(十九)", §一条 GEMM 的三种缩放组合):
//
//   kModeBlock   y = sum_b P_b * s_x[i][b] * s_w[j/128][b]   (128x128 weight blocks,
//                1x128 activation groups).  The tensor core produces P_b, the FP32
//                sum over one 128-wide K block, into TMEM; the epilogue warps read
//                it back and promote it into FP32 registers with one FMA per
//                element and K block (the per-128-K promotion of "GLM-5.3 推理全链路
//                (十七)", DeepSeek-V3 Fig. 7 paragraph).  TMEM holds two partial
//                buffers so the MMA of block b+1 overlaps the promotion of block b.
//   kModeTensor  y = (sum_k q w) * s_x * s_w[p(j)]: full-K accumulation in TMEM,
//                one scale product per column in the epilogue.
//   kModeMx      y = sum_g P_g * 2^(ua-127) * 2^(uw-127) with the block-scaled MMA
//                (kind::mxf8f6f4, one UE8M0 scale per 32 K); the scale factors are
//                written into TMEM by dedicated warps, so no dequantisation runs in
//                software ("GLM-5.3 推理全链路(十七)", §第7站).
//
// Roles (warp index):
//   0            TMA producer: A and B tiles, 128 K per stage, 128B-swizzled.
//   1            TMEM allocator and single-thread MMA issuer.
//   2 .. 2+SFW   (MX only) scale-factor writers, one per TMEM lane quarter.
//   rest         epilogue: TMEM -> registers -> promotion -> BF16 -> global.
//
// Two tile orientations:
//   normal  UMMA M = 128 tokens, UMMA N = BN weight rows (prefill).
//   swap    UMMA M = 128 weight rows, UMMA N = BN tokens (decode, M <= 64), with
//           split-K across CTAs and a deterministic last-CTA reduction in
//           ascending split order.
//
// Every wait is bounded (see ptx.cuh); a CTA that gives up records a timeout in
// the workspace status word, lets its in-flight copies and MMAs land, frees its
// TMEM and exits.
#pragma once
#include <cuda_bf16.h>

#include "common.cuh"
#include "ptx.cuh"

namespace fp8bq {
namespace {

constexpr int kBM = 128;           // UMMA M
constexpr int kAbytes = kBM * 128; // one A stage (128 rows x 128 B)

constexpr uint32_t pow2_at_least(uint32_t v) {
  uint32_t p = 32;
  while (p < v) p <<= 1;
  return p;
}

template <int MODE, bool SWAP, int BN, int STAGES, int EPI_WARPS>
struct Cfg {
  static constexpr int kSfWarps = (MODE == kModeMx) ? 4 : 0;
  static constexpr int kSfSlots = 4;
  static constexpr int kSfColsA = 4;            // 128 rows / 32
  static constexpr int kSfColsB = (MODE == kModeMx) ? BN / 32 : 4;
  static constexpr int kSfSlotCols = 16;        // A at +0, B at +8
  static constexpr int kThreads = 64 + 32 * (kSfWarps + EPI_WARPS);
  static constexpr int kEpiThreads = 32 * EPI_WARPS;
  static constexpr int kEpiBase = 2 + kSfWarps;  // first epilogue warp
  static constexpr int kColGroups = EPI_WARPS / 4;
  static constexpr int kCPT = BN / kColGroups;    // columns per epilogue thread
  static constexpr int kCW = (kCPT % 32 == 0) ? 32 : 16;  // tcgen05.ld chunk width
  static constexpr int kBatch = (kCPT < 64) ? kCPT : 64;  // columns per wait::ld
  static constexpr int kBbytes = BN * 128;
  static constexpr int kStageBytes = kAbytes + kBbytes;
  static constexpr int kAccCols = 2 * BN;  // double-buffered accumulators / partials
  static constexpr int kSfBase = kAccCols;
  static constexpr uint32_t kTmemCols =
      pow2_at_least(kAccCols + (MODE == kModeMx ? kSfSlots * kSfSlotCols : 0));
  static constexpr int kBarBytes = 512;
  // dynamic shared memory: [align slack][A stages][B stages][barriers][sx stage]
  static constexpr size_t kFixedSmem = 1024 + size_t(STAGES) * kStageBytes + kBarBytes;

  static_assert(EPI_WARPS % 4 == 0, "epilogue warps must cover the 4 TMEM lane quarters");
  static_assert(BN % 16 == 0 && BN >= 16 && BN <= 256, "UMMA N for M = 128");
  static_assert(kCPT % kCW == 0 && kBatch % kCW == 0 && kCPT % kBatch == 0, "chunking");
  static_assert(kTmemCols <= 512, "TMEM columns");
  static_assert(MODE != kModeMx || (!SWAP && BN % 32 == 0 && kSfColsB <= 8), "MX tiles");
};

struct SmemBarriers {
  uint64_t full[8], empty[8];
  uint64_t tfull[2], tempty[2];
  uint64_t sf_full[4], sf_empty[4];
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

__device__ __forceinline__ void record_timeout(const GemmArgs &a) {
  if (a.status) atomicExch(a.status, kStatusTimeout);
}

// every lane waits; the warp proceeds only if all lanes saw the phase complete
__device__ __forceinline__ bool warp_wait(uint64_t *bar, uint32_t parity, volatile uint32_t *ab,
                                          uint64_t limit) {
  const bool ok = mbar_wait(bar, parity, ab, limit);
  return __all_sync(0xffffffffu, ok);
}

// Work unit -> (row0 of A, row0 of B, kb range, split, tile id for counters).
struct Unit {
  int a_row0, b_row0, kb0, kb1, split, tile;
};

template <bool SWAP>
__device__ __forceinline__ Unit decode_unit(int u, int num_a_tiles, int splits, int kps, int KB,
                                            int bn) {
  Unit r;
  if (SWAP) {
    // A = weight rows (128 per tile), B = all tokens; units = tiles x splits
    r.tile = u / splits;
    r.split = u - r.tile * splits;
    r.a_row0 = r.tile * kBM;
    r.b_row0 = 0;
  } else {
    // A = tokens (128 per tile), B = weight rows (bn per tile); M fastest so
    // concurrently running CTAs share weight tiles in L2
    const int mt = u % num_a_tiles, nt = u / num_a_tiles;
    r.tile = u;
    r.split = 0;
    r.a_row0 = mt * kBM;
    r.b_row0 = nt * bn;
  }
  r.kb0 = r.split * kps;
  r.kb1 = min(KB, r.kb0 + kps);
  return r;
}

template <int MODE, bool SWAP, int BN, int STAGES, int EPI_WARPS>
__global__ void __launch_bounds__(Cfg<MODE, SWAP, BN, STAGES, EPI_WARPS>::kThreads, 1)
    fp8_gemm_kernel(const __grid_constant__ CUtensorMap tmA,
                    const __grid_constant__ CUtensorMap tmB,
                    const __grid_constant__ GemmArgs args, const LaunchShape shape) {
  using C = Cfg<MODE, SWAP, BN, STAGES, EPI_WARPS>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t *smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
  uint8_t *sA = smem;
  uint8_t *sB = smem + STAGES * kAbytes;
  SmemBarriers *bars = reinterpret_cast<SmemBarriers *>(smem + STAGES * C::kStageBytes);
  float *sx_stage = reinterpret_cast<float *>(smem + STAGES * C::kStageBytes + C::kBarBytes);
  volatile uint32_t *abort_flag = &bars->abort;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint64_t limit = args.wait_limit_ns;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&bars->full[s], 1);
      mbar_init(&bars->empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&bars->tfull[b], 1);
      mbar_init(&bars->tempty[b], EPI_WARPS);
    }
    for (int s = 0; s < C::kSfSlots; ++s) {
      mbar_init(&bars->sf_full[s], C::kSfWarps > 0 ? C::kSfWarps : 1);
      mbar_init(&bars->sf_empty[s], 1);
    }
    mbar_init(&bars->drain, 1);
    bars->abort = 0;
    bars->is_last = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
  }
  if (warp == 1) {
    tmem_alloc(&bars->tmem_base, C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = bars->tmem_base;

  const int KB = shape.KB;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      int last_phase[STAGES];
      for (int s = 0; s < STAGES; ++s) last_phase[s] = -1;
      uint32_t it = 0;
      bool ok = true;
      for (int u = blockIdx.x; ok && u < shape.units; u += gridDim.x) {
        const Unit w = decode_unit<SWAP>(u, shape.num_a_tiles, shape.splits, shape.kps, KB, BN);
        for (int kb = w.kb0; kb < w.kb1; ++kb, ++it) {
          const uint32_t s = it % STAGES, ph = (it / STAGES) & 1u;
          if (!mbar_wait(&bars->empty[s], ph ^ 1u, abort_flag, limit)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&bars->full[s], C::kStageBytes);
          tma_load_2d(sA + s * kAbytes, &tmA, &bars->full[s], kb * 128, w.a_row0);
          tma_load_2d(sB + s * C::kBbytes, &tmB, &bars->full[s], kb * 128, w.b_row0);
          last_phase[s] = static_cast<int>(ph);
        }
      }
      if (!ok) {
        record_timeout(args);
        // let every copy this thread issued land before the CTA's smem goes away
        for (int s = 0; s < STAGES; ++s)
          if (last_phase[s] >= 0) {
            uint32_t dummy = 0;
            mbar_wait(&bars->full[s], static_cast<uint32_t>(last_phase[s]), &dummy, limit);
          }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      uint32_t it = 0, kit = 0, uit = 0, sfit = 0;
      bool ok = true;
      for (int u = blockIdx.x; ok && u < shape.units; u += gridDim.x, ++uit) {
        const Unit w = decode_unit<SWAP>(u, shape.num_a_tiles, shape.splits, shape.kps, KB, BN);
        if (MODE != kModeBlock) {
          const uint32_t b = uit & 1u, ph = (uit >> 1) & 1u;
          if (!mbar_wait(&bars->tempty[b], ph ^ 1u, abort_flag, limit)) {
            ok = false;
            break;
          }
          tc_fence_after();
        }
        for (int kb = w.kb0; kb < w.kb1; ++kb, ++it) {
          uint32_t d_tmem;
          if (MODE == kModeBlock) {
            const uint32_t b = kit & 1u, ph = (kit >> 1) & 1u;
            if (!mbar_wait(&bars->tempty[b], ph ^ 1u, abort_flag, limit)) {
              ok = false;
              break;
            }
            d_tmem = tmem_base + b * BN;
          } else {
            d_tmem = tmem_base + (uit & 1u) * BN;
          }
          const uint32_t s = it % STAGES, ph = (it / STAGES) & 1u;
          if (!mbar_wait(&bars->full[s], ph, abort_flag, limit)) {
            ok = false;
            break;
          }
          uint32_t sfslot = 0;
          if (MODE == kModeMx) {
            sfslot = sfit % C::kSfSlots;
            if (!mbar_wait(&bars->sf_full[sfslot], (sfit / C::kSfSlots) & 1u, abort_flag,
                           limit)) {
              ok = false;
              break;
            }
          }
          tc_fence_after();
          const uint64_t adesc = sdesc_kmajor_sw128(smem_u32(sA + s * kAbytes));
          const uint64_t bdesc = sdesc_kmajor_sw128(smem_u32(sB + s * C::kBbytes));
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            // advance 32 K-bytes inside the 128-byte swizzled row: +2 in the >>4 field
            const uint32_t acc = (MODE == kModeBlock) ? (k > 0) : (kb > w.kb0 || k > 0);
            if (MODE == kModeMx) {
              const uint32_t sfcol = tmem_base + C::kSfBase + sfslot * C::kSfSlotCols;
              umma_mxf8f6f4(d_tmem, adesc + 2 * k, bdesc + 2 * k, idesc_mxf8_e4m3(kBM, BN, k, k),
                            sfcol, sfcol + 8, acc);
            } else {
              umma_f8f6f4(d_tmem, adesc + 2 * k, bdesc + 2 * k, idesc_f8f6f4_e4m3(kBM, BN), acc);
            }
          }
          umma_commit(&bars->empty[s]);
          if (MODE == kModeMx) {
            umma_commit(&bars->sf_empty[sfslot]);
            ++sfit;
          }
          if (MODE == kModeBlock) {
            umma_commit(&bars->tfull[kit & 1u]);
            ++kit;
          }
        }
        if (!ok) break;
        if (MODE != kModeBlock) umma_commit(&bars->tfull[uit & 1u]);
      }
      if (!ok) record_timeout(args);
      // every MMA issued by this thread has completed once `drain` flips
      umma_commit(&bars->drain);
      uint32_t dummy = 0;
      mbar_wait(&bars->drain, 0, &dummy, limit);
    }
    __syncwarp();
  } else if (warp < C::kEpiBase) {
    // ------------------------------------------------------------ MX scale-factor writers
    // Warp with lane quarter q writes TMEM lanes 32q..32q+31.  Layout (replicated in
    // every quarter): lane i, column c of a slot holds the four UE8M0 codes of stage
    // kb (K groups 4kb..4kb+3, one byte per MMA, selected by the sf id) of tile row
    // i + 32c.
    if (MODE == kModeMx) {
      const int q = warp & 3;
      const int G = args.K / 32;
      uint32_t sfit = 0;
      bool ok = true;
      for (int u = blockIdx.x; ok && u < shape.units; u += gridDim.x) {
        const Unit w = decode_unit<SWAP>(u, shape.num_a_tiles, shape.splits, shape.kps, KB, BN);
        for (int kb = w.kb0; kb < w.kb1; ++kb, ++sfit) {
          uint32_t va[C::kSfColsA], vb[C::kSfColsB];
#pragma unroll
          for (int c = 0; c < C::kSfColsA; ++c) {
            const int r = w.a_row0 + lane + 32 * c;
            uint32_t v = 0;
            if (r < args.M) {
              const uint8_t *p = args.ux + static_cast<int64_t>(r) * G + 4 * kb;
#pragma unroll
              for (int g = 0; g < 4; ++g)
                if (4 * kb + g < G) v |= static_cast<uint32_t>(__ldg(p + g)) << (8 * g);
            }
            va[c] = v;
          }
#pragma unroll
          for (int c = 0; c < C::kSfColsB; ++c) {
            const int r = w.b_row0 + lane + 32 * c;
            uint32_t v = 0;
            if (r < args.N) {
              const uint8_t *p = args.uw + static_cast<int64_t>(r) * G + 4 * kb;
#pragma unroll
              for (int g = 0; g < 4; ++g)
                if (4 * kb + g < G) v |= static_cast<uint32_t>(__ldg(p + g)) << (8 * g);
            }
            vb[c] = v;
          }
          const uint32_t slot = sfit % C::kSfSlots;
          if (!warp_wait(&bars->sf_empty[slot], ((sfit / C::kSfSlots) & 1u) ^ 1u, abort_flag,
                         limit)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t col =
              tmem_base + (static_cast<uint32_t>(32 * q) << 16) + C::kSfBase + slot * C::kSfSlotCols;
          tmem_st4(col, va[0], va[1], va[2], va[3]);
#pragma unroll
          for (int c = 0; c < C::kSfColsB; c += 4)
            tmem_st4(col + 8 + c, vb[c], vb[c + 1], vb[c + 2], vb[c + 3]);
          tmem_st_wait();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&bars->sf_full[slot]);
        }
      }
      if (!ok && lane == 0) record_timeout(args);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    const int ew = warp - C::kEpiBase;
    const int quarter = warp & 3;
    const int cg = ew >> 2;  // column group
    const int et = ew * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>(32 * quarter) << 16;
    const int NB = (args.N + kBlockN - 1) / kBlockN;
    uint32_t kit = 0, uit = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < shape.units; u += gridDim.x, ++uit) {
      const Unit w = decode_unit<SWAP>(u, shape.num_a_tiles, shape.splits, shape.kps, KB, BN);
      const int d_row = w.a_row0 + 32 * quarter + lane;  // row of D held by this thread
      const int col0 = cg * C::kCPT;                     // first D column of this thread
      float acc[C::kCPT];
#pragma unroll
      for (int j = 0; j < C::kCPT; ++j) acc[j] = 0.0f;

      if (MODE == kModeBlock && SWAP) {
        // stage s_x[token][kb] for this unit's K range: sx_stage[(kb-kb0)*BN + token]
        const int nkb = w.kb1 - w.kb0;
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
      }

      if (MODE == kModeBlock) {
        const bool row_ok = d_row < (SWAP ? args.N : args.M);
        auto sx_at = [&](int kb) -> float {
          if (!row_ok || kb >= w.kb1) return 0.0f;
          return __ldg(args.sx + (args.sx_layout == 0
                                      ? static_cast<int64_t>(d_row) * args.ldsx + kb
                                      : static_cast<int64_t>(kb) * args.ldsx + d_row));
        };
        float sx_next = SWAP ? 0.0f : sx_at(w.kb0);
        for (int kb = w.kb0; kb < w.kb1 && ok; ++kb, ++kit) {
          const uint32_t b = kit & 1u, ph = (kit >> 1) & 1u;
          const float sx_cur = sx_next;
          if (!SWAP) sx_next = sx_at(kb + 1);
          if (!warp_wait(&bars->tfull[b], ph, abort_flag, limit)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t tbase = tmem_base + lane_base + b * BN + col0;
#pragma unroll
          for (int bt = 0; bt < C::kCPT / C::kBatch; ++bt) {
            uint32_t r[C::kBatch];
#pragma unroll
            for (int c = 0; c < C::kBatch / C::kCW; ++c) {
              if (C::kCW == 32) tmem_ld32(tbase + bt * C::kBatch + c * 32, r + c * 32);
              else tmem_ld16(tbase + bt * C::kBatch + c * 16, r + c * 16);
            }
            tmem_ld_wait();
            if (bt == C::kCPT / C::kBatch - 1) {
              tc_fence_before();
              __syncwarp();
              if (lane == 0) mbar_arrive(&bars->tempty[b]);
            }
            if (SWAP) {
              // lanes are weight rows of one 128-row block: one s_w per K block
              const float swv = __ldg(args.sw + static_cast<int64_t>(w.a_row0 / kBlockN) * KB + kb);
              const float *sxk = sx_stage + (kb - w.kb0) * BN;
#pragma unroll
              for (int j = 0; j < C::kBatch; ++j) {
                const int jj = bt * C::kBatch + j;
                acc[jj] = fmaf(__uint_as_float(r[j]), sxk[col0 + jj] * swv, acc[jj]);
              }
            } else {
#pragma unroll
              for (int c = 0; c < C::kBatch / C::kCW; ++c) {
                const int n = w.b_row0 + col0 + bt * C::kBatch + c * C::kCW;
                const int nb = min(n / kBlockN, NB - 1);
                const float f = sx_cur * __ldg(args.sw + static_cast<int64_t>(nb) * KB + kb);
#pragma unroll
                for (int j = 0; j < C::kCW; ++j) {
                  const int jj = bt * C::kBatch + c * C::kCW + j;
                  acc[jj] = fmaf(__uint_as_float(r[c * C::kCW + j]), f, acc[jj]);
                }
              }
            }
          }
        }
      } else if (ok) {
        // kModeTensor / kModeMx: one read of the full-K accumulator
        const uint32_t b = uit & 1u, ph = (uit >> 1) & 1u;
        if (!warp_wait(&bars->tfull[b], ph, abort_flag, limit)) {
          ok = false;
        } else {
          tc_fence_after();
          const uint32_t tbase = tmem_base + lane_base + b * BN + col0;
#pragma unroll
          for (int bt = 0; bt < C::kCPT / C::kBatch; ++bt) {
            uint32_t r[C::kBatch];
#pragma unroll
            for (int c = 0; c < C::kBatch / C::kCW; ++c) {
              if (C::kCW == 32) tmem_ld32(tbase + bt * C::kBatch + c * 32, r + c * 32);
              else tmem_ld16(tbase + bt * C::kBatch + c * 16, r + c * 16);
            }
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < C::kBatch; ++j) acc[bt * C::kBatch + j] = __uint_as_float(r[j]);
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&bars->tempty[b]);
          if (MODE == kModeTensor) {
            const float sxs = __ldg(args.sx_scalar);
            if (SWAP) {
              // one output partition per lane (weight row)
              int p = 0;
              while (p < args.n_parts - 1 && d_row >= args.part_end[p]) ++p;
              const float f = sxs * __ldg(args.sw_part + p);
#pragma unroll
              for (int j = 0; j < C::kCPT; ++j) acc[j] *= f;
            } else {
#pragma unroll
              for (int j = 0; j < C::kCPT; ++j) {
                const int n = w.b_row0 + col0 + j;
                int p = 0;
                while (p < args.n_parts - 1 && n >= args.part_end[p]) ++p;
                acc[j] *= sxs * __ldg(args.sw_part + p);
              }
            }
          }
        }
      }

      // all epilogue warps agree on the outcome before anything is stored
      named_bar_sync(2, C::kEpiThreads);
      if (*abort_flag) {
        ok = false;
        break;
      }

      const __nv_bfloat16 *bias = static_cast<const __nv_bfloat16 *>(args.bias);
      uint16_t *y = static_cast<uint16_t *>(args.y);
      if (!SWAP) {
        // thread holds row d_row, columns b_row0 + col0 + [0, kCPT)
        const int m = d_row;
        const int nbase = w.b_row0 + col0;
        if (m < args.M) {
          if (bias) {
#pragma unroll
            for (int j = 0; j < C::kCPT; ++j)
              if (nbase + j < args.N)
                acc[j] += bf16_bits_to_float(reinterpret_cast<const uint16_t *>(bias)[nbase + j]);
          }
          uint16_t *yr = y + static_cast<int64_t>(m) * args.N;
          if ((args.N & 7) == 0) {
#pragma unroll
            for (int j = 0; j < C::kCPT; j += 8) {
              if (nbase + j < args.N) {
                uint4 v;
                v.x = pack_bf16x2(acc[j], acc[j + 1]);
                v.y = pack_bf16x2(acc[j + 2], acc[j + 3]);
                v.z = pack_bf16x2(acc[j + 4], acc[j + 5]);
                v.w = pack_bf16x2(acc[j + 6], acc[j + 7]);
                *reinterpret_cast<uint4 *>(yr + nbase + j) = v;
              }
            }
          } else {
#pragma unroll
            for (int j = 0; j < C::kCPT; ++j)
              if (nbase + j < args.N) {
                __nv_bfloat16 h = __float2bfloat16_rn(acc[j]);
                yr[nbase + j] = *reinterpret_cast<uint16_t *>(&h);
              }
          }
        }
      } else {
        // swap: thread holds weight row n = d_row, tokens col0 + [0, kCPT)
        const int n = d_row;
        const bool n_ok = n < args.N;
        const float bv = (bias && n_ok)
                             ? bf16_bits_to_float(reinterpret_cast<const uint16_t *>(bias)[n])
                             : 0.0f;
        if (shape.splits == 1) {
          if (n_ok) {
#pragma unroll
            for (int j = 0; j < C::kCPT; ++j) {
              const int m = col0 + j;
              if (m < args.M) {
                __nv_bfloat16 h = __float2bfloat16_rn(acc[j] + bv);
                y[static_cast<int64_t>(m) * args.N + n] = *reinterpret_cast<uint16_t *>(&h);
              }
            }
          }
        } else {
          // split-K: publish FP32 partials, the last CTA of the tile reduces them
          float *part = args.partials;
          if (n_ok) {
#pragma unroll
            for (int j = 0; j < C::kCPT; ++j) {
              const int m = col0 + j;
              if (m < args.M)
                __stcg(part + (static_cast<int64_t>(w.split) * args.M + m) * args.N + n, acc[j]);
            }
          }
          __threadfence();
          named_bar_sync(2, C::kEpiThreads);
          if (et == 0) {
            const uint32_t prev = atomicAdd(args.counters + w.tile, 1u);
            bars->is_last = (prev == static_cast<uint32_t>(shape.splits - 1)) ? 1u : 0u;
          }
          named_bar_sync(2, C::kEpiThreads);
          if (bars->is_last) {
            __threadfence();
            if (n_ok) {
#pragma unroll
              for (int j = 0; j < C::kCPT; ++j) {
                const int m = col0 + j;
                if (m < args.M) {
                  float sum = 0.0f;
                  for (int sp = 0; sp < shape.splits; ++sp)
                    sum += (sp == w.split)
                               ? acc[j]
                               : __ldcg(part + (static_cast<int64_t>(sp) * args.M + m) * args.N + n);
                  __nv_bfloat16 h = __float2bfloat16_rn(sum + bv);
                  y[static_cast<int64_t>(m) * args.N + n] = *reinterpret_cast<uint16_t *>(&h);
                }
              }
            }
            if (et == 0) args.counters[w.tile] = 0u;  // ready for the next call
          }
          named_bar_sync(2, C::kEpiThreads);
        }
      }
    }
    if (!ok && et == 0) record_timeout(args);
  }

  // ------------------------------------------------------------ teardown
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, C::kTmemCols);
  }
}

template <int MODE, bool SWAP, int BN, int STAGES, int EPI_WARPS>
cudaError_t run(const GemmArgs &a, const void *q_act, const void *w, const LaunchShape &sh,
                int grid, cudaStream_t st, int *status) {
  using C = Cfg<MODE, SWAP, BN, STAGES, EPI_WARPS>;
  CUtensorMap ta, tb;
  const void *a_ptr = SWAP ? w : q_act;
  const void *b_ptr = SWAP ? q_act : w;
  const int64_t a_rows = SWAP ? a.N : a.M;
  const int64_t b_rows = SWAP ? a.M : a.N;
  if (!make_kmajor_map(&ta, a_ptr, a_rows, a.K, kBM) ||
      !make_kmajor_map(&tb, b_ptr, b_rows, a.K, BN)) {
    *status = 4;  // FP8BQ_ERR_UNSUPPORTED: tensor map rejected
    return cudaSuccess;
  }
  const size_t smem = C::kFixedSmem + static_cast<size_t>(sh.sx_stage) * sizeof(float);
  auto kern = fp8_gemm_kernel<MODE, SWAP, BN, STAGES, EPI_WARPS>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  kern<<<grid, C::kThreads, smem, st>>>(ta, tb, a, sh);
  return cudaGetLastError();
}

}  // namespace
}  // namespace fp8bq
