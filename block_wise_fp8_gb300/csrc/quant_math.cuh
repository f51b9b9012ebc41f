// quant_math.cuh -- exact quantiser arithmetic shared by the activation
// quantisers and the fused residual-add + RMSNorm + quantisation kernel:
// scales s = amax / 448 from a table, E4M3 codes of RN(x / s) from an
// FMA-corrected quotient, BF16 unpacking and clamping.  Every result equals
// the one from IEEE binary32 divisions ("SGLang 源码完全拆解(十九)", §从浮点到
// FP8 的基本公式; "GLM-5.3 推理全链路(十七)", §第1站, s_g = max|x|/448,
// q = round(x/s_g)).
#pragma once
#include <cuda_fp8.h>

#include <cstdint>

namespace fp8bq {
namespace {

constexpr float kFloor = 1e-10f;  // amax floor (the pages' E8M0 rule; avoids 0/0)

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__device__ __forceinline__ void unpack16(const uint4 (&v)[2], float (&f)[16]) {
  const uint32_t w[8] = {v[0].x, v[0].y, v[0].z, v[0].w, v[1].x, v[1].y, v[1].z, v[1].w};
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    f[2 * i] = bf16_lo(w[i]);
    f[2 * i + 1] = bf16_hi(w[i]);
  }
}

// Prefetch the cache line holding `p` into L2 (no data returned).
__device__ __forceinline__ void prefetch_l2(const void *p) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

__device__ __forceinline__ uint4 ld_stream(const void *p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

__device__ __forceinline__ float amax16(const float (&f)[16]) {
  float m = 0.0f;
#pragma unroll
  for (int i = 0; i < 16; ++i) m = fmaxf(m, fabsf(f[i]));
  return m;
}


// 16 binary32 values -> 16 E4M3 codes (RNE, saturating), packed little-endian.
__device__ __forceinline__ uint4 to_e4m3x16(const float (&t)[16]) {
  uint32_t w[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t lo = __nv_cvt_float2_to_fp8x2(make_float2(t[4 * i], t[4 * i + 1]),
                                                 __NV_SATFINITE, __NV_E4M3);
    const uint32_t hi = __nv_cvt_float2_to_fp8x2(make_float2(t[4 * i + 2], t[4 * i + 3]),
                                                 __NV_SATFINITE, __NV_E4M3);
    w[i] = (lo & 0xFFFFu) | (hi << 16);
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}

// Group scales from a table.  The group amax is a BF16 value m * 2^k with an
// 8-bit significand m in [1, 2) (128 possibilities), and 448 = 7 * 2^6, so
// RN(amax / 448) = RN(m / 448) * 2^k and RN(1 / s) = RN(1 / RN(m / 448)) * 2^-k
// exactly whenever every value involved is a binary32 normal number, which
// holds for amax >= 1e-10.  Each CTA fills the table for the 128 significands
// with IEEE divisions once; a group then costs one shared-memory load and two
// exponent additions instead of two correctly rounded divisions.  Entry m holds
// {s, RN(1/s)} for amax = 1 + m/128.
struct ScaleTable {
  float2 e[128];
  float2 floor_entry;  // amax below the 1e-10 floor
};

__device__ __forceinline__ void fill_scale_table(ScaleTable &t) {
  for (int m = threadIdx.x; m <= 128; m += blockDim.x) {
    const float a = m < 128 ? 1.0f + static_cast<float>(m) * 0.0078125f : kFloor;
    const float sv = __fdiv_rn(a, 448.0f);
    const float2 v = make_float2(sv, __frcp_rn(sv));
    if (m < 128) t.e[m] = v;
    else t.floor_entry = v;
  }
}

// {s, RN(1/s)} for a group with maximum magnitude amax (a BF16 value).
__device__ __forceinline__ float2 scale_of(const ScaleTable &t, float amax) {
  if (!(amax >= kFloor)) return t.floor_entry;
  const uint32_t b = __float_as_uint(amax);
  const float2 v = t.e[(b >> 16) & 0x7Fu];
  const int k = static_cast<int>((b >> 23) & 0xFFu) - 127;  // amax = (1 + m/128) * 2^k
  return make_float2(__uint_as_float(__float_as_uint(v.x) + (static_cast<uint32_t>(k) << 23)),
                     __uint_as_float(__float_as_uint(v.y) - (static_cast<uint32_t>(k) << 23)));
}

// E4M3 codes of RN(x / s) for 2 NW BF16 values x (NW packed pairs w, the same
// values unpacked in f), without a division: with r = RN(1/s), q0 = RN(x r)
// and q1 = RN(q0 + RN(x - s q0) r) (FMAs, two values per instruction), and
// with CORRECTIONS = 2 once more from q1.  By Markstein's theorem the corrected
// quotient is RN(x / s) once the previous one is within an ulp; checked with
// exact rational arithmetic for one correction over every pair of BF16
// significand and group-scale significand (s = RN(m/448)), and for both forms
// on random scales.  Where the remainder underflows the quotient lies far
// below the smallest E4M3 value and encodes to zero either way.  The FMA form
// turns x = -0 into +0, so the codes take the sign bits of x (which every
// nonzero quotient shares).  out receives NW / 2 words of four codes.
template <int CORRECTIONS, int NW>
__device__ __forceinline__ void quant_words(const uint32_t (&w)[NW], const float (&f)[2 * NW],
                                            float s, float r, uint32_t (&out)[NW / 2]) {
  const float2 r2 = make_float2(r, r), ns2 = make_float2(-s, -s);
#pragma unroll
  for (int i = 0; i < NW / 2; ++i) {
    uint32_t half[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const float2 x = make_float2(f[4 * i + 2 * h], f[4 * i + 2 * h + 1]);
      float2 q = __fmul2_rn(x, r2);
#pragma unroll
      for (int c = 0; c < CORRECTIONS; ++c) q = __ffma2_rn(__ffma2_rn(ns2, q, x), r2, q);
      half[h] = __nv_cvt_float2_to_fp8x2(q, __NV_SATFINITE, __NV_E4M3);
    }
    const uint32_t codes = (half[0] & 0xFFFFu) | (half[1] << 16);
    out[i] = codes | (__byte_perm(w[2 * i], w[2 * i + 1], 0x7531) & 0x80808080u);
  }
}

// quant_words over 16 values held as two 16-byte words.
template <int CORRECTIONS>
__device__ __forceinline__ uint4 quant16(const uint4 (&v)[2], const float (&f)[16], float s,
                                        float r) {
  const uint32_t w[8] = {v[0].x, v[0].y, v[0].z, v[0].w, v[1].x, v[1].y, v[1].z, v[1].w};
  uint32_t out[4];
  quant_words<CORRECTIONS, 8>(w, f, s, r, out);
  return make_uint4(out[0], out[1], out[2], out[3]);
}

// Each BF16 pair of the four words clamped to [lo, hi] (BF16 pairs).
__device__ __forceinline__ void clamp_bf16x2(uint4 &v, uint32_t lo, uint32_t hi) {
  uint32_t *w = reinterpret_cast<uint32_t *>(&v);
#pragma unroll
  for (int i = 0; i < 4; ++i)
    asm("{\n\t.reg .b32 t;\n\tmax.bf16x2 t, %1, %2;\n\tmin.bf16x2 %0, t, %3;\n\t}"
        : "=r"(w[i])
        : "r"(w[i]), "r"(lo), "r"(hi));
}

// A static per-tensor scale prepared for quant_words<2>.  x / s may overflow
// binary32 (x is not bounded by the scale), and the FMA form would turn the
// infinity into NaN.  Every |x| >= 448 s encodes to the saturated 448 anyway,
// so inputs are clamped to +-L with L = 464 s rounded up to a BF16 value:
// values within L are unchanged, values beyond give quotients in [464, 469],
// which saturate to the same code.  A scale below 2^-100 would make L
// underflow; such scales divide instead (`divide`, uniform over a launch).
struct StaticScale {
  float s, r;
  bool divide;
  uint32_t lim2, nlim2;  // +L and -L as BF16 pairs
};

__device__ __forceinline__ StaticScale static_scale(float sv) {
  StaticScale c;
  c.s = sv;
  c.r = __frcp_rn(sv);
  c.divide = !(sv >= 0x1p-100f);
  uint32_t lim = __float_as_uint(__fmul_ru(sv, 464.0f));
  lim = (lim & 0xFFFFu) ? (lim + 0x10000u) & 0xFFFF0000u : lim;
  c.lim2 = (lim >> 16) | (lim & 0xFFFF0000u);
  c.nlim2 = c.lim2 | 0x80008000u;
  return c;
}

}  // namespace
}  // namespace fp8bq
