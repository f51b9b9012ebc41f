// quant.cu -- activation / weight quantisation kernels (HBM-streaming).
//
// Every kernel reads BF16 with 16-byte vector loads, reduces |x| with warp
// shuffles inside its group, and converts with the hardware's saturating
// round-to-nearest-even FP32 -> E4M3 conversion.  Scales and quotients are
// IEEE binary32 divisions (__fdiv_rn), so codes and scales are bit-identical
// to the definitions on the pages ("SGLang 源码完全拆解(十九)", §从浮点到 FP8 的
// 基本公式; "GLM-5.3 推理全链路(十七)", §第1站, s_g = max|x|/448, q = round(x/s_g)).
#include <cuda_fp8.h>

#include <climits>

#include "common.cuh"
#include "ptx.cuh"
#include "quant_math.cuh"

namespace fp8bq {
namespace {

constexpr int kThreads = 256;

// ---------------------------------------------------------------- group-128 activation quant
// 8 threads per 128-channel group, 16 channels (32 bytes) per thread; a
// partial last group masks whole 16-channel chunks (K % 16 == 0).  The grid is
// persistent: each warp takes 4 consecutive groups per step and walks the
// groups with the grid's stride, loading its next chunk before converting the
// current one, so two chunks per thread are in flight.
// UE8M0: the scale is the power of two 2^e, e = ceil(log2(max(amax,1e-10)/448))
// (the MXFP8 rule on a 128-channel group, "SGLang 源码完全拆解(十九)", §分块
// GEMM 的后端分派, act_scale_ue8m0), stored as the code e + 127 in uint8 s[M][G].
template <bool UE8M0>
__global__ void __launch_bounds__(kThreads) quant_group128_kernel(
    const uint8_t *__restrict__ x, int64_t M, int K, int64_t ldx_bytes, int G,
    uint8_t *__restrict__ q, void *__restrict__ s_out, int s_layout, int64_t lds) {
  float *s = static_cast<float *>(s_out);
  __shared__ ScaleTable table;
  griddep_launch_dependents();
  const int lane = threadIdx.x & 31, sub = lane & 7;
  const int64_t total = M * G;
  const int64_t step = static_cast<int64_t>(gridDim.x) * (kThreads / 8);  // groups per step
  const int64_t warp_g0 = (static_cast<int64_t>(blockIdx.x) * (kThreads / 32) + (threadIdx.x >> 5)) * 4;
  const int64_t gid = warp_g0 + (lane >> 3);
  // (row, group) of this thread's group, advanced by (drow, dg) per step
  int64_t row = gid / G;
  int g = static_cast<int>(gid - row * G);
  // Before the preceding kernel has completed, only an L2 prefetch of this
  // thread's first chunk: L2 is the point of coherence, so a later load still
  // sees whatever that kernel writes there
  if (row < M && g * 128 + sub * 16 < K)
    prefetch_l2(x + row * ldx_bytes + static_cast<int64_t>(g * 128 + sub * 16) * 2);
  fill_scale_table(table);
  __syncthreads();
  griddep_wait();
  const int64_t drow = step / G;
  const int dg = static_cast<int>(step - drow * G);
  auto load = [&](int64_t r, int gg, uint4 (&v)[2]) {
    const int k = gg * 128 + sub * 16;
    if (r < M && k < K) {
      const uint8_t *p = x + r * ldx_bytes + static_cast<int64_t>(k) * 2;
      v[0] = ld_stream(p);
      v[1] = ld_stream(p + 16);
    } else {
      v[0] = v[1] = make_uint4(0, 0, 0, 0);
    }
  };
  uint4 cur[2];
  load(row, g, cur);
  for (int64_t base = warp_g0; base < total; base += step) {
    int64_t row_n = row + drow;
    int g_n = g + dg;
    if (g_n >= G) {
      g_n -= G;
      ++row_n;
    }
    uint4 nxt[2];
    load(row_n, g_n, nxt);
    float f[16];
    unpack16(cur, f);
    float amax = amax16(f);
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 4));
    const float2 sc = scale_of(table, amax);
    const float sg = sc.x;
    uint4 out;
    uint32_t u = 0u;
    if (UE8M0) {
      const uint32_t rb = __float_as_uint(sg);                        // RN(max(amax,1e-10)/448)
      u = (rb >> 23) + ((rb & 0x7FFFFFu) != 0u ? 1u : 0u);            // e + 127
      const float inv = __uint_as_float((254u - u) << 23);            // 2^-e, exact
      float t[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) t[i] = __fmul_rn(f[i], inv);
      out = to_e4m3x16(t);
    } else {
      out = quant16<1>(cur, f, sg, sc.y);
    }
    const int k = g * 128 + sub * 16;
    if (row < M) {
      if (k < K) *reinterpret_cast<uint4 *>(q + row * K + k) = out;
      if (sub == 0) {
        if (UE8M0) static_cast<uint8_t *>(s_out)[row * G + g] = static_cast<uint8_t>(u);
        else if (s_layout == 0) s[row * lds + g] = sg;
        else s[static_cast<int64_t>(g) * lds + row] = sg;
      }
    }
    cur[0] = nxt[0];
    cur[1] = nxt[1];
    row = row_n;
    g = g_n;
  }
}

// ---------------------------------------------------------------- MXFP8 [1,32] quant
// 2 threads per 32-channel group (16 per warp step), persistent like the
// group-128 kernel.  e = ceil(log2(r)), r = max(amax,1e-10)/448 read from r's
// bits (r is a positive normal float): biased exponent plus one unless the
// mantissa is zero.  The UE8M0 code is e + 127.
__global__ void __launch_bounds__(kThreads) quant_mx_kernel(const uint8_t *__restrict__ x,
                                                            int64_t M, int K,
                                                            int64_t ldx_bytes,
                                                            uint8_t *__restrict__ q,
                                                            uint8_t *__restrict__ s) {
  __shared__ ScaleTable table;
  griddep_launch_dependents();
  const int G = K / 32;
  const int lane = threadIdx.x & 31, sub = lane & 1;
  const int64_t total = M * G;
  const int64_t step = static_cast<int64_t>(gridDim.x) * (kThreads / 2);
  const int64_t warp_g0 = (static_cast<int64_t>(blockIdx.x) * (kThreads / 32) + (threadIdx.x >> 5)) * 16;
  const int64_t gid = warp_g0 + (lane >> 1);
  int64_t row = gid / G;
  int g = static_cast<int>(gid - row * G);
  // before the preceding kernel completes: an L2 prefetch of the first chunk
  if (row < M) prefetch_l2(x + row * ldx_bytes + static_cast<int64_t>(g * 32 + sub * 16) * 2);
  fill_scale_table(table);
  __syncthreads();
  griddep_wait();
  const int64_t drow = step / G;
  const int dg = static_cast<int>(step - drow * G);
  auto load = [&](int64_t r, int gg, uint4 (&v)[2]) {
    if (r < M) {
      const uint8_t *p = x + r * ldx_bytes + static_cast<int64_t>(gg * 32 + sub * 16) * 2;
      v[0] = ld_stream(p);
      v[1] = ld_stream(p + 16);
    } else {
      v[0] = v[1] = make_uint4(0, 0, 0, 0);
    }
  };
  uint4 cur[2];
  load(row, g, cur);
  for (int64_t base = warp_g0; base < total; base += step) {
    int64_t row_n = row + drow;
    int g_n = g + dg;
    if (g_n >= G) {
      g_n -= G;
      ++row_n;
    }
    uint4 nxt[2];
    load(row_n, g_n, nxt);
    float f[16];
    unpack16(cur, f);
    float amax = amax16(f);
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
    const uint32_t rb = __float_as_uint(scale_of(table, amax).x);  // RN(max(amax,1e-10)/448)
    const uint32_t u = (rb >> 23) + ((rb & 0x7FFFFFu) != 0u ? 1u : 0u);  // e + 127
    const float inv = __uint_as_float((254u - u) << 23);                 // 2^-e, exact
    float t[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) t[i] = __fmul_rn(f[i], inv);
    const uint4 out = to_e4m3x16(t);
    if (row < M) {
      *reinterpret_cast<uint4 *>(q + row * K + g * 32 + sub * 16) = out;
      if (sub == 0) s[row * G + g] = static_cast<uint8_t>(u);
    }
    cur[0] = nxt[0];
    cur[1] = nxt[1];
    row = row_n;
    g = g_n;
  }
}

// ---------------------------------------------------------------- per-token (per-row) quant
// One scale per row, the group rule with the group spanning the row ("SGLang
// 源码完全拆解(十九)", §激活量化的三种选择: sglang_per_token_quant_fp8, one scale per
// token; §装载后的三个分支: per_token_group_quant_fp8 with group_size = K).
// One CTA per row, persistent over rows: pass 1 reduces max|x| over the row,
// pass 2 re-reads it (an L1 hit) and converts with the row's scale, 16
// channels (two 16-byte words) per thread per step.  The warp maxima are
// double-buffered by row parity, so one barrier per row suffices.
__global__ void __launch_bounds__(kThreads) quant_token_kernel(const uint8_t *__restrict__ x,
                                                               int64_t M, int K,
                                                               int64_t ldx_bytes,
                                                               uint8_t *__restrict__ q,
                                                               float *__restrict__ s) {
  __shared__ ScaleTable table;
  __shared__ float red[2][kThreads / 32];
  griddep_launch_dependents();
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const int C = K / 16;
  // before the preceding kernel completes: an L2 prefetch of the first row
  // (one 128-byte line per four 32-byte chunks)
  if (blockIdx.x < M)
    for (int c = 4 * t; c < C; c += 4 * kThreads) prefetch_l2(x + blockIdx.x * ldx_bytes + c * 32);
  fill_scale_table(table);
  __syncthreads();
  griddep_wait();
  int par = 0;
  for (int64_t row = blockIdx.x; row < M; row += gridDim.x, par ^= 1) {
    const uint8_t *xr = x + row * ldx_bytes;
    float amax = 0.0f;
    for (int c = t; c < C; c += kThreads) {
      uint4 v[2];
      v[0] = __ldg(reinterpret_cast<const uint4 *>(xr + c * 32));
      v[1] = __ldg(reinterpret_cast<const uint4 *>(xr + c * 32 + 16));
      float f[16];
      unpack16(v, f);
      amax = fmaxf(amax, amax16(f));
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
    if (lane == 0) red[par][warp] = amax;
    __syncthreads();
#pragma unroll
    for (int i = 0; i < kThreads / 32; ++i) amax = fmaxf(amax, red[par][i]);
    const float2 sc = scale_of(table, amax);
    for (int c = t; c < C; c += kThreads) {
      uint4 v[2];
      v[0] = __ldg(reinterpret_cast<const uint4 *>(xr + c * 32));
      v[1] = __ldg(reinterpret_cast<const uint4 *>(xr + c * 32 + 16));
      float f[16];
      unpack16(v, f);
      *reinterpret_cast<uint4 *>(q + row * K + c * 16) = quant16<1>(v, f, sc.x, sc.y);
    }
    if (t == 0) s[row] = sc.x;
  }
}

// ---------------------------------------------------------------- static per-tensor quant
// One thread per 16-channel chunk, persistent grid, next chunk loaded first.
__global__ void __launch_bounds__(kThreads) quant_static_kernel(const uint8_t *__restrict__ x,
                                                                int64_t M, int K,
                                                                int64_t ldx_bytes,
                                                                const float *__restrict__ s_ptr,
                                                                uint8_t *__restrict__ q) {
  griddep_launch_dependents();
  const int C = K / 16;
  const int64_t total = M * C;
  const int64_t step = static_cast<int64_t>(gridDim.x) * kThreads;
  const int64_t cid0 = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x;
  int64_t row = cid0 / C;
  int c = static_cast<int>(cid0 - row * C);
  // before the preceding kernel completes: an L2 prefetch of the first chunk
  // (the scale, which that kernel may write, is read after the wait)
  if (row < M) prefetch_l2(x + row * ldx_bytes + static_cast<int64_t>(c) * 32);
  griddep_wait();
  const int64_t drow = step / C;
  const int dc = static_cast<int>(step - drow * C);
  const StaticScale sc = static_scale(__ldg(s_ptr));
  const float sv = sc.s, rv = sc.r;
  const bool divide = sc.divide;
  const uint32_t lim2 = sc.lim2, nlim2 = sc.nlim2;
  auto load = [&](int64_t r, int cc, uint4 (&v)[2]) {
    if (r < M) {
      const uint8_t *p = x + r * ldx_bytes + static_cast<int64_t>(cc) * 32;
      v[0] = ld_stream(p);
      v[1] = ld_stream(p + 16);
    }
  };
  uint4 cur[2];
  load(row, c, cur);
  for (int64_t cid = cid0; cid < total; cid += step) {
    int64_t row_n = row + drow;
    int c_n = c + dc;
    if (c_n >= C) {
      c_n -= C;
      ++row_n;
    }
    uint4 nxt[2];
    load(row_n, c_n, nxt);
    uint4 clamped[2] = {cur[0], cur[1]};
    if (!divide) {
      clamp_bf16x2(clamped[0], nlim2, lim2);
      clamp_bf16x2(clamped[1], nlim2, lim2);
    }
    float f[16];
    unpack16(clamped, f);
    uint4 out;
    if (divide) {
      float t[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) t[i] = __fdiv_rn(f[i], sv);
      out = to_e4m3x16(t);
    } else {
      out = quant16<2>(cur, f, sv, rv);
    }
    *reinterpret_cast<uint4 *>(q + row * K + static_cast<int64_t>(c) * 16) = out;
    cur[0] = nxt[0];
    cur[1] = nxt[1];
    row = row_n;
    c = c_n;
  }
}

// ---------------------------------------------------------------- 128x128 weight blocks
// One CTA per block; thread t covers row t/2 of the block and 64 channels.
__global__ void __launch_bounds__(kThreads) quant_weight_block_kernel(
    const uint8_t *__restrict__ w, int N, int K, int64_t ldw_bytes, uint8_t *__restrict__ q,
    float *__restrict__ s, int KB) {
  __shared__ float red[kThreads / 32];
  griddep_launch_dependents();
  griddep_wait();
  const int nb = blockIdx.y, kb = blockIdx.x;
  const int r = nb * 128 + (threadIdx.x >> 1);
  const int kbase = kb * 128 + (threadIdx.x & 1) * 64;
  float f[4][16];
  bool ok[4];
  float amax = 0.0f;
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const int k = kbase + c * 16;
    ok[c] = r < N && k < K;
    uint4 v[2] = {make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0)};
    if (ok[c]) {
      const uint8_t *p = w + static_cast<int64_t>(r) * ldw_bytes + static_cast<int64_t>(k) * 2;
      v[0] = ld_stream(p);
      v[1] = ld_stream(p + 16);
    }
    unpack16(v, f[c]);
    amax = fmaxf(amax, amax16(f[c]));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = amax;
  __syncthreads();
  amax = red[0];
#pragma unroll
  for (int i = 1; i < kThreads / 32; ++i) amax = fmaxf(amax, red[i]);
  const float sb = __fdiv_rn(fmaxf(amax, kFloor), 448.0f);
  if (threadIdx.x == 0) s[nb * KB + kb] = sb;
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    float t[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) t[i] = __fdiv_rn(f[c][i], sb);
    const uint4 out = to_e4m3x16(t);
    if (ok[c])
      *reinterpret_cast<uint4 *>(q + static_cast<int64_t>(r) * K + kbase + c * 16) = out;
  }
}

// ---------------------------------------------------------------- per-tensor absmax scale
// amax over the matrix via atomicMax on the bit patterns of non-negative floats
// (their integer order equals their numeric order), then s = max(amax,1e-10)/448.
__global__ void __launch_bounds__(kThreads) absmax_kernel(const uint8_t *__restrict__ x,
                                                          int64_t rows, int K,
                                                          int64_t ldx_bytes,
                                                          uint32_t *__restrict__ acc) {
  griddep_launch_dependents();
  griddep_wait();
  const int C = K / 16;
  const int64_t total = rows * C;
  float m = 0.0f;
  for (int64_t cid = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x; cid < total;
       cid += static_cast<int64_t>(gridDim.x) * kThreads) {
    const int64_t row = cid / C;
    const int k = static_cast<int>(cid - row * C) * 16;
    const uint8_t *p = x + row * ldx_bytes + static_cast<int64_t>(k) * 2;
    uint4 v[2] = {ld_stream(p), ld_stream(p + 16)};
    float f[16];
    unpack16(v, f);
    m = fmaxf(m, amax16(f));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  if ((threadIdx.x & 31) == 0) atomicMax(acc, __float_as_uint(m));
}

__global__ void absmax_finalize_kernel(float *s) {
  griddep_launch_dependents();
  griddep_wait();
  const float amax = __uint_as_float(*reinterpret_cast<uint32_t *>(s));
  *s = __fdiv_rn(fmaxf(amax, kFloor), 448.0f);
}

// ---------------------------------------------------------------- FP32 -> UE8M0 weight requant
// One CTA per 128 x 128 block (one-time weight preparation): the FP32 block
// scale s becomes 2^e, e = ceil(log2 s) (the nearest power of two at or above
// s, read from s's bits), and every code is re-encoded from its value,
// q' = RNE_sat(dec(q) * s * 2^-e): the product of a 4-bit and a 24-bit
// significand is exact in binary64, then rounded once to E4M3 ("SGLang 源码完全
// 拆解(十九)", §分块路径的后处理).  q' may
// be q itself (each code is read before it is written, by the same thread).
__global__ void __launch_bounds__(kThreads) requant_ue8m0_kernel(const uint8_t *q, const float *__restrict__ s,
                                                                 int N, int K, int KB, uint8_t *q2,
                                                                 uint8_t *__restrict__ u) {
  griddep_launch_dependents();
  griddep_wait();
  const int kb = blockIdx.x, nb = blockIdx.y;
  const float sv = __ldg(s + static_cast<int64_t>(nb) * KB + kb);
  const uint32_t sb = __float_as_uint(sv);  // a positive normal scale
  const int e = static_cast<int>(sb >> 23) - 127 + ((sb & 0x7FFFFFu) != 0u ? 1 : 0);
  const double m = static_cast<double>(sv) * ldexp(1.0, -e);  // s / 2^e, in (1/2, 1]
  if (threadIdx.x == 0) u[static_cast<int64_t>(nb) * KB + kb] = static_cast<uint8_t>(e + 127);
  const int rows = min(128, N - nb * 128), cols = min(128, K - kb * 128);
  for (int idx = threadIdx.x; idx < rows * cols; idx += blockDim.x) {
    const int r = idx / cols, c = idx - r * cols;
    const int64_t off = static_cast<int64_t>(nb * 128 + r) * K + kb * 128 + c;
    const __half_raw hr = __nv_cvt_fp8_to_halfraw(static_cast<__nv_fp8_storage_t>(q[off]), __NV_E4M3);
    const double v = static_cast<double>(__half2float(__half(hr))) * m;
    q2[off] = static_cast<uint8_t>(__nv_cvt_double_to_fp8(v, __NV_SATFINITE, __NV_E4M3));
  }
}

// Scale check: per entry, the class of an unusable dequantisation multiplier
// (the unloaded sentinel -FLT_MAX, NaN or infinity, any other value <= 0);
// counts added into out[0..2], the smallest bad index min-ed into out[3].
__global__ void __launch_bounds__(kThreads) check_scales_kernel(const float *__restrict__ s,
                                                                 int64_t n,
                                                                 unsigned long long *out) {
  griddep_launch_dependents();
  griddep_wait();
  unsigned long long c[3] = {0, 0, 0};
  long long first = LLONG_MAX;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
       i += stride) {
    const float v = s[i];
    const uint32_t b = __float_as_uint(v);
    const bool sentinel = b == 0xff7fffffu;
    const bool nonfinite = (b & 0x7f800000u) == 0x7f800000u;
    const bool nonpositive = !sentinel && !nonfinite && !(v > 0.0f);
    c[0] += sentinel;
    c[1] += nonfinite;
    c[2] += nonpositive;
    if ((sentinel || nonfinite || nonpositive) && i < first) first = i;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
#pragma unroll
    for (int k = 0; k < 3; ++k) c[k] += __shfl_xor_sync(0xffffffffu, c[k], o);
    first = min(first, __shfl_xor_sync(0xffffffffu, first, o));
  }
  if ((threadIdx.x & 31) == 0) {
#pragma unroll
    for (int k = 0; k < 3; ++k)
      if (c[k]) atomicAdd(out + k, c[k]);
    if (first != LLONG_MAX) atomicMin(reinterpret_cast<long long *>(out + 3), first);
  }
}

inline unsigned blocks_for(int64_t work, int per_block) {
  return static_cast<unsigned>((work + per_block - 1) / per_block);
}

}  // namespace

// Persistent grids: enough CTAs for the work, at most as many as fit on the
// device at once (the kernel's occupancy, queried once per kernel).
template <auto KERN>
unsigned persistent_grid(int64_t work, int per_block, int num_sms) {
  // per kernel (the template argument is the kernel itself, not its type)
  static int per_sm = [] {
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, KERN, kThreads, 0) != cudaSuccess ||
        n < 1)
      n = 1;
    return n;
  }();
  const int64_t need = (work + per_block - 1) / per_block;
  const int64_t cap = static_cast<int64_t>(num_sms) * per_sm;
  return static_cast<unsigned>(need < 1 ? 1 : need < cap ? need : cap);
}

void launch_quant_group(const void *x, int64_t M, int64_t K, int64_t ldx, void *q, float *s,
                        int s_layout, int num_sms, cudaStream_t st) {
  const int G = static_cast<int>((K + 127) / 128);
  const int64_t lds = s_layout == 0 ? G : ((M + 3) / 4) * 4;
  launch_pdl(quant_group128_kernel<false>,
             persistent_grid<quant_group128_kernel<false>>(M * G, kThreads / 8, num_sms), kThreads, 0,
             st, static_cast<const uint8_t *>(x), M, static_cast<int>(K), ldx * 2, G,
             static_cast<uint8_t *>(q), static_cast<void *>(s), s_layout, lds);
}

void launch_quant_group_ue8m0(const void *x, int64_t M, int64_t K, int64_t ldx, void *q,
                              uint8_t *u, int num_sms, cudaStream_t st) {
  const int G = static_cast<int>((K + 127) / 128);
  launch_pdl(quant_group128_kernel<true>,
             persistent_grid<quant_group128_kernel<true>>(M * G, kThreads / 8, num_sms), kThreads, 0,
             st, static_cast<const uint8_t *>(x), M, static_cast<int>(K), ldx * 2, G,
             static_cast<uint8_t *>(q), static_cast<void *>(u), 0, static_cast<int64_t>(G));
}

void launch_quant_mx(const void *x, int64_t M, int64_t K, int64_t ldx, void *q, uint8_t *s,
                     int num_sms, cudaStream_t st) {
  launch_pdl(quant_mx_kernel, persistent_grid<quant_mx_kernel>(M * (K / 32), kThreads / 2, num_sms), kThreads,
             0, st, static_cast<const uint8_t *>(x), M, static_cast<int>(K), ldx * 2,
             static_cast<uint8_t *>(q), s);
}

void launch_quant_token(const void *x, int64_t M, int64_t K, int64_t ldx, void *q, float *s,
                        int num_sms, cudaStream_t st) {
  launch_pdl(quant_token_kernel, persistent_grid<quant_token_kernel>(M, 1, num_sms), kThreads, 0, st,
             static_cast<const uint8_t *>(x), M, static_cast<int>(K), ldx * 2,
             static_cast<uint8_t *>(q), s);
}

void launch_quant_static(const void *x, int64_t M, int64_t K, int64_t ldx, const float *s,
                         void *q, int num_sms, cudaStream_t st) {
  launch_pdl(quant_static_kernel, persistent_grid<quant_static_kernel>(M * (K / 16), kThreads, num_sms), kThreads, 0,
             st, static_cast<const uint8_t *>(x), M, static_cast<int>(K), ldx * 2, s,
             static_cast<uint8_t *>(q));
}

void launch_quant_weight_block(const void *w, int64_t N, int64_t K, int64_t ldw, void *q,
                               float *s, cudaStream_t st) {
  const int KB = static_cast<int>((K + 127) / 128);
  const int NB = static_cast<int>((N + 127) / 128);
  launch_pdl(quant_weight_block_kernel, dim3(KB, NB), kThreads, 0, st,
             static_cast<const uint8_t *>(w), static_cast<int>(N), static_cast<int>(K), ldw * 2,
             static_cast<uint8_t *>(q), s, KB);
}

void launch_requant_ue8m0(const void *q, const float *s, int64_t N, int64_t K, void *q2, uint8_t *u,
                          cudaStream_t st) {
  const int KB = static_cast<int>((K + 127) / 128);
  const int NB = static_cast<int>((N + 127) / 128);
  launch_pdl(requant_ue8m0_kernel, dim3(KB, NB), kThreads, 0, st, static_cast<const uint8_t *>(q), s,
             static_cast<int>(N), static_cast<int>(K), KB, static_cast<uint8_t *>(q2), u);
}

// The binary32 -> E4M3 conversion of every quantiser (the paired, saturating,
// round-to-nearest-even conversion of quant_words and to_e4m3x16) applied to
// consecutive bit patterns: codes[i] = E4M3(bits first + i).  Each thread
// converts 8 patterns, two per conversion, and stores them as one 8-byte word.
__global__ void __launch_bounds__(kThreads) e4m3_bits_kernel(uint32_t first, int64_t n,
                                                             uint8_t *__restrict__ codes) {
  griddep_launch_dependents();
  griddep_wait();
  const int64_t groups = (n + 7) / 8;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t g = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; g < groups;
       g += stride) {
    const int64_t i0 = g * 8;
    uint32_t w[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      uint32_t word = 0;
#pragma unroll
      for (int p = 0; p < 2; ++p) {
        const uint32_t b = first + static_cast<uint32_t>(i0 + 4 * h + 2 * p);
        const float2 v = make_float2(__uint_as_float(b), __uint_as_float(b + 1u));
        const uint32_t c = __nv_cvt_float2_to_fp8x2(v, __NV_SATFINITE, __NV_E4M3);
        word |= (c & 0xFFFFu) << (16 * p);
      }
      w[h] = word;
    }
    if (i0 + 8 <= n) {
      *reinterpret_cast<uint2 *>(codes + i0) = make_uint2(w[0], w[1]);
    } else {
      for (int j = 0; i0 + j < n; ++j) codes[i0 + j] = static_cast<uint8_t>(w[j / 4] >> (8 * (j % 4)));
    }
  }
}

void launch_e4m3_bits(uint32_t first, int64_t n, uint8_t *codes, int num_sms, cudaStream_t st) {
  unsigned grid = blocks_for((n + 7) / 8, kThreads);
  const unsigned cap = static_cast<unsigned>(num_sms) * 8u;
  if (grid > cap) grid = cap;
  if (grid == 0) grid = 1;
  launch_pdl(e4m3_bits_kernel, grid, kThreads, 0, st, first, n, codes);
}

void launch_check_scales(const float *s, int64_t n, unsigned long long *out, int num_sms,
                         cudaStream_t st) {
  // counts to 0, first index to 0x7f7f7f7f7f7f7f7f (above any index)
  cudaMemsetAsync(out, 0, 3 * sizeof(unsigned long long), st);
  cudaMemsetAsync(out + 3, 0x7f, sizeof(unsigned long long), st);
  unsigned grid = blocks_for(n, kThreads * 4);
  const unsigned cap = static_cast<unsigned>(num_sms) * 4u;
  if (grid > cap) grid = cap;
  if (grid == 0) grid = 1;
  launch_pdl(check_scales_kernel, grid, kThreads, 0, st, s, n, out);
}

void launch_absmax_scale(const void *x, int64_t rows, int64_t K, int64_t ldx, float *s,
                         int num_sms, cudaStream_t st) {
  cudaMemsetAsync(s, 0, sizeof(float), st);
  const int64_t work = rows * (K / 16);
  unsigned grid = blocks_for(work, kThreads);
  const unsigned cap = static_cast<unsigned>(num_sms) * 8u;
  if (grid > cap) grid = cap;
  if (grid == 0) grid = 1;
  launch_pdl(absmax_kernel, grid, kThreads, 0, st, static_cast<const uint8_t *>(x), rows,
             static_cast<int>(K), ldx * 2, reinterpret_cast<uint32_t *>(s));
  launch_pdl(absmax_finalize_kernel, 1, 1, 0, st, s);
}

}  // namespace fp8bq
