/*
 * fp8bq_oracle.c -- plain CPU oracle for the block-wise FP8 W8A8 linear.
 *
 * TEST INFRASTRUCTURE ONLY: used by the tests, the smoke check and the CPU
 * baseline of the benchmark, never by the library.  Shares no code with the
 * CUDA path.  Citations: see fp8bq_oracle.h.
 *
 * Readings taken where the pages leave a step open:
 *   - s = amax / 448 and q = x / s are IEEE binary32 divisions.
 *   - amax is floored at 1e-10 (the pages' E8M0 scale rule floors it; the FP32
 *     rule is silent, and an all-zero group would otherwise give 0/0).
 *   - rounding is round-to-nearest-even, saturating to +-448; the sign of zero
 *     is kept.
 *   - the UE8M0 exponent is ceil(log2(max(amax,1e-10)/448)).
 *   - ragged edge groups/blocks use only their valid elements.
 */
#include "fp8bq_oracle.h"

#include <math.h>
#include <pthread.h>
#include <stdlib.h>
#include <string.h>

/* ======================================================================= */
/* Number formats                                                           */
/* ======================================================================= */

/* Round a non-negative binary64 value to the nearest integer, ties to even.
 * All callers pass values whose fractional part is exact in binary64. */
static uint32_t rne_uint(double t) {
  double n = floor(t);
  double d = t - n;
  uint32_t k = (uint32_t)n;
  if (d > 0.5) return k + 1;
  if (d == 0.5) return k + (k & 1u);
  return k;
}

/* E4M3 ("e4m3fn"): 1 sign, 4 exponent (bias 7), 3 mantissa bits; largest
 * finite value 448, smallest normal 2^-6, no infinities, S.1111.111 = NaN
 * ([SGL-19] §三种 scale 的存储形状 "E4M3 ... 最大可表示 448"; [GLM-17] §先把
 * GLM-5.3 的数值常量摆出来).  Encoding rounds to nearest even and clamps to
 * +-448 ([SGL-19] §从浮点到 FP8 的基本公式: q = clamp(round(x/s), -448, 448),
 * round is RNE in real kernels).  Exact in binary64: every step scales by a
 * power of two. */
uint8_t orc_e4m3_encode(double v) {
  if (v != v) return 0x7F;
  uint8_t sign = signbit(v) ? 0x80 : 0x00;
  double a = fabs(v);
  if (a >= 448.0) return sign | 0x7E;
  if (a < 0x1p-6) {
    /* subnormal range: codes 0..7 are multiples of 2^-9; n == 8 is 2^-6, which
     * is exactly the smallest normal code 0x08 */
    uint32_t n = rne_uint(a * 512.0);
    return sign | (uint8_t)n;
  }
  int ex;
  double f = frexp(a, &ex); /* a = f * 2^ex, f in [0.5, 1) */
  int e = ex - 1;           /* a = (2f) * 2^e,  2f in [1, 2) */
  uint32_t n = rne_uint((2.0 * f - 1.0) * 8.0);
  if (n == 8) {
    n = 0;
    e += 1;
  }
  int code = ((e + 7) << 3) | (int)n;
  if (code > 0x7E) code = 0x7E;
  return sign | (uint8_t)code;
}

double orc_e4m3_decode(uint8_t c) {
  int s = c >> 7, E = (c >> 3) & 15, m = c & 7;
  if (E == 15 && m == 7) return NAN;
  double v = (E == 0) ? ldexp((double)m, -9) : ldexp((double)(8 + m), E - 10);
  return s ? -v : v;
}

int32_t orc_e4m3_sig(uint8_t c) {
  int s = c >> 7, E = (c >> 3) & 15, m = c & 7;
  int32_t v = (E == 0) ? m : ((8 + m) << (E - 1));
  return s ? -v : v;
}

/* UE8M0: an 8-bit biased exponent with no mantissa, 2^-127 .. 2^127
 * ([SGL-19] §Triton 分块内核在做什么, the act_scale_ue8m0 paragraph). */
double orc_ue8m0_decode(uint8_t u) {
  if (u == 255) return NAN;
  return ldexp(1.0, (int)u - 127);
}

float orc_bf16_to_f32(uint16_t b) {
  union {
    uint32_t u;
    float f;
  } c;
  c.u = ((uint32_t)b) << 16;
  return c.f;
}

void orc_e4m3_encode_f32_array(const float *v, int64_t n, uint8_t *out) {
  for (int64_t i = 0; i < n; ++i) out[i] = orc_e4m3_encode((double)v[i]);
}

void orc_e4m3_decode_array(const uint8_t *c, int64_t n, double *out) {
  for (int64_t i = 0; i < n; ++i) out[i] = orc_e4m3_decode(c[i]);
}

/* The encoder over consecutive binary32 bit patterns: out[i] = the code of the
 * binary32 value whose bits are first + i (i < n, first + n <= 2^32).  Every
 * binary32 value is exact in binary64, so this is orc_e4m3_encode on each
 * pattern; the threads take contiguous ranges. */
typedef struct {
  uint32_t first;
  int64_t i0, i1;
  uint8_t *out;
} bits_job;

static void *bits_worker(void *p) {
  bits_job *j = (bits_job *)p;
  for (int64_t i = j->i0; i < j->i1; ++i) {
    union {
      uint32_t u;
      float f;
    } c;
    c.u = j->first + (uint32_t)i;
    j->out[i] = orc_e4m3_encode((double)c.f);
  }
  return NULL;
}

void orc_e4m3_encode_bits_range(uint32_t first, int64_t n, uint8_t *out, int nthreads) {
  enum { MAX_THREADS = 256 };
  if (n <= 0) return;
  if (nthreads < 1) nthreads = 1;
  if (nthreads > MAX_THREADS) nthreads = MAX_THREADS;
  pthread_t th[MAX_THREADS];
  int joined[MAX_THREADS];
  bits_job jobs[MAX_THREADS];
  int64_t per = (n + nthreads - 1) / nthreads;
  for (int t = 0; t < nthreads; ++t) {
    jobs[t].first = first;
    jobs[t].out = out;
    jobs[t].i0 = (int64_t)t * per < n ? (int64_t)t * per : n;
    jobs[t].i1 = jobs[t].i0 + per < n ? jobs[t].i0 + per : n;
    joined[t] = pthread_create(&th[t], NULL, bits_worker, &jobs[t]) == 0;
    if (!joined[t]) bits_worker(&jobs[t]); /* no thread available: run inline */
  }
  for (int t = 0; t < nthreads; ++t)
    if (joined[t]) pthread_join(th[t], NULL);
}

/* binary32 amax floored at 1e-10, then the binary32 division amax / 448. */
static float group_scale(float amax) {
  volatile float a = amax < 1e-10f ? 1e-10f : amax;
  volatile float s = a / 448.0f;
  return s;
}

static uint8_t quant_one(float x, float s) {
  volatile float t = x / s; /* binary32 quotient, then RNE to E4M3 */
  return orc_e4m3_encode((double)t);
}

/* ======================================================================= */
/* Quantisers                                                               */
/* ======================================================================= */

/* Per-token group quantisation ([SGL-19] §Triton 分块内核在做什么, first step
 * per_token_group_quant_fp8(input_2d, block_size[1]); [GLM-17] §第1站 eq.
 * s_g = max|x_i| / 448, q_i = round(x_i / s_g)).  One scale per token per
 * group of `group` channels; the last group may be partial. */
void orc_quant_group(const uint16_t *x, int64_t M, int64_t K, int64_t ldx,
                     int64_t group, uint8_t *q, float *s) {
  int64_t G = (K + group - 1) / group;
  for (int64_t i = 0; i < M; ++i) {
    const uint16_t *xr = x + i * ldx;
    for (int64_t g = 0; g < G; ++g) {
      int64_t k0 = g * group, k1 = k0 + group < K ? k0 + group : K;
      float amax = 0.0f;
      for (int64_t k = k0; k < k1; ++k) {
        float a = fabsf(orc_bf16_to_f32(xr[k]));
        if (a > amax) amax = a;
      }
      float sg = group_scale(amax);
      s[i * G + g] = sg;
      for (int64_t k = k0; k < k1; ++k)
        q[i * K + k] = quant_one(orc_bf16_to_f32(xr[k]), sg);
    }
  }
}

/* ceil(log2 r) for a positive, finite binary64 r, from frexp. */
static int ceil_log2(double r) {
  int ex;
  double f = frexp(r, &ex); /* r = f * 2^ex, f in [0.5, 1) */
  return (f == 0.5) ? ex - 1 : ex;
}

/* MXFP8: blocks of [1,32] with a UE8M0 scale ([SGL-19] §checkpoint 里的量化元数据,
 * use_mxfp8 forces [1, 32]; [SGL-FP8] §1 and §4, uint8 scales).  The exponent
 * is the power of two rounded up from max(amax, 1e-10)/448 so that no value
 * overflows ([GLM-17] §第4站, the fused_indexer_q_rope_quant scale rule), then
 * q = RNE_sat(x * 2^-e) with an exact power-of-two scaling. */
void orc_quant_mx(const uint16_t *x, int64_t M, int64_t K, int64_t ldx,
                  uint8_t *q, uint8_t *u) {
  int64_t G = K / 32;
  for (int64_t i = 0; i < M; ++i) {
    const uint16_t *xr = x + i * ldx;
    for (int64_t g = 0; g < G; ++g) {
      float amax = 0.0f;
      for (int64_t k = g * 32; k < g * 32 + 32; ++k) {
        float a = fabsf(orc_bf16_to_f32(xr[k]));
        if (a > amax) amax = a;
      }
      float r = group_scale(amax);
      int e = ceil_log2((double)r);
      u[i * G + g] = (uint8_t)(e + 127);
      for (int64_t k = g * 32; k < g * 32 + 32; ++k)
        q[i * K + k] = orc_e4m3_encode(ldexp((double)orc_bf16_to_f32(xr[k]), -e));
    }
  }
}

/* Static activation quantisation: one fixed FP32 scale read from the
 * checkpoint ([SGL-19] §激活量化的三种选择, static_quant_fp8). */
void orc_quant_static(const uint16_t *x, int64_t M, int64_t K, int64_t ldx,
                      float s, uint8_t *q) {
  for (int64_t i = 0; i < M; ++i)
    for (int64_t k = 0; k < K; ++k)
      q[i * K + k] = quant_one(orc_bf16_to_f32(x[i * ldx + k]), s);
}

/* Per-tensor scale s = max|W| / 448 ([SGL-19] §从浮点到 FP8 的基本公式,
 * s_tensor), floored like every other scale here. */
float orc_absmax_scale(const uint16_t *x, int64_t r0, int64_t r1, int64_t K,
                       int64_t ldx) {
  float amax = 0.0f;
  for (int64_t i = r0; i < r1; ++i)
    for (int64_t k = 0; k < K; ++k) {
      float a = fabsf(orc_bf16_to_f32(x[i * ldx + k]));
      if (a > amax) amax = a;
    }
  return group_scale(amax);
}

/* Block quantisation of a weight [N, K]: one scale per bn x bk block, grid
 * ceil(N/bn) x ceil(K/bk); a partial edge block uses only its valid elements
 * ([SGL-19] §三种 scale 的存储形状, the ceil grid and the masking paragraph). */
void orc_quant_weight_block(const uint16_t *w, int64_t N, int64_t K,
                            int64_t ldw, int64_t bn, int64_t bk, uint8_t *q,
                            float *s) {
  int64_t NB = (N + bn - 1) / bn, KB = (K + bk - 1) / bk;
  for (int64_t nb = 0; nb < NB; ++nb)
    for (int64_t kb = 0; kb < KB; ++kb) {
      int64_t n0 = nb * bn, n1 = n0 + bn < N ? n0 + bn : N;
      int64_t k0 = kb * bk, k1 = k0 + bk < K ? k0 + bk : K;
      float amax = 0.0f;
      for (int64_t n = n0; n < n1; ++n)
        for (int64_t k = k0; k < k1; ++k) {
          float a = fabsf(orc_bf16_to_f32(w[n * ldw + k]));
          if (a > amax) amax = a;
        }
      float sb = group_scale(amax);
      s[nb * KB + kb] = sb;
      for (int64_t n = n0; n < n1; ++n)
        for (int64_t k = k0; k < k1; ++k)
          q[n * K + k] = quant_one(orc_bf16_to_f32(w[n * ldw + k]), sb);
    }
}

/* One scale per logical output partition of a fused weight ([SGL-FP8] §5
 * PerTensorScaleParameter of len(output_partition_sizes)). */
void orc_quant_weight_static(const uint16_t *w, int64_t N, int64_t K,
                             int64_t ldw, const int64_t *part_sizes,
                             int n_parts, uint8_t *q, float *s_part) {
  (void)N;
  int64_t r0 = 0;
  for (int p = 0; p < n_parts; ++p) {
    int64_t r1 = r0 + part_sizes[p];
    float sp = orc_absmax_scale(w, r0, r1, K, ldw);
    s_part[p] = sp;
    orc_quant_static(w + r0 * ldw, r1 - r0, K, ldw, sp, q + r0 * K);
    r0 = r1;
  }
}

/* ======================================================================= */
/* Reference GEMMs                                                          */
/* ======================================================================= */

int64_t orc_e4m3_dot_int(const uint8_t *a, const uint8_t *b, int64_t n) {
  int64_t acc = 0;
  for (int64_t k = 0; k < n; ++k)
    acc += (int64_t)orc_e4m3_sig(a[k]) * (int64_t)orc_e4m3_sig(b[k]);
  return acc;
}

double orc_e4m3_dot_f64(const uint8_t *a, const uint8_t *b, int64_t n) {
  double acc = 0.0;
  for (int64_t k = 0; k < n; ++k)
    acc += orc_e4m3_decode(a[k]) * orc_e4m3_decode(b[k]);
  return acc;
}

enum { KIND_BLOCK = 0, KIND_MX = 1, KIND_STATIC = 2, KIND_CHANNEL = 3, KIND_GROUPED = 4 };

typedef struct {
  int kind;
  const uint8_t *qa, *qw;
  const float *sa, *sw;    /* block: row-major grids; static: sa[0] = s_x, sw = s_part;
                              channel: sa[M] per token, sw[N] per output channel */
  const uint8_t *ua, *uw;  /* MX scale codes */
  const int64_t *part_sizes;
  int n_parts;
  const int32_t *row_expert; /* grouped: expert of each activation row, -1 = none */
  const uint16_t *bias;
  int64_t M, N, K, bn, bk;
  const int64_t *rows, *cols; /* sampled mode when non-NULL */
  int64_t n;                  /* number of outputs */
  double *y;
  int64_t t0, t1;             /* this worker's output range */
} gemm_job;

/* Block-scaled element ([SGL-19] §一条 GEMM 的三种缩放组合, the block-wise
 * equation: Y_ij = sum_b (sum_{k in b} Qx[i,k] Qw[j,k]) * s_x[i,b] * s_w[j,b],
 * with s_w indexed by the 128-row block of j). */
static double elem_block(const gemm_job *g, int64_t i, int64_t j) {
  int64_t KB = (g->K + g->bk - 1) / g->bk;
  const uint8_t *a = g->qa + i * g->K, *w = g->qw + j * g->K;
  double y = 0.0;
  for (int64_t kb = 0; kb < KB; ++kb) {
    int64_t k0 = kb * g->bk, k1 = k0 + g->bk < g->K ? k0 + g->bk : g->K;
    double p = orc_e4m3_dot_f64(a + k0, w + k0, k1 - k0);
    y += p * (double)g->sa[i * KB + kb] * (double)g->sw[(j / g->bn) * KB + kb];
  }
  return y;
}

/* MXFP8 element: per 32-wide group, the partial sum times both power-of-two
 * scales ([GLM-17] §第7站: UE8M0 scales consumed by the MMA). */
static double elem_mx(const gemm_job *g, int64_t i, int64_t j) {
  int64_t G = g->K / 32;
  const uint8_t *a = g->qa + i * g->K, *w = g->qw + j * g->K;
  double y = 0.0;
  for (int64_t gi = 0; gi < G; ++gi) {
    double p = orc_e4m3_dot_f64(a + gi * 32, w + gi * 32, 32);
    y += p * orc_ue8m0_decode(g->ua[i * G + gi]) *
         orc_ue8m0_decode(g->uw[j * G + gi]);
  }
  return y;
}

/* Per-tensor element: Y = (Qx Qw^T) * (s_x s_w^T) with scalar s_x and the
 * per-partition weight scale expanded to its output rows ([SGL-19] §一条 GEMM
 * 的三种缩放组合; §装载后的三个分支, convert_to_channelwise). */
static double elem_static(const gemm_job *g, int64_t i, int64_t j) {
  int64_t r0 = 0;
  int p = 0;
  for (; p < g->n_parts; ++p) {
    if (j < r0 + g->part_sizes[p]) break;
    r0 += g->part_sizes[p];
  }
  double acc = orc_e4m3_dot_f64(g->qa + i * g->K, g->qw + j * g->K, g->K);
  return acc * (double)g->sa[0] * (double)g->sw[p];
}

/* Channelwise element: one dynamic scale per token (activation row) and one
 * per output channel (weight row) come out of the full-K sum ([SGL-19]
 * §一条 GEMM 的三种缩放组合, the per-token x per-channel case:
 * Y_ij = (sum_k Qx[i,k] Qw[j,k]) * s_x[i] * s_w[j]). */
static double elem_channel(const gemm_job *g, int64_t i, int64_t j) {
  double acc = orc_e4m3_dot_f64(g->qa + i * g->K, g->qw + j * g->K, g->K);
  return acc * (double)g->sa[i] * (double)g->sw[j];
}

/* Grouped (MoE) element: the block-wise element of row i against the weight
 * [N][K] and scale grid [ceil(N/bn)][ceil(K/bk)] of that row's expert
 * ([SGL-19] §MoE:专家权重多一个维度: expert weights [E, N, K] with the block
 * scales replicated per expert, [E, ceil(N/b_n), ceil(K/b_k)]; the grouped GEMM
 * takes tokens sorted by expert).  Rows of no expert give NaN. */
static double elem_grouped(const gemm_job *g, int64_t i, int64_t j) {
  int32_t e = g->row_expert[i];
  if (e < 0) return NAN;
  int64_t KB = (g->K + g->bk - 1) / g->bk, NB = (g->N + g->bn - 1) / g->bn;
  gemm_job ge = *g;
  ge.qw = g->qw + (int64_t)e * g->N * g->K;
  ge.sw = g->sw + (int64_t)e * NB * KB;
  return elem_block(&ge, i, j);
}

static void *gemm_worker(void *arg) {
  const gemm_job *g = (const gemm_job *)arg;
  for (int64_t t = g->t0; t < g->t1; ++t) {
    int64_t i, j;
    if (g->rows) {
      i = g->rows[t];
      j = g->cols[t];
    } else {
      i = t / g->N;
      j = t % g->N;
    }
    double y;
    if (g->kind == KIND_BLOCK) y = elem_block(g, i, j);
    else if (g->kind == KIND_MX) y = elem_mx(g, i, j);
    else if (g->kind == KIND_CHANNEL) y = elem_channel(g, i, j);
    else if (g->kind == KIND_GROUPED) y = elem_grouped(g, i, j);
    else y = elem_static(g, i, j);
    if (g->bias) y += (double)orc_bf16_to_f32(g->bias[j]); /* epilogue bias */
    g->y[t] = y;
  }
  return NULL;
}

/* Splits the outputs into contiguous ranges, one per thread.  Each output is
 * computed independently, so the thread count never changes a result. */
static void run_gemm(gemm_job base, int nthreads) {
  enum { MAX_THREADS = 256 };
  if (nthreads < 1) nthreads = 1;
  if (nthreads > MAX_THREADS) nthreads = MAX_THREADS;
  if (base.n < (int64_t)nthreads * 16) nthreads = 1;
  if (nthreads == 1) {
    base.t0 = 0;
    base.t1 = base.n;
    gemm_worker(&base);
    return;
  }
  pthread_t th[MAX_THREADS];
  int joined[MAX_THREADS];
  gemm_job jobs[MAX_THREADS];
  int64_t per = (base.n + nthreads - 1) / nthreads;
  for (int t = 0; t < nthreads; ++t) {
    jobs[t] = base;
    jobs[t].t0 = (int64_t)t * per < base.n ? (int64_t)t * per : base.n;
    jobs[t].t1 = jobs[t].t0 + per < base.n ? jobs[t].t0 + per : base.n;
    joined[t] = pthread_create(&th[t], NULL, gemm_worker, &jobs[t]) == 0;
    if (!joined[t]) gemm_worker(&jobs[t]); /* no thread available: run inline */
  }
  for (int t = 0; t < nthreads; ++t)
    if (joined[t]) pthread_join(th[t], NULL);
}

static gemm_job job0(int kind, int64_t M, int64_t N, int64_t K, double *y,
                     const uint16_t *bias) {
  gemm_job g;
  memset(&g, 0, sizeof g);
  g.kind = kind;
  g.M = M;
  g.N = N;
  g.K = K;
  g.y = y;
  g.bias = bias;
  g.n = M * N;
  return g;
}

void orc_gemm_block(const uint8_t *qa, const float *sa, const uint8_t *qw,
                    const float *sw, const uint16_t *bias, int64_t M,
                    int64_t N, int64_t K, int64_t bn, int64_t bk, double *y,
                    int nthreads) {
  gemm_job g = job0(KIND_BLOCK, M, N, K, y, bias);
  g.qa = qa; g.qw = qw; g.sa = sa; g.sw = sw; g.bn = bn; g.bk = bk;
  run_gemm(g, nthreads);
}

void orc_gemm_block_sampled(const uint8_t *qa, const float *sa,
                            const uint8_t *qw, const float *sw,
                            const uint16_t *bias, int64_t M, int64_t N,
                            int64_t K, int64_t bn, int64_t bk,
                            const int64_t *rows, const int64_t *cols,
                            int64_t n, double *y, int nthreads) {
  gemm_job g = job0(KIND_BLOCK, M, N, K, y, bias);
  g.qa = qa; g.qw = qw; g.sa = sa; g.sw = sw; g.bn = bn; g.bk = bk;
  g.rows = rows; g.cols = cols; g.n = n;
  run_gemm(g, nthreads);
}

void orc_gemm_mx(const uint8_t *qa, const uint8_t *ua, const uint8_t *qw,
                 const uint8_t *uw, const uint16_t *bias, int64_t M, int64_t N,
                 int64_t K, double *y, int nthreads) {
  gemm_job g = job0(KIND_MX, M, N, K, y, bias);
  g.qa = qa; g.qw = qw; g.ua = ua; g.uw = uw;
  run_gemm(g, nthreads);
}

void orc_gemm_mx_sampled(const uint8_t *qa, const uint8_t *ua,
                         const uint8_t *qw, const uint8_t *uw,
                         const uint16_t *bias, int64_t M, int64_t N, int64_t K,
                         const int64_t *rows, const int64_t *cols, int64_t n,
                         double *y, int nthreads) {
  gemm_job g = job0(KIND_MX, M, N, K, y, bias);
  g.qa = qa; g.qw = qw; g.ua = ua; g.uw = uw;
  g.rows = rows; g.cols = cols; g.n = n;
  run_gemm(g, nthreads);
}

void orc_gemm_static(const uint8_t *qa, float s_x, const uint8_t *qw,
                     const float *s_part, const int64_t *part_sizes,
                     int n_parts, const uint16_t *bias, int64_t M, int64_t N,
                     int64_t K, double *y, int nthreads) {
  gemm_job g = job0(KIND_STATIC, M, N, K, y, bias);
  g.qa = qa; g.qw = qw; g.sa = &s_x; g.sw = s_part;
  g.part_sizes = part_sizes; g.n_parts = n_parts;
  run_gemm(g, nthreads);
}

void orc_gemm_static_sampled(const uint8_t *qa, float s_x, const uint8_t *qw,
                             const float *s_part, const int64_t *part_sizes,
                             int n_parts, const uint16_t *bias, int64_t M,
                             int64_t N, int64_t K, const int64_t *rows,
                             const int64_t *cols, int64_t n, double *y,
                             int nthreads) {
  gemm_job g = job0(KIND_STATIC, M, N, K, y, bias);
  g.qa = qa; g.qw = qw; g.sa = &s_x; g.sw = s_part;
  g.part_sizes = part_sizes; g.n_parts = n_parts;
  g.rows = rows; g.cols = cols; g.n = n;
  run_gemm(g, nthreads);
}

/* ======================================================================= */
/* Residual add + RMSNorm                                                   */
/* ======================================================================= */

/* binary64 -> BF16 bits, round to nearest even; beyond the largest finite
 * BF16 (plus half an ulp) -> infinity; NaN -> quiet NaN with the sign kept. */
uint16_t orc_bf16_from_f64(double v) {
  uint16_t sign = signbit(v) ? 0x8000u : 0u;
  if (v != v) return sign | 0x7FC0u;
  double a = fabs(v);
  if (a == 0.0) return sign;
  if (isinf(a)) return sign | 0x7F80u;
  int ex;
  frexp(a, &ex);             /* a in [2^(ex-1), 2^ex) */
  int e = ex - 1;
  if (e < -126) e = -126;    /* subnormal BF16: quantum 2^-133 */
  double quantum = ldexp(1.0, e - 7);
  uint32_t n = rne_uint(a / quantum); /* exact scaling by a power of two */
  double r = (double)n * quantum;     /* n may be 256: the next binade */
  if (r >= 0x1p128) return sign | 0x7F80u;
  union {
    float f;
    uint32_t u;
  } c;
  c.f = (float)r; /* exact: r has at most 8 significant bits */
  return sign | (uint16_t)(c.u >> 16);
}

/* Sum of r_i^2 over a row of BF16 values, computed exactly and rounded once to
 * binary32 (nearest, ties to even).  The page fixes only that the sum is taken
 * in FP32 ([GLM-17] §第1站 "求和与开方在 FP32 上完成"); its order is open, and
 * the correctly rounded value is the one every order approximates.  Each
 * nonzero finite r = m * 2^(E-134) with an integer m <= 255 and a biased
 * exponent E in 1..254, so r^2 = m^2 * 2^(2E-268): the row sum is the integer
 * A = sum m^2 * 2^(2E-2) times 2^-266, accumulated in 32-bit limbs.  NaN in the
 * row gives NaN, otherwise an infinity gives +infinity. */
#define SUMSQ_LIMBS 20
float orc_sumsq_f32(const uint16_t *r, int64_t d) {
  uint32_t A[SUMSQ_LIMBS];
  memset(A, 0, sizeof A);
  int any_nan = 0, any_inf = 0;
  for (int64_t i = 0; i < d; ++i) {
    uint32_t b = r[i] & 0x7FFFu;
    uint32_t E = b >> 7, frac = b & 0x7Fu;
    if (E == 0xFF) {
      if (frac) any_nan = 1;
      else any_inf = 1;
      continue;
    }
    uint32_t m = E ? (frac | 0x80u) : frac;
    if (E == 0) E = 1;
    if (m == 0) continue;
    uint32_t k = 2 * E - 2; /* bit position of m^2 in A */
    uint64_t add = (uint64_t)(m * m) << (k % 32);
    for (uint32_t l = k / 32; add != 0 && l < SUMSQ_LIMBS; ++l) {
      uint64_t t = (uint64_t)A[l] + (add & 0xFFFFFFFFu);
      A[l] = (uint32_t)t;
      add = (add >> 32) + (t >> 32);
    }
  }
  if (any_nan) return NAN;
  if (any_inf) return INFINITY;
  int p = -1; /* highest set bit of A */
  for (int l = SUMSQ_LIMBS - 1; l >= 0 && p < 0; --l)
    if (A[l]) {
      int h = 31;
      while (!((A[l] >> h) & 1u)) --h;
      p = 32 * l + h;
    }
  if (p < 0) return 0.0f;
  /* keep 24 significant bits, or fewer where the result is subnormal
   * (binary32 quantum 2^-149 = bit 117 of A) */
  int lsb = p - 23 > 117 ? p - 23 : 117;
  uint64_t mant = 0;
  for (int bit = p; bit >= lsb; --bit)
    mant = (mant << 1) | ((A[bit / 32] >> (bit % 32)) & 1u);
  int half = lsb > 0 ? (int)((A[(lsb - 1) / 32] >> ((lsb - 1) % 32)) & 1u) : 0;
  int sticky = 0;
  for (int bit = lsb - 2; bit >= 0 && !sticky; --bit)
    if ((A[bit / 32] >> (bit % 32)) & 1u) sticky = 1;
  if (half && (sticky || (mant & 1u))) ++mant;
  double v = ldexp((double)mant, lsb - 266); /* exact; >= 2^128 overflows below */
  return (float)v;
}

/* Residual add and RMSNorm of one decoder-layer input ([GLM-17] §第1站):
 *   r = x + residual, the BF16 residual stream (the add rounded to BF16 once);
 *   y = r / sqrt(mean(r^2) + eps) * g, sums and root in FP32, output BF16.
 * Readings: the mean is RN32(S / d) with S = orc_sumsq_f32(r); then
 * RN32(mean + eps), the correctly rounded FP32 square root, the FP32 quotient
 * r / rms and the FP32 product with g, rounded to BF16 once at the end.
 * residual may be NULL (plain RMSNorm: r = x).  r_out and y are [M][d]. */
void orc_add_rmsnorm(const uint16_t *x, int64_t ldx, const uint16_t *res,
                     int64_t ldr, const uint16_t *g, float eps, int64_t M,
                     int64_t d, uint16_t *r_out, uint16_t *y) {
  for (int64_t i = 0; i < M; ++i) {
    uint16_t *ri = r_out + i * d;
    for (int64_t k = 0; k < d; ++k) {
      double a = (double)orc_bf16_to_f32(x[i * ldx + k]);
      if (res) a += (double)orc_bf16_to_f32(res[i * ldr + k]);
      ri[k] = orc_bf16_from_f64(a); /* the sum of two BF16 values is exact in
                                       binary64 unless one is negligible */
    }
    volatile float S = orc_sumsq_f32(ri, d);
    volatile float ms = S / (float)d;
    volatile float t = ms + eps;
    volatile float rms = sqrtf(t);
    for (int64_t k = 0; k < d; ++k) {
      volatile float a = orc_bf16_to_f32(ri[k]) / rms;
      volatile float b = a * orc_bf16_to_f32(g[k]);
      y[i * d + k] = orc_bf16_from_f64((double)b);
    }
  }
}

void orc_gemm_channel(const uint8_t *qa, const float *sa, const uint8_t *qw,
                      const float *sw, const uint16_t *bias, int64_t M, int64_t N,
                      int64_t K, double *y, int nthreads) {
  gemm_job g = job0(KIND_CHANNEL, M, N, K, y, bias);
  g.qa = qa; g.qw = qw; g.sa = sa; g.sw = sw;
  run_gemm(g, nthreads);
}

void orc_gemm_channel_sampled(const uint8_t *qa, const float *sa,
                              const uint8_t *qw, const float *sw,
                              const uint16_t *bias, int64_t M, int64_t N,
                              int64_t K, const int64_t *rows,
                              const int64_t *cols, int64_t n, double *y,
                              int nthreads) {
  gemm_job g = job0(KIND_CHANNEL, M, N, K, y, bias);
  g.qa = qa; g.qw = qw; g.sa = sa; g.sw = sw;
  g.rows = rows; g.cols = cols; g.n = n;
  run_gemm(g, nthreads);
}

/* ======================================================================= */
/* Block FP8 with UE8M0 (power-of-two) scales                               */
/* ======================================================================= */

/* Smallest e with 2^e >= r, for a positive finite binary64 r. */
static int ceil_pow2_exponent(double r) {
  int ex;
  double f = frexp(r, &ex); /* r = f * 2^ex, f in [0.5, 1) */
  return f == 0.5 ? ex - 1 : ex;
}

/* Per-token group quantisation with the scale restricted to a power of two
 * ([SGL-19] §分块 GEMM 的后端分派: with act_scale_ue8m0 the activation
 * quantiser keeps the per-token-group layout but limits each scale to 2^e).
 * Reading: e is the smallest exponent keeping every value of the group within
 * +-448, e = ceil(log2(max(amax, 1e-10) / 448)) with the binary32 division;
 * u = e + 127; q = RNE_sat(x * 2^-e), an exact power-of-two scaling.  The last
 * group may be partial.  u is [M][ceil(K/group)]. */
void orc_quant_ue8m0(const uint16_t *x, int64_t M, int64_t K, int64_t ldx,
                     int64_t group, uint8_t *q, uint8_t *u) {
  int64_t G = (K + group - 1) / group;
  for (int64_t i = 0; i < M; ++i) {
    for (int64_t g = 0; g < G; ++g) {
      int64_t k0 = g * group, k1 = k0 + group < K ? k0 + group : K;
      float amax = 0.0f;
      for (int64_t k = k0; k < k1; ++k) {
        float a = fabsf(orc_bf16_to_f32(x[i * ldx + k]));
        if (a > amax) amax = a;
      }
      volatile float floored = amax < 1e-10f ? 1e-10f : amax;
      volatile float r = floored / 448.0f;
      int e = ceil_pow2_exponent((double)r);
      u[i * G + g] = (uint8_t)(e + 127);
      for (int64_t k = k0; k < k1; ++k)
        q[i * K + k] = orc_e4m3_encode(ldexp((double)orc_bf16_to_f32(x[i * ldx + k]), -e));
    }
  }
}

/* FP32 block scales of a quantised weight re-expressed as UE8M0 ([SGL-19]
 * §分块路径的后处理: for the SM100 runner
 * the FP32 block scale is requantised to a power-of-two scale, since only
 * powers of two convert exactly in the kernel).  Reading: per bn x bk block,
 * s' = 2^e with e = ceil(log2 s) (the nearest power of two at or above s, so
 * no value grows), u = e + 127, and every code re-encoded from its value:
 * q' = RNE_sat(dec(q) * s / s'), exact in binary64.  s is [ceil(N/bn)][ceil(K/bk)],
 * u the same shape. */
void orc_requant_weight_ue8m0(const uint8_t *q, const float *s, int64_t N, int64_t K,
                              int64_t bn, int64_t bk, uint8_t *q2, uint8_t *u) {
  int64_t NB = (N + bn - 1) / bn, KB = (K + bk - 1) / bk;
  for (int64_t nb = 0; nb < NB; ++nb)
    for (int64_t kb = 0; kb < KB; ++kb) {
      double sv = (double)s[nb * KB + kb];
      int e = ceil_pow2_exponent(sv);
      u[nb * KB + kb] = (uint8_t)(e + 127);
      double m = ldexp(sv, -e); /* s / s', in (1/2, 1] */
      for (int64_t n = nb * bn; n < N && n < (nb + 1) * bn; ++n)
        for (int64_t k = kb * bk; k < K && k < (kb + 1) * bk; ++k)
          q2[n * K + k] = orc_e4m3_encode(orc_e4m3_decode(q[n * K + k]) * m);
    }
}

void orc_gemm_grouped(const uint8_t *qa, const float *sa, const uint8_t *qw,
                      const float *sw, const int32_t *row_expert, int64_t M,
                      int64_t N, int64_t K, double *y, int nthreads) {
  gemm_job g = job0(KIND_GROUPED, M, N, K, y, NULL);
  g.qa = qa; g.qw = qw; g.sa = sa; g.sw = sw; g.bn = 128; g.bk = 128;
  g.row_expert = row_expert;
  run_gemm(g, nthreads);
}

void orc_gemm_grouped_sampled(const uint8_t *qa, const float *sa, const uint8_t *qw,
                              const float *sw, const int32_t *row_expert, int64_t M,
                              int64_t N, int64_t K, const int64_t *rows,
                              const int64_t *cols, int64_t n, double *y, int nthreads) {
  gemm_job g = job0(KIND_GROUPED, M, N, K, y, NULL);
  g.qa = qa; g.qw = qw; g.sa = sa; g.sw = sw; g.bn = 128; g.bk = 128;
  g.row_expert = row_expert;
  g.rows = rows; g.cols = cols; g.n = n;
  run_gemm(g, nthreads);
}
