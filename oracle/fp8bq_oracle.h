/*
 * fp8bq_oracle.h -- plain, slow CPU oracle for the block-wise FP8 W8A8 linear.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may include, link or
 * call this code; only the test-suite, the smoke check and the CPU-baseline leg
 * of the benchmark use it.  It shares no code with the CUDA library.
 *
 * Every routine restates a passage of the source pages; citations name the page
 * and its section:
 *   [SGL-19]  "SGLang 源码完全拆解(十九): 量化方法的注册与层分派" (pinghaoyang.com.cn)
 *   [SGL-FP8] "[SGLang] FP8: 8비트 부동소수점 양자화의 구현과 성능" (blog.secrett2633.cloud)
 *   [GLM-17]  "GLM-5.3 推理全链路(十七): 一条请求的精度账本" (pinghaoyang.com.cn)
 *
 * Arithmetic rules: scales and quotients are IEEE binary32 divisions (the pages
 * write s = amax/448 and q = round(x/s)); everything after decoding is binary64.
 * Build with -O2 -ffp-contract=off -fno-fast-math so x86-64 and aarch64 agree.
 *
 * Parity status: every function here is pinned by tests/test_oracle_*.py
 * (closed forms, library special cases, brute force on tiny inputs); none is
 * "parity unpinned".
 */
#ifndef FP8BQ_ORACLE_H
#define FP8BQ_ORACLE_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- number formats ---------------------------------------------------- */
uint8_t orc_e4m3_encode(double v);       /* RNE, saturate to +-448, NaN -> 0x7F */
double  orc_e4m3_decode(uint8_t c);      /* 0x7F/0xFF -> NaN                    */
int32_t orc_e4m3_sig(uint8_t c);         /* decode(c) * 2^9 as an exact integer */
double  orc_ue8m0_decode(uint8_t u);     /* 2^(u-127); 255 -> NaN               */
float   orc_bf16_to_f32(uint16_t b);
/* Array forms of the codecs (binary32 inputs, as a kernel converts them). */
void    orc_e4m3_encode_f32_array(const float *v, int64_t n, uint8_t *out);
void    orc_e4m3_decode_array(const uint8_t *c, int64_t n, double *out);
/* codes of the binary32 values with bit patterns first .. first + n - 1 */
void    orc_e4m3_encode_bits_range(uint32_t first, int64_t n, uint8_t *out, int nthreads);

/* ---- quantisers (activation side) -------------------------------------- */
/* Per-token group quantisation, FP32 scales, row-major s[M][ceil(K/group)]. */
void orc_quant_group(const uint16_t *x, int64_t M, int64_t K, int64_t ldx,
                     int64_t group, uint8_t *q, float *s);
/* MXFP8 [1,32] quantisation, UE8M0 scale codes u[M][K/32].                  */
void orc_quant_mx(const uint16_t *x, int64_t M, int64_t K, int64_t ldx,
                  uint8_t *q, uint8_t *u);
/* Static per-tensor quantisation with a given scale.                        */
void orc_quant_static(const uint16_t *x, int64_t M, int64_t K, int64_t ldx,
                      float s, uint8_t *q);
/* Per-tensor scale max(amax, 1e-10)/448 over rows [r0, r1) of a matrix.     */
float orc_absmax_scale(const uint16_t *x, int64_t r0, int64_t r1, int64_t K,
                       int64_t ldx);

/* Channelwise (per-token x per-channel): y = (sum_k qa*qw) * sa[i] * sw[j]. */
void orc_gemm_channel(const uint8_t *qa, const float *sa, const uint8_t *qw,
                      const float *sw, const uint16_t *bias, int64_t M, int64_t N,
                      int64_t K, double *y, int nthreads);
void orc_gemm_channel_sampled(const uint8_t *qa, const float *sa,
                              const uint8_t *qw, const float *sw,
                              const uint16_t *bias, int64_t M, int64_t N,
                              int64_t K, const int64_t *rows,
                              const int64_t *cols, int64_t n, double *y,
                              int nthreads);

/* Grouped (MoE) block-scaled GEMM: row i uses expert row_expert[i]'s weight
 * qw[e] [N][K] and scales sw[e] [ceil(N/128)][ceil(K/128)]; -1 gives NaN.    */
void orc_gemm_grouped(const uint8_t *qa, const float *sa, const uint8_t *qw,
                      const float *sw, const int32_t *row_expert, int64_t M,
                      int64_t N, int64_t K, double *y, int nthreads);
void orc_gemm_grouped_sampled(const uint8_t *qa, const float *sa, const uint8_t *qw,
                              const float *sw, const int32_t *row_expert, int64_t M,
                              int64_t N, int64_t K, const int64_t *rows,
                              const int64_t *cols, int64_t n, double *y, int nthreads);

/* ---- block FP8 with UE8M0 scales ---------------------------------------- */
/* Group quantisation with power-of-two scales: u[M][ceil(K/group)].          */
void orc_quant_ue8m0(const uint16_t *x, int64_t M, int64_t K, int64_t ldx,
                     int64_t group, uint8_t *q, uint8_t *u);
/* FP32 block scales -> UE8M0 (rounded up), codes re-encoded per block.       */
void orc_requant_weight_ue8m0(const uint8_t *q, const float *s, int64_t N, int64_t K,
                              int64_t bn, int64_t bk, uint8_t *q2, uint8_t *u);

/* ---- residual add + RMSNorm (the step before the activation quantiser) -- */
/* binary64 -> BF16 (RNE, overflow to infinity).                             */
uint16_t orc_bf16_from_f64(double v);
/* sum of squares of a BF16 row, exact, rounded once to binary32 (RNE).      */
float   orc_sumsq_f32(const uint16_t *r, int64_t d);
/* r = BF16(x + residual) (residual may be NULL), y = BF16 RMSNorm(r) * g.   */
void    orc_add_rmsnorm(const uint16_t *x, int64_t ldx, const uint16_t *res,
                        int64_t ldr, const uint16_t *g, float eps, int64_t M,
                        int64_t d, uint16_t *r_out, uint16_t *y);

/* ---- quantisers (weight side, used to build test weights) -------------- */
/* 128x128 (bn x bk) block quantisation: s[ceil(N/bn)][ceil(K/bk)].          */
void orc_quant_weight_block(const uint16_t *w, int64_t N, int64_t K,
                            int64_t ldw, int64_t bn, int64_t bk,
                            uint8_t *q, float *s);
/* Per-partition static weight quantisation; s_part[n_parts].                */
void orc_quant_weight_static(const uint16_t *w, int64_t N, int64_t K,
                             int64_t ldw, const int64_t *part_sizes,
                             int n_parts, uint8_t *q, float *s_part);

/* ---- reference GEMMs (binary64) ---------------------------------------- */
/* Block-scaled: y[i][j] = sum_kb (sum_{k in kb} qa*qw) * sa[i][kb] * sw[j/bn][kb]
 * (+ bias[j]).  sa is row-major [M][ceil(K/bk)].  bias may be NULL.         */
void orc_gemm_block(const uint8_t *qa, const float *sa, const uint8_t *qw,
                    const float *sw, const uint16_t *bias, int64_t M,
                    int64_t N, int64_t K, int64_t bn, int64_t bk, double *y,
                    int nthreads);
void orc_gemm_block_sampled(const uint8_t *qa, const float *sa,
                            const uint8_t *qw, const float *sw,
                            const uint16_t *bias, int64_t M, int64_t N,
                            int64_t K, int64_t bn, int64_t bk,
                            const int64_t *rows, const int64_t *cols,
                            int64_t n, double *y, int nthreads);
/* MXFP8: groups of 32 along K, factors 2^(ua-127) * 2^(uw-127).             */
void orc_gemm_mx(const uint8_t *qa, const uint8_t *ua, const uint8_t *qw,
                 const uint8_t *uw, const uint16_t *bias, int64_t M, int64_t N,
                 int64_t K, double *y, int nthreads);
void orc_gemm_mx_sampled(const uint8_t *qa, const uint8_t *ua,
                         const uint8_t *qw, const uint8_t *uw,
                         const uint16_t *bias, int64_t M, int64_t N, int64_t K,
                         const int64_t *rows, const int64_t *cols, int64_t n,
                         double *y, int nthreads);
/* Static: (sum_k qa*qw) * s_x * s_part[p(j)], partitions in output order.   */
void orc_gemm_static(const uint8_t *qa, float s_x, const uint8_t *qw,
                     const float *s_part, const int64_t *part_sizes,
                     int n_parts, const uint16_t *bias, int64_t M, int64_t N,
                     int64_t K, double *y, int nthreads);
void orc_gemm_static_sampled(const uint8_t *qa, float s_x, const uint8_t *qw,
                             const float *s_part, const int64_t *part_sizes,
                             int n_parts, const uint16_t *bias, int64_t M,
                             int64_t N, int64_t K, const int64_t *rows,
                             const int64_t *cols, int64_t n, double *y,
                             int nthreads);

/* Exact integer dot of E4M3 significands (each value * 2^9), for cross-checks. */
int64_t orc_e4m3_dot_int(const uint8_t *a, const uint8_t *b, int64_t n);
/* Binary64 dot of decoded E4M3 values (the inner sum of the GEMMs above).    */
double orc_e4m3_dot_f64(const uint8_t *a, const uint8_t *b, int64_t n);

#ifdef __cplusplus
}
#endif
#endif
