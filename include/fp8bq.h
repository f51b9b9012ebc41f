/*
 * fp8bq.h -- C ABI of the block-wise FP8 W8A8 linear for one NVIDIA GB300 (sm_103a).
 *
 * The operation is the forward of an FP8 linear layer as the pages describe it
 * (apply(layer, x, bias) -> y, with the layer's E4M3 weight and its scales):
 *
 *   1. activation quantisation: per token, per group of 128 channels,
 *      s = max|x| / 448 and q = round_to_nearest_even(x / s), saturated to +-448
 *      ("SGLang 源码完全拆解(十九)", §从浮点到 FP8 的基本公式 and
 *      §Triton 分块内核在做什么; "GLM-5.3 推理全链路(十七)", §第1站 eq. for s_g, q_i);
 *   2. block-scaled FP8 GEMM: y[i][j] = sum_b (sum_{k in block b} q[i][k] w[j][k])
 *      * s_x[i][b] * s_w[j/128][b], FP32 accumulation, promoted once per 128-wide
 *      K block, BF16 output ("SGLang 源码完全拆解(十九)", §一条 GEMM 的三种缩放组合,
 *      the block-wise equation; §Triton 分块内核在做什么);
 *   3. the two fused: BF16 in, BF16 out (same page, §一次前向的完整时序);
 *   plus an MXFP8 variant ([1,32] blocks, UE8M0 scales; same page §checkpoint
 *   里的量化元数据 and "[SGLang] FP8" §4), a static per-tensor variant
 *   (one activation scale, one weight scale per output partition; "SGLang 源码完全
 *   拆解(十九)", §激活量化的三种选择 and "[SGLang] FP8" §5), a channelwise
 *   variant (per-token x per-channel scales; §一条 GEMM 的三种缩放组合), block
 *   FP8 with power-of-two (UE8M0) scales run on the block-scaled MMA
 *   (§分块 GEMM 的后端分派), the residual add + RMSNorm that precedes the
 *   activation quantiser, fused with it ("GLM-5.3 推理全链路(十七)", §第1站),
 *   and the grouped (MoE) block GEMM over experts' weights [E, N, K]
 *   ("SGLang 源码完全拆解(十九)", §MoE:专家权重多一个维度).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - All tensor pointers are DEVICE pointers owned by the caller; the library
 *    allocates nothing and keeps no per-call state.  Host pointers are named
 *    `*_host`.
 *  - Layouts are row-major.  X is BF16 [M, K] with row pitch `ldx` elements;
 *    Q (E4M3 codes) is [M, K] with pitch K; W is E4M3 [N, K] with pitch K;
 *    Y is BF16 [M, N] with pitch N.  bias, when not NULL, is BF16 [N].
 *  - Block path scales: s_w is FP32 [ceil(N/128)][ceil(K/128)] ("weight_scale_inv",
 *    the dequantisation multiplier); s_x is FP32 and either row-major
 *    [M][ceil(K/128)] (FP8BQ_SCALE_ROW_MAJOR) or column-major
 *    [ceil(K/128)][round_up(M,4)] (FP8BQ_SCALE_COL_MAJOR).
 *  - MX path scales are UE8M0 codes (uint8, value 2^(u-127)), row-major
 *    [rows][K/32] for both activations and weights.
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *    Calls are asynchronous and stream-ordered.
 *  - Arguments are validated on the host before anything is launched; on an
 *    error nothing is launched and no output is touched.  M == 0 is a valid
 *    empty batch: FP8BQ_OK without launching, and the tensor pointers may be NULL.
 *  - Requirements: x, q, w, y 16-byte aligned; ldx >= K and ldx % 8 == 0;
 *    K % 16 == 0 for the E4M3 paths and K % 32 == 0 for MX; FP32 scale
 *    pointers 4-byte aligned; bias 2-byte aligned.
 *  - GEMM and linear entry points take a workspace `ws` of at least
 *    fp8bq_workspace_bytes(op, M, N, K) bytes, 256-byte aligned, zeroed once
 *    with fp8bq_workspace_init before its first use.  The library keeps it in a
 *    valid state between calls (every partial-sum slot a call fills is read
 *    and cleared again within the same call).  Besides a status word and tile
 *    counters it holds FP32 partial sums: the split-K decode tiles' (M <= 64) and, for the
 *    block GEMM and linear above 64 rows, those of the last wave's tiles,
 *    which run split into K ranges on otherwise idle SMs (256 KB per split,
 *    at most 80 splits: up to 20 MB).  Calls that share a workspace must not overlap
 *    on the GPU (same stream, or ordered by events).
 *  - Every device-side wait is bounded: a wait that runs out sets a status word
 *    in the workspace, the kernel exits cleanly, and fp8bq_poll_status reports
 *    FP8BQ_ERR_TIMEOUT.  The limit is 1 s per wait, or FP8BQ_WAIT_LIMIT_MS from
 *    the environment, read once.  After a timeout the outputs are undefined
 *    and the workspace must be zeroed again (fp8bq_workspace_init).  For
 *    tests, FP8BQ_FAULT_INJECT=skip_first_load:<n> (read once) makes the next
 *    n GEMM launches skip one tile copy so that their waits run out.
 *  - No C++ exception crosses this interface.
 */
#ifndef FP8BQ_H
#define FP8BQ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define FP8BQ_API __attribute__((visibility("default")))

/* Status codes returned by every int-returning entry point. */
typedef enum fp8bq_status {
  FP8BQ_OK = 0,
  FP8BQ_ERR_NULL = 1,        /* a required pointer is NULL                          */
  FP8BQ_ERR_SHAPE = 2,       /* M < 0, N < 1, K < 1, ldx < K, bad partitions         */
  FP8BQ_ERR_ALIGN = 3,       /* pointer or pitch breaks the alignment rules above   */
  FP8BQ_ERR_UNSUPPORTED = 4, /* bad enum value or a shape the kernels do not cover  */
  FP8BQ_ERR_ARCH = 5,        /* current device is not compute capability 10.3       */
  FP8BQ_ERR_WORKSPACE = 6,   /* workspace NULL or smaller than required             */
  FP8BQ_ERR_CUDA = 7,        /* a CUDA runtime call failed; see fp8bq_last_cuda_error */
  FP8BQ_ERR_TIMEOUT = 8,     /* a device wait gave up (reported by fp8bq_poll_status) */
  FP8BQ_ERR_BOUNDS = 9       /* debug builds only: a GEMM epilogue write fell outside its
                                buffer and was skipped (reported by fp8bq_poll_status) */
} fp8bq_status;

enum { FP8BQ_SCALE_ROW_MAJOR = 0, FP8BQ_SCALE_COL_MAJOR = 1 };

/* Operation ids for fp8bq_workspace_bytes. */
enum {
  FP8BQ_OP_GEMM = 0,
  FP8BQ_OP_LINEAR = 1,
  FP8BQ_OP_MX_GEMM = 2,
  FP8BQ_OP_MX_LINEAR = 3,
  FP8BQ_OP_STATIC_GEMM = 4,
  FP8BQ_OP_STATIC_LINEAR = 5,
  FP8BQ_OP_CHANNEL_GEMM = 6,
  FP8BQ_OP_CHANNEL_LINEAR = 7,
  FP8BQ_OP_UE8M0_GEMM = 8,
  FP8BQ_OP_UE8M0_LINEAR = 9,
  FP8BQ_OP_GROUPED_GEMM = 10 /* both grouped forms; M = rows of A and Y in all */
};

/* ---------------------------------------------------------------- utility
 * Library plumbing with no counterpart on the pages (there, the framework
 * owns memory and streams): version, status strings, workspace sizing and
 * the status word that the bounded device waits report through. */

/* Library version, major*10000 + minor*100 + patch. */
FP8BQ_API int fp8bq_version(void);

/* Static string for a status code ("unknown status" for other values). */
FP8BQ_API const char *fp8bq_status_string(int status);

/* cudaError_t of the last FP8BQ_ERR_CUDA returned on the calling thread (0 if none). */
FP8BQ_API int fp8bq_last_cuda_error(void);

/* Workspace bytes needed by `op` at this shape (a multiple of 256; never 0). */
FP8BQ_API size_t fp8bq_workspace_bytes(int op, int64_t M, int64_t N, int64_t K);

/* Zeroes `ws_bytes` bytes of a workspace on `stream` (required once before first use). */
FP8BQ_API int fp8bq_workspace_init(void *ws, size_t ws_bytes, void *stream);

/* Synchronises `stream`, then returns and clears the workspace status word:
 * FP8BQ_OK, or FP8BQ_ERR_TIMEOUT if a kernel's bounded wait ran out, or (a
 * library built with FP8BQ_DEBUG_CHECKS) FP8BQ_ERR_BOUNDS if a GEMM's bounds
 * check skipped a write. */
FP8BQ_API int fp8bq_poll_status(void *ws, void *stream);

/* ------------------------------------------------ block path (group/block 128) */

/* Per-token group-128 activation quantisation (per_token_group_quant_fp8):
 * "GLM-5.3 推理全链路(十七)", §第1站 (s_g = max|x| / 448 per group of 128
 * channels, q = round(x / s_g)) and "SGLang 源码完全拆解(十九)", §从浮点到 FP8
 * 的基本公式 (clamp to +-448, round to nearest even).
 * x: BF16 [M, K] pitch ldx.  q: E4M3 [M, K].  s: FP32 scales in `s_layout`.
 * Bit-exact rule: amax = max|x| over the group (floored at 1e-10),
 * s = amax / 448 and q = RNE_sat(x / s), both IEEE binary32 divisions.
 * Errors: ERR_NULL (q or s NULL), ERR_SHAPE, ERR_ALIGN (x, q not 16-byte
 * aligned, ldx % 8, K % 16), ERR_UNSUPPORTED (layout value). */
FP8BQ_API int fp8bq_quant_act(const void *x, int64_t M, int64_t K, int64_t ldx,
                              void *q, float *s, int s_layout, void *stream);

/* Block-scaled FP8 GEMM: y = BF16(sum_b P_b * s_x[:, b] * s_w[n/128, b] + bias),
 * P_b the FP32 tensor-core sum over K block b -- "SGLang 源码完全拆解(十九)",
 * §一条 GEMM 的三种缩放组合 (the block-wise equation) and §Triton 分块内核在
 * 做什么 (one scale read per K block and tile, dequantisation in the
 * epilogue); "GLM-5.3 推理全链路(十七)", §先把 GLM-5.3 的数值常量摆出来 (FP32
 * promotion of every 128-wide K slice, the DeepSeek-V3 Fig. 7 scheme).
 * q: E4M3 [M, K]; s_x in `s_layout`; w: E4M3 [N, K]; s_w: FP32
 * [ceil(N/128)][ceil(K/128)]; bias: BF16 [N] or NULL; y: BF16 [M, N].
 * Errors: ERR_NULL, ERR_SHAPE, ERR_ALIGN, ERR_UNSUPPORTED (layout value, or
 * K > 65536 when M <= 64), ERR_WORKSPACE, ERR_CUDA; a
 * timed-out device wait is reported later by fp8bq_poll_status. */
FP8BQ_API int fp8bq_gemm(const void *q, const float *s_x, int s_layout,
                         const void *w, const float *s_w, const void *bias,
                         void *y, int64_t M, int64_t N, int64_t K, void *ws,
                         size_t ws_bytes, void *stream);

/* Fused linear, BF16 in and BF16 out ("SGLang 源码完全拆解(十九)", §一次前向的
 * 完整时序: quantise the activations, block-scaled GEMM, bias, output dtype):
 * the result of fp8bq_quant_act (row-major scales) followed by fp8bq_gemm,
 * bit for bit.  Up to 16 tokens it is one launch: the GEMM quantises the
 * activations of each K block itself as they arrive; above, the quantiser
 * writes codes and scales into the workspace first.  Arguments and errors as
 * fp8bq_quant_act and fp8bq_gemm; workspace fp8bq_workspace_bytes(FP8BQ_OP_LINEAR, ...). */
FP8BQ_API int fp8bq_linear(const void *x, int64_t ldx, const void *w,
                           const float *s_w, const void *bias, void *y,
                           int64_t M, int64_t N, int64_t K, void *ws,
                           size_t ws_bytes, void *stream);

/* Size of the fixed scratch array behind fp8bq_gemm_noalloc (16 MiB per device). */
#define FP8BQ_NOALLOC_SCRATCH_BYTES (16u * 1024u * 1024u)

/* fp8bq_gemm without a caller workspace.  The pages have no counterpart: this
 * entry point exists for callers that cannot hand the library device memory of
 * its own -- an operator interface whose argument list is fixed and has no
 * room for a workspace, or a runtime that plans all device memory ahead of time
 * and forbids allocations (cudaMalloc, a framework's caching allocator) inside
 * its operators.  Arguments, layouts, checks and results are those of
 * fp8bq_gemm; the caller still owns q, s_x, w, s_w, bias and y.
 *
 * In place of `ws` it uses one array of FP8BQ_NOALLOC_SCRATCH_BYTES that the
 * library holds in device memory on every GPU that loads it, until the process
 * exits; it calls no allocating routine.
 *  - Limit: the scratch holds the workspace of fp8bq_gemm at this shape
 *    without the split tail tiles' partials (below), and shapes that need more
 *    than FP8BQ_NOALLOC_SCRATCH_BYTES are rejected with FP8BQ_ERR_WORKSPACE
 *    before anything is launched.  For M > 64 that is a status word and one
 *    counter per 128 output columns (at least 160), so every N up to about
 *    5 * 10^8 fits; for M <= 64 it adds FP32 split-K partials (32 *
 *    round_up(M, 4) * N bytes), so round_up(M, 4) * N must stay below about
 *    524,000: every M <= 64 at N = 6144, M <= 16 at N = 24576.  Without the partials, the last wave's
 *    tiles run whole: results agree with fp8bq_gemm's within the GEMM
 *    tolerance, not bit for bit.
 *  - Set-up: the first call on a device, with that device current, looks up
 *    the array's device address (cudaGetSymbolAddress) and keeps it; make that
 *    first call before any stream capture begins.  A failed look-up returns
 *    FP8BQ_ERR_CUDA then and on every later call on that device.
 *  - Each call clears the array's status word and split-K counters on `stream`
 *    (cudaMemsetAsync) before its kernel.  Every call on a device shares the one
 *    array, which keeps what the last call left there: calls that may overlap
 *    on the GPU (different streams without ordering between them) race on it
 *    and give undefined results.  Calls on one stream are ordered and safe.
 *  - A device-side wait that runs out leaves the outputs undefined and sets
 *    the array's status word; fp8bq_noalloc_poll_status reports it (the next
 *    call clears it in any case). */
FP8BQ_API int fp8bq_gemm_noalloc(const void *q, const float *s_x, int s_layout,
                                 const void *w, const float *s_w,
                                 const void *bias, void *y, int64_t M,
                                 int64_t N, int64_t K, void *stream);

/* The status of the fp8bq_gemm_noalloc calls on the current device: synchronises
 * `stream`, then returns and clears the scratch array's status word -- FP8BQ_OK,
 * or FP8BQ_ERR_TIMEOUT if a bounded device wait of one of those calls ran out
 * (its output is then undefined).  No counterpart on the pages; it allocates
 * nothing.  Like fp8bq_gemm_noalloc, the first call on a device looks up the
 * array's address. */
FP8BQ_API int fp8bq_noalloc_poll_status(void *stream);

/* ------------------------------------------------ MXFP8 path ([1,32], UE8M0) */

/* MXFP8 activation quantisation ("SGLang 源码完全拆解(十九)", §checkpoint 里的
 * 量化元数据 and "[SGLang] FP8" §1: blocks of [1, 32]; "GLM-5.3 推理全链路(十七)",
 * §第4站: the E8M0 exponent rounded up, amax floored at 1e-10): per 32-channel
 * group, e = ceil(log2(max(amax, 1e-10) / 448)) (binary32 division),
 * s = e + 127 (UE8M0), q = RNE_sat(x * 2^-e).  s: uint8 [M][K/32].  Also
 * quantises weights (rows = N).  K % 32 == 0 (ERR_ALIGN otherwise). */
FP8BQ_API int fp8bq_mx_quant_act(const void *x, int64_t M, int64_t K,
                                 int64_t ldx, void *q, uint8_t *s,
                                 void *stream);

/* MXFP8 GEMM on the tensor cores' block-scaled MMA ("GLM-5.3 推理全链路(十七)",
 * §第7站: the UE8M0 scales are consumed by the MMA itself): s_x uint8
 * [M][K/32], s_w uint8 [N][K/32]; y = BF16(sum_g P_g * 2^(s_x-127) *
 * 2^(s_w-127) + bias).  Workspace fp8bq_workspace_bytes(FP8BQ_OP_MX_GEMM, ...)
 * (it holds the scale codes rearranged for the MMA).  Errors as fp8bq_gemm. */
FP8BQ_API int fp8bq_mx_gemm(const void *q, const uint8_t *s_x, const void *w,
                            const uint8_t *s_w, const void *bias, void *y,
                            int64_t M, int64_t N, int64_t K, void *ws,
                            size_t ws_bytes, void *stream);

/* Fused MXFP8 linear (the same page sequence as fp8bq_linear with the MXFP8
 * formats): fp8bq_mx_quant_act into the workspace, then fp8bq_mx_gemm. */
FP8BQ_API int fp8bq_mx_linear(const void *x, int64_t ldx, const void *w,
                              const uint8_t *s_w, const void *bias, void *y,
                              int64_t M, int64_t N, int64_t K, void *ws,
                              size_t ws_bytes, void *stream);

/* ------------------------------------------------ residual add + RMSNorm + quant */

/* The step before the linear's activation quantiser, fused with it
 * ("GLM-5.3 推理全链路(十七)", §第1站 RMSNorm 的两个出口: residual add, RMSNorm
 * y = x / sqrt(mean(x^2) + eps) * g with the sum and the root in FP32, BF16 out;
 * the static per-tensor path fuses the quantisation into the same launch):
 *   r = BF16(x + residual)          (residual == NULL: r = x)
 *   S = sum_k r_k^2, the exact sum rounded once to binary32
 *   rms = sqrt(RN32(RN32(S / K) + eps))          (IEEE binary32 operations)
 *   y_k = BF16(RN32(RN32(r_k / rms) * gamma_k))
 * then q, s = the group-128 quantisation of y (fp8bq_quant_act's rule), bit for
 * bit the same as quantising a separately written y.
 * x: BF16 [M, K] pitch ldx; residual: BF16 [M, K] pitch ld_res or NULL;
 * residual_out: BF16 [M, K] (contiguous) or NULL -- it may be the residual
 * buffer itself (in place) when ld_res == K, no other outputs may overlap an
 * input; gamma: BF16 [K]; eps: finite, >= 0; y: BF16 [M, K] or NULL.  q: E4M3
 * [M, K] and s: FP32 scales in `s_layout`, or q == NULL for the norm alone.
 * K % 16 == 0, K <= 16384; every pointer 16-byte aligned (s: 4). */
FP8BQ_API int fp8bq_add_rmsnorm_quant_act(const void *x, int64_t ldx,
                                          const void *residual, int64_t ld_res,
                                          void *residual_out, const void *gamma,
                                          float eps, int64_t M, int64_t K, void *y,
                                          void *q, float *s, int s_layout,
                                          void *stream);

/* As fp8bq_add_rmsnorm_quant_act, then static per-tensor quantisation of y with
 * the device-resident scale s_x[0] (fp8bq_static_quant_act's rule) into q. */
FP8BQ_API int fp8bq_add_rmsnorm_static_quant_act(const void *x, int64_t ldx,
                                                 const void *residual, int64_t ld_res,
                                                 void *residual_out, const void *gamma,
                                                 float eps, const float *s_x, int64_t M,
                                                 int64_t K, void *y, void *q,
                                                 void *stream);

/* ------------------------------------------------ static per-tensor path */

/* Static per-tensor quantisation ("SGLang 源码完全拆解(十九)", §激活量化的三种选择:
 * one calibrated scale for the whole tensor; "[SGLang] FP8" §5) with one
 * device-resident FP32 scale s_x[0]: q = RNE_sat(x / s_x), binary32 division;
 * values beyond 448 s_x saturate.  Errors: ERR_NULL, ERR_SHAPE, ERR_ALIGN. */
FP8BQ_API int fp8bq_static_quant_act(const void *x, int64_t M, int64_t K,
                                     int64_t ldx, const float *s_x, void *q,
                                     void *stream);

/* Per-tensor FP8 GEMM ("SGLang 源码完全拆解(十九)", §一条 GEMM 的三种缩放组合: the
 * per-tensor scales come out of the sum; "[SGLang] FP8" §5: one weight scale
 * per output partition of a fused weight): y = BF16((sum_k q w) * s_x[0] *
 * s_w_part[p(j)] + bias), p(j) the output partition of row j.
 * part_sizes_host[n_parts] (host memory, 1 <= n_parts <= 64) must sum to N
 * (ERR_SHAPE otherwise); s_w_part is a device FP32 [n_parts]. */
FP8BQ_API int fp8bq_static_gemm(const void *q, const float *s_x, const void *w,
                                const float *s_w_part,
                                const int64_t *part_sizes_host, int n_parts,
                                const void *bias, void *y, int64_t M, int64_t N,
                                int64_t K, void *ws, size_t ws_bytes,
                                void *stream);

/* Fused static linear ("GLM-5.3 推理全链路(十七)", §第1站: the static per-tensor
 * path multiplies by the fixed FP8 scale): fp8bq_static_quant_act into the
 * workspace, then fp8bq_static_gemm. */
FP8BQ_API int fp8bq_static_linear(const void *x, int64_t ldx, const float *s_x,
                                  const void *w, const float *s_w_part,
                                  const int64_t *part_sizes_host, int n_parts,
                                  const void *bias, void *y, int64_t M,
                                  int64_t N, int64_t K, void *ws,
                                  size_t ws_bytes, void *stream);

/* ------------------------------------------------ channelwise path (W8A8) */

/* Per-token dynamic quantisation: one FP32 scale per row,
 * s[i] = max(max_k |x[i,k]|, 1e-10) / 448 and q = RNE_sat(x / s[i]) (binary32
 * divisions) -- the group rule with the group spanning the row ("SGLang
 * 源码完全拆解(十九)", §激活量化的三种选择, sglang_per_token_quant_fp8).  Applied to a
 * BF16 weight [N, K] it gives the per-channel weight scales (§装载后的三个分支:
 * per_token_group_quant_fp8 with group_size = K).  x: BF16 [M, K] pitch ldx;
 * q: E4M3 [M, K]; s: FP32 [M].  K % 16 == 0. */
FP8BQ_API int fp8bq_channel_quant_act(const void *x, int64_t M, int64_t K,
                                      int64_t ldx, void *q, float *s,
                                      void *stream);

/* Channelwise GEMM: y[i, j] = BF16((sum_k q[i,k] w[j,k]) * s_x[i] * s_w[j] + bias[j])
 * (§一条 GEMM 的三种缩放组合, the per-token x per-channel outer product of the
 * scales, applied after the FP32 full-K sum).  s_x: FP32 [M]; s_w: FP32 [N]. */
FP8BQ_API int fp8bq_channel_gemm(const void *q, const float *s_x, const void *w,
                                 const float *s_w, const void *bias, void *y,
                                 int64_t M, int64_t N, int64_t K, void *ws,
                                 size_t ws_bytes, void *stream);

/* Fused channelwise linear: fp8bq_channel_quant_act into the workspace, then
 * fp8bq_channel_gemm. */
FP8BQ_API int fp8bq_channel_linear(const void *x, int64_t ldx, const void *w,
                                   const float *s_w, const void *bias, void *y,
                                   int64_t M, int64_t N, int64_t K, void *ws,
                                   size_t ws_bytes, void *stream);

/* ------------------------------------------------ block FP8 with UE8M0 scales */

/* Group-128 activation quantisation with power-of-two scales ("SGLang 源码完全
 * 拆解(十九)", §分块 GEMM 的后端分派: act_scale_ue8m0 keeps the per-token-group
 * layout and limits each scale to 2^e): e = ceil(log2(max(amax, 1e-10) / 448))
 * with the binary32 division, u = e + 127, q = RNE_sat(x * 2^-e).
 * u: uint8 [M][ceil(K/128)]. */
FP8BQ_API int fp8bq_quant_act_ue8m0(const void *x, int64_t M, int64_t K,
                                    int64_t ldx, void *q, uint8_t *u,
                                    void *stream);

/* One-time weight preparation (§分块路径的后处理:
 * FP32 block scales requantised to power-of-two UE8M0 for the block-scaled
 * MMA): per 128 x 128 block, s' = 2^ceil(log2 s) (s > 0 finite), u_w = the code
 * of s', and every code re-encoded, q' = RNE_sat(dec(q) * s / s') (exact in
 * binary64, one rounding).  q: E4M3 [N, K]; s_w: FP32 [ceil(N/128)][ceil(K/128)];
 * q_out: E4M3 [N, K] (may be q); u_w: uint8, the shape of s_w. */
FP8BQ_API int fp8bq_requant_weight_ue8m0(const void *q, const float *s_w,
                                         int64_t N, int64_t K, void *q_out,
                                         uint8_t *u_w, void *stream);

/* Block FP8 GEMM with UE8M0 128 x 128 block scales, run as an MXFP8 view on the
 * block-scaled MMA (each code standing for four 32-groups): y = BF16(sum_b P_b *
 * 2^(u_x[i][b]-127) * 2^(u_w[j/128][b]-127) + bias), FP32 accumulation over the
 * whole K inside the MMA.  u_x: uint8 [M][ceil(K/128)]; u_w: uint8
 * [ceil(N/128)][ceil(K/128)].  K % 32 == 0. */
FP8BQ_API int fp8bq_ue8m0_gemm(const void *q, const uint8_t *u_x, const void *w,
                               const uint8_t *u_w, const void *bias, void *y,
                               int64_t M, int64_t N, int64_t K, void *ws,
                               size_t ws_bytes, void *stream);

/* Fused: fp8bq_quant_act_ue8m0 into the workspace, then fp8bq_ue8m0_gemm. */
FP8BQ_API int fp8bq_ue8m0_linear(const void *x, int64_t ldx, const void *w,
                                 const uint8_t *u_w, const void *bias, void *y,
                                 int64_t M, int64_t N, int64_t K, void *ws,
                                 size_t ws_bytes, void *stream);

/* ------------------------------------------------ grouped (MoE) block FP8 */

/* Block-scaled FP8 GEMM over E experts at once ("SGLang 源码完全拆解(十九)",
 * §MoE:专家权重多一个维度: expert weights carry a leading expert dimension,
 * w [E, N, K] with one FP32 128 x 128 scale grid per expert, s_w
 * [E][ceil(N/128)][ceil(K/128)]; the grouped GEMM takes the activation rows
 * sorted by expert, a contiguous layout that the dispatch step produces).
 * Rows offsets[e] .. offsets[e+1]-1 of q, s_x and y belong to expert e:
 *
 *   y[i][j] = BF16(sum_b P_b * s_x[i][b] * s_w[e][j/128][b]),  e the expert of row i,
 *
 * with the arithmetic of fp8bq_gemm.  q: E4M3 [M, K] (the M sorted rows);
 * s_x: FP32 [M][ceil(K/128)] or column-major [ceil(K/128)][round_up(M,4)];
 * y: BF16 [M, N].  offsets: DEVICE int32 [E+1], non-decreasing, offsets[0] >= 0,
 * offsets[E] <= M; it is read by the kernel (written, e.g., by a routing
 * kernel earlier on the stream), so the host never synchronises.  Rows outside
 * every segment are not written.  Bounds outside [0, M] are clamped on the
 * device; decreasing offsets make overlapping segments, whose rows then get
 * unspecified values (nothing outside q, s_x, w, s_w, y is accessed).
 * 1 <= E <= 1024, E * N < 2^31.  No bias (the pages' expert weights carry
 * none).  For a fused gate/up weight with intermediate size I_p per shard the
 * scale rows follow j/128, which is the pages' per-shard rounding when I_p is a
 * multiple of 128; otherwise pad each shard to a multiple of 128 rows.
 * Workspace: fp8bq_workspace_bytes(FP8BQ_OP_GROUPED_GEMM, M, N, K). */
FP8BQ_API int fp8bq_grouped_gemm(const void *q, const float *s_x, int s_layout,
                                 const void *w, const float *s_w,
                                 const int32_t *offsets, int64_t E, void *y,
                                 int64_t M, int64_t N, int64_t K, void *ws,
                                 size_t ws_bytes, void *stream);

/* The masked form of the same GEMM: A is [E, max_m, K] (rows e * max_m ..
 * e * max_m + masked_m[e] - 1 are expert e's, the rest of each slot unused),
 * y [E, max_m, N], s_x over the E * max_m rows as above.  masked_m: DEVICE
 * int32 [E], each clamped to [0, max_m] on the device.  Unused rows are not
 * written.  Workspace: fp8bq_workspace_bytes(FP8BQ_OP_GROUPED_GEMM,
 * E * max_m, N, K). */
FP8BQ_API int fp8bq_grouped_gemm_masked(const void *q, const float *s_x,
                                        int s_layout, const void *w,
                                        const float *s_w,
                                        const int32_t *masked_m, int64_t E,
                                        int64_t max_m, void *y, int64_t N,
                                        int64_t K, void *ws, size_t ws_bytes,
                                        void *stream);

/* ------------------------------------------------ weight / calibration set-up */

/* 128x128 block quantisation of a BF16 weight [N, K] (pitch ldw) into E4M3
 * [N, K] and FP32 s_w [ceil(N/128)][ceil(K/128)]; a partial edge block uses
 * only its valid elements.  Same arithmetic as fp8bq_quant_act. */
FP8BQ_API int fp8bq_quant_weight_block(const void *w, int64_t N, int64_t K,
                                       int64_t ldw, void *q, float *s_w,
                                       void *stream);

/* One per-tensor scale s[0] = max(max|x|, 1e-10) / 448 over a BF16 [rows, K]
 * matrix (pitch ldx): a calibration batch, or one weight partition. */
FP8BQ_API int fp8bq_absmax_scale(const void *x, int64_t rows, int64_t K,
                                 int64_t ldx, float *s, void *stream);

/* Debug helper for scales that come from outside the library (a checkpoint,
 * a caller's calibration): classifies the entries of a device FP32 scale array
 * that are not usable dequantisation multipliers.  "SGLang 源码完全拆解(十九)",
 * §scale 的初始值不是零: every scale is registered at the sentinel
 * torch.finfo(float32).min and only a checkpoint entry overwrites it, so a
 * scale still holding the sentinel was never loaded.
 *   counts_host[0]  entries equal to the sentinel -FLT_MAX (bits 0xff7fffff)
 *   counts_host[1]  NaN or infinite entries
 *   counts_host[2]  other entries <= 0 (zero, -0 or negative multipliers)
 *   *first_bad_host the smallest index in any class, or -1
 * s: n FP32 values (any layout; n >= 0; s may be NULL when n == 0).  scratch:
 * 32 bytes of device memory, 8-byte aligned, overwritten.  Host outputs are
 * written after the call synchronises `stream`.  No GEMM entry point calls
 * this: the check is for loading time, not the forward path. */
FP8BQ_API int fp8bq_check_scales(const float *s, int64_t n, void *scratch,
                                 int64_t *counts_host, int64_t *first_bad_host,
                                 void *stream);

/* Test helper for the conversion every quantiser ends with: codes[i] = the
 * E4M3 code of the binary32 value whose bit pattern is first + i (0 <= i < n,
 * first + n <= 2^32), from the same saturating round-to-nearest-even hardware
 * conversion the quantisers apply to their quotients ("SGLang 源码完全拆解(十九)",
 * §从浮点到 FP8 的基本公式: q = clamp(round(x/s), -448, 448), RNE; |v| >= 448
 * and infinities give +-448).  Lets a test compare the conversion with an
 * independent encoder over all 2^32 inputs.  codes: device uint8 [n], 8-byte
 * aligned.  FP8BQ_ERR_SHAPE for n < 0 or a range past 2^32 - 1. */
FP8BQ_API int fp8bq_e4m3_from_bits(uint32_t first, int64_t n, uint8_t *codes, void *stream);

#ifdef __cplusplus
}
#endif
#endif /* FP8BQ_H */
