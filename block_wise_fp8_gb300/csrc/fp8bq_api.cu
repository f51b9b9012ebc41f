// fp8bq_api.cu -- the C ABI (include/fp8bq.h): host-side validation, per-device
// attribute cache, workspace bookkeeping and kernel launches.  Nothing here
// computes on the host; every step of the path runs in the kernels of quant.cu
// and gemm_*.cu.
#include <cuda_runtime.h>

#include <atomic>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "../../include/fp8bq.h"
#include "common.cuh"

using namespace fp8bq;

namespace {

thread_local int g_last_cuda_error = 0;

constexpr int kMaxDevices = 64;
struct DevSlot {
  std::once_flag once;
  DeviceInfo info;
  cudaError_t err;
};
DevSlot g_dev[kMaxDevices];

uint64_t wait_limit_ns() {
  static uint64_t v = [] {
    uint64_t ms = 1000;
    if (const char *e = std::getenv("FP8BQ_WAIT_LIMIT_MS")) {
      char *end = nullptr;
      unsigned long long x = std::strtoull(e, &end, 10);
      if (end != e && x > 0) ms = x;
    }
    return ms * 1000000ull;
  }();
  return v;
}

// Fault injection for the timeout tests, off unless the environment (read
// once) has FP8BQ_FAULT_INJECT=skip_first_load:<n>: then CTA 0 of each of the
// next n GEMM launches issues no copy for its first K block, the waits on that
// stage run out after the wait limit, and the GEMM reports FP8BQ_ERR_TIMEOUT
// through the workspace status word.  Later launches run normally.
int fault_skip_first_load() {
  static std::atomic<long> remaining{[] {
    const char *e = std::getenv("FP8BQ_FAULT_INJECT");
    const char *key = "skip_first_load:";
    if (!e || std::strncmp(e, key, std::strlen(key)) != 0) return 0L;
    return std::strtol(e + std::strlen(key), nullptr, 10);
  }()};
  if (remaining.load(std::memory_order_relaxed) <= 0) return 0;
  return remaining.fetch_sub(1) > 0 ? 1 : 0;
}

int cuda_fail(cudaError_t e) {
  g_last_cuda_error = static_cast<int>(e);
  return FP8BQ_ERR_CUDA;
}

// Current device must be compute capability 10.3 (GB300).
int device_info(DeviceInfo *out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e);
  if (dev < 0 || dev >= kMaxDevices) return FP8BQ_ERR_ARCH;
  DevSlot &s = g_dev[dev];
  std::call_once(s.once, [&] {
    s.err = cudaSuccess;
    int v = 0;
    cudaError_t r;
    if ((r = cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) s.err = r;
    s.info.num_sms = v;
    if ((r = cudaDeviceGetAttribute(&v, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess) s.err = r;
    s.info.cc_major = v;
    if ((r = cudaDeviceGetAttribute(&v, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess) s.err = r;
    s.info.cc_minor = v;
    if ((r = cudaDeviceGetAttribute(&v, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev)) != cudaSuccess) s.err = r;
    s.info.max_smem_optin = static_cast<size_t>(v);
  });
  if (s.err != cudaSuccess) return cuda_fail(s.err);
  if (s.info.cc_major != 10 || s.info.cc_minor != 3) return FP8BQ_ERR_ARCH;
  *out = s.info;
  return FP8BQ_OK;
}

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

// Common checks for an activation matrix [M, K] with pitch ldx.
int check_act(const void *x, int64_t M, int64_t K, int64_t ldx, int kmod) {
  if (!x) return FP8BQ_ERR_NULL;
  if (M < 0 || K < 1 || ldx < K || M > (int64_t(1) << 31) - 1 || K > (int64_t(1) << 30))
    return FP8BQ_ERR_SHAPE;
  if (!aligned(x, 16) || (ldx % 8) != 0 || (K % kmod) != 0) return FP8BQ_ERR_ALIGN;
  return FP8BQ_OK;
}

int check_gemm_shape(int64_t M, int64_t N, int64_t K, int kmod) {
  if (M < 0 || N < 1 || K < 1) return FP8BQ_ERR_SHAPE;
  if (M > (int64_t(1) << 31) - 1 || N > (int64_t(1) << 31) - 1 || K > (int64_t(1) << 30))
    return FP8BQ_ERR_SHAPE;
  if (K % kmod) return FP8BQ_ERR_ALIGN;
  return FP8BQ_OK;
}

int check_ws(void *ws, size_t ws_bytes, int op, int64_t M, int64_t N, int64_t K) {
  if (!ws) return FP8BQ_ERR_WORKSPACE;
  if (!aligned(ws, 256)) return FP8BQ_ERR_ALIGN;
  if (ws_bytes < workspace_layout(op, M, N, K).total) return FP8BQ_ERR_WORKSPACE;
  return FP8BQ_OK;
}

// `tail`: the workspace holds the split tail tiles' partials (every caller
// workspace does; the fixed scratch of fp8bq_gemm_noalloc does not)
GemmArgs base_args(int mode, int64_t M, int64_t N, int64_t K, const void *bias, void *y,
                   void *ws, int op, bool tail = true) {
  GemmArgs a;
  std::memset(&a, 0, sizeof a);
  a.mode = mode;
  a.M = static_cast<int>(M);
  a.N = static_cast<int>(N);
  a.K = static_cast<int>(K);
  a.bias = bias;
  a.y = y;
  const WorkspaceLayout L = workspace_layout(op, M, N, K, tail);
  uint8_t *w = static_cast<uint8_t *>(ws);
  a.status = reinterpret_cast<uint32_t *>(w + L.status);
  a.counters = reinterpret_cast<uint32_t *>(w + L.counters);
  a.partials = reinterpret_cast<float *>(w + L.partials);
  a.partials_bytes = static_cast<int64_t>(L.q - L.partials);
  a.wait_limit_ns = wait_limit_ns();
  a.fault_skip_first_load = fault_skip_first_load();
  return a;
}

int finish_launch(int st, cudaError_t e) {
  if (st != 0) return st;
  if (e != cudaSuccess) return cuda_fail(e);
  return FP8BQ_OK;
}

#define RETURN_IF(x)            \
  do {                          \
    int _r = (x);               \
    if (_r != FP8BQ_OK) return _r; \
  } while (0)

// ------------------------------------------------------------------ shared bodies

int gemm_block_impl(const void *q, const float *s_x, int s_layout, const void *w,
                    const float *s_w, const void *bias, void *y, int64_t M, int64_t N, int64_t K,
                    void *ws, int op, cudaStream_t st, const DeviceInfo &dev, bool tail = true) {
  GemmArgs a = base_args(kModeBlock, M, N, K, bias, y, ws, op, tail);
  a.sx = s_x;
  a.sx_layout = s_layout;
  a.ldsx = s_layout == FP8BQ_SCALE_ROW_MAJOR ? static_cast<int>((K + 127) / 128)
                                             : static_cast<int>((M + 3) / 4 * 4);
  a.sw = s_w;
  cudaError_t e;
  int r = launch_gemm(a, q, w, dev, st, &e);
  return finish_launch(r, e);
}

// MXFP8 GEMM; `block128`: the scale codes are one per 128-wide K block (and per
// 128 weight rows), the block-FP8-with-UE8M0 view of the same kernel.
int gemm_mx_impl(const void *q, const uint8_t *s_x, const void *w, const uint8_t *s_w,
                 const void *bias, void *y, int64_t M, int64_t N, int64_t K, void *ws, int op,
                 cudaStream_t st, const DeviceInfo &dev, bool block128 = false) {
  GemmArgs a = base_args(kModeMx, M, N, K, bias, y, ws, op);
  const WorkspaceLayout L = workspace_layout(op, M, N, K);
  uint8_t *sfa = static_cast<uint8_t *>(ws) + L.sfa;
  uint8_t *sfb = static_cast<uint8_t *>(ws) + L.sfb;
  if (block128) launch_ue8m0_sf_tiles(s_x, M, s_w, N, K, sfa, sfb, dev.num_sms, st);
  else launch_mx_sf_tiles(s_x, M, s_w, N, K, sfa, sfb, dev.num_sms, st);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e);
  a.ux = sfa;  // the GEMM reads the chunks
  a.uw = sfb;
  int r = launch_gemm(a, q, w, dev, st, &e);
  return finish_launch(r, e);
}

int gemm_channel_impl(const void *q, const float *s_x, const void *w, const float *s_w,
                      const void *bias, void *y, int64_t M, int64_t N, int64_t K, void *ws, int op,
                      cudaStream_t st, const DeviceInfo &dev) {
  GemmArgs a = base_args(kModeChannel, M, N, K, bias, y, ws, op);
  a.sx = s_x;
  a.sw = s_w;
  cudaError_t e;
  int r = launch_gemm(a, q, w, dev, st, &e);
  return finish_launch(r, e);
}

int gemm_static_impl(const void *q, const float *s_x, const void *w, const float *s_w_part,
                     const int64_t *parts, int n_parts, const void *bias, void *y, int64_t M,
                     int64_t N, int64_t K, void *ws, int op, cudaStream_t st,
                     const DeviceInfo &dev) {
  GemmArgs a = base_args(kModeTensor, M, N, K, bias, y, ws, op);
  a.sx_scalar = s_x;
  a.sw_part = s_w_part;
  a.n_parts = n_parts;
  int64_t end = 0;
  for (int p = 0; p < n_parts; ++p) {
    end += parts[p];
    a.part_end[p] = static_cast<int>(end);
  }
  cudaError_t e;
  int r = launch_gemm(a, q, w, dev, st, &e);
  return finish_launch(r, e);
}

// An empty batch (M == 0) launches nothing; only the other extents are checked
// and pointers may be NULL.
// Grouped block-scaled GEMM over E experts.  The segment bounds stay on the
// device (the routing kernel that wrote them ran on the stream before); the
// launcher bounds the tiles they can hold from E, M and max_m alone.
int gemm_grouped_impl(const void *q, const float *s_x, int s_layout, const void *w,
                      const float *s_w, const int32_t *offsets, const int32_t *masked_m,
                      int64_t E, int64_t max_m, void *y, int64_t M, int64_t N, int64_t K, void *ws,
                      cudaStream_t st, const DeviceInfo &dev) {
  GemmArgs a = base_args(kModeBlock, M, N, K, nullptr, y, ws, FP8BQ_OP_GROUPED_GEMM);
  a.sx = s_x;
  a.sx_layout = s_layout;
  a.ldsx = s_layout == FP8BQ_SCALE_ROW_MAJOR ? static_cast<int>((K + 127) / 128)
                                             : static_cast<int>((M + 3) / 4 * 4);
  a.sw = s_w;
  a.g_experts = static_cast<int>(E);
  a.g_offsets = offsets;
  a.g_masked = masked_m;
  a.g_max_m = static_cast<int>(max_m);
  cudaError_t e;
  int r = launch_gemm(a, q, w, dev, st, &e);
  return finish_launch(r, e);
}

// Checks shared by both grouped forms (M rows of A and Y in all).
int check_grouped(const void *q, const float *s_x, int s_layout, const void *w, const float *s_w,
                  const void *bounds, int64_t E, int64_t M, int64_t N, int64_t K, int64_t cap,
                  void *y) {
  if (!q || !s_x || !w || !s_w || !bounds || !y) return FP8BQ_ERR_NULL;
  RETURN_IF(check_gemm_shape(M, N, K, 16));
  if (E < 1 || E > kMaxExperts) return FP8BQ_ERR_SHAPE;
  // expert rows E * N and (128-row) tile counts x weight tiles stay 32-bit
  if (E * N > (int64_t(1) << 31) - 1 || cap * ((N + 255) / 256) > (int64_t(1) << 31) - 1)
    return FP8BQ_ERR_SHAPE;
  if (s_layout != FP8BQ_SCALE_ROW_MAJOR && s_layout != FP8BQ_SCALE_COL_MAJOR)
    return FP8BQ_ERR_UNSUPPORTED;
  if (!aligned(q, 16) || !aligned(w, 16) || !aligned(y, 16) || !aligned(s_x, 4) ||
      !aligned(s_w, 4) || !aligned(bounds, 4))
    return FP8BQ_ERR_ALIGN;
  return FP8BQ_OK;
}

int empty_batch(int64_t K, int64_t N) { return (K >= 1 && N >= 1) ? FP8BQ_OK : FP8BQ_ERR_SHAPE; }

int check_parts(const int64_t *parts, int n_parts, int64_t N) {
  if (!parts) return FP8BQ_ERR_NULL;
  if (n_parts < 1 || n_parts > kMaxParts) return FP8BQ_ERR_SHAPE;
  int64_t sum = 0;
  for (int p = 0; p < n_parts; ++p) {
    if (parts[p] < 1) return FP8BQ_ERR_SHAPE;
    sum += parts[p];
  }
  return sum == N ? FP8BQ_OK : FP8BQ_ERR_SHAPE;
}

}  // namespace

// ------------------------------------------------------------------ no-allocation scratch
//
// Scratch of fp8bq_gemm_noalloc: a fixed array in this library's device image.
// Each device gets its own copy when the library's module is loaded on it, and
// keeps it until the process exits.  On the host this name is only a handle
// for cudaGetSymbolAddress, never an address to pass to a kernel.
static __device__ __align__(256) uint8_t fp8bq_noalloc_scratch[FP8BQ_NOALLOC_SCRATCH_BYTES];

namespace {

struct ScratchSlot {
  std::once_flag once;
  void *ptr;
  cudaError_t err;
};
ScratchSlot g_scratch[kMaxDevices];

// Device address of the scratch on device `dev`, looked up by the first call
// on that device, with that device current (the caller's current device).
// A failed look-up is remembered and returned by every later call.
int noalloc_scratch(int dev, void **out) {
  ScratchSlot &s = g_scratch[dev];
  std::call_once(s.once, [&] {
    s.ptr = nullptr;
    s.err = cudaGetSymbolAddress(&s.ptr, fp8bq_noalloc_scratch);
  });
  if (s.err != cudaSuccess) return cuda_fail(s.err);
  *out = s.ptr;
  return FP8BQ_OK;
}

}  // namespace

extern "C" {

int fp8bq_version(void) { return 10000; }

const char *fp8bq_status_string(int s) {
  switch (s) {
    case FP8BQ_OK: return "ok";
    case FP8BQ_ERR_NULL: return "a required pointer is NULL";
    case FP8BQ_ERR_SHAPE: return "invalid shape";
    case FP8BQ_ERR_ALIGN: return "pointer or pitch misaligned";
    case FP8BQ_ERR_UNSUPPORTED: return "unsupported argument";
    case FP8BQ_ERR_ARCH: return "device is not compute capability 10.3";
    case FP8BQ_ERR_WORKSPACE: return "workspace missing or too small";
    case FP8BQ_ERR_CUDA: return "CUDA runtime error";
    case FP8BQ_ERR_TIMEOUT: return "a device-side wait timed out";
    case FP8BQ_ERR_BOUNDS: return "a device-side bounds check skipped a write (debug build)";
    default: return "unknown status";
  }
}

int fp8bq_last_cuda_error(void) { return g_last_cuda_error; }

size_t fp8bq_workspace_bytes(int op, int64_t M, int64_t N, int64_t K) {
  if (op < FP8BQ_OP_GEMM || op > FP8BQ_OP_GROUPED_GEMM || M < 0 || N < 1 || K < 1) return 256;
  return workspace_layout(op, M, N, K).total;
}

int fp8bq_workspace_init(void *ws, size_t ws_bytes, void *stream) {
  if (!ws) return FP8BQ_ERR_NULL;
  if (!aligned(ws, 256)) return FP8BQ_ERR_ALIGN;
  cudaError_t e = cudaMemsetAsync(ws, 0, ws_bytes, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FP8BQ_OK : cuda_fail(e);
}

int fp8bq_poll_status(void *ws, void *stream) {
  if (!ws) return FP8BQ_ERR_NULL;
  if (!aligned(ws, 256)) return FP8BQ_ERR_ALIGN;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint32_t word = 0;
  cudaError_t e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_fail(e);
  e = cudaMemcpy(&word, ws, sizeof word, cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e);
  if (word != 0) {
    e = cudaMemset(ws, 0, sizeof word);
    if (e != cudaSuccess) return cuda_fail(e);
    return word == kStatusBounds ? FP8BQ_ERR_BOUNDS : FP8BQ_ERR_TIMEOUT;
  }
  return FP8BQ_OK;
}

// ------------------------------------------------------------------ block path

int fp8bq_quant_act(const void *x, int64_t M, int64_t K, int64_t ldx, void *q, float *s,
                    int s_layout, void *stream) {
  if (M == 0) return empty_batch(K, 1);
  if (!q || !s) return FP8BQ_ERR_NULL;
  RETURN_IF(check_act(x, M, K, ldx, 16));
  if (s_layout != FP8BQ_SCALE_ROW_MAJOR && s_layout != FP8BQ_SCALE_COL_MAJOR)
    return FP8BQ_ERR_UNSUPPORTED;
  if (!aligned(q, 16) || !aligned(s, 4)) return FP8BQ_ERR_ALIGN;
  if (M == 0) return FP8BQ_OK;
  DeviceInfo dev;
  RETURN_IF(device_info(&dev));
  launch_quant_group(x, M, K, ldx, q, s, s_layout, dev.num_sms, static_cast<cudaStream_t>(stream));
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? FP8BQ_OK : cuda_fail(e);
}

int fp8bq_gemm(const void *q, const float *s_x, int s_layout, const void *w, const float *s_w,
               const void *bias, void *y, int64_t M, int64_t N, int64_t K, void *ws,
               size_t ws_bytes, void *stream) {
  if (M == 0) return empty_batch(K, N);
  if (!q || !s_x || !w || !s_w || !y) return FP8BQ_ERR_NULL;
  RETURN_IF(check_gemm_shape(M, N, K, 16));
  if (s_layout != FP8BQ_SCALE_ROW_MAJOR && s_layout != FP8BQ_SCALE_COL_MAJOR)
    return FP8BQ_ERR_UNSUPPORTED;
  if (!aligned(q, 16) || !aligned(w, 16) || !aligned(y, 16) || !aligned(s_x, 4) ||
      !aligned(s_w, 4) || !aligned(bias, 2))
    return FP8BQ_ERR_ALIGN;
  RETURN_IF(check_ws(ws, ws_bytes, FP8BQ_OP_GEMM, M, N, K));
  if (M == 0) return FP8BQ_OK;
  DeviceInfo dev;
  RETURN_IF(device_info(&dev));
  return gemm_block_impl(q, s_x, s_layout, w, s_w, bias, y, M, N, K, ws, FP8BQ_OP_GEMM,
                         static_cast<cudaStream_t>(stream), dev);
}

// Up to this many tokens the decode linear quantises inside the GEMM (every
// weight tile's CTAs quantise the same activations again, which pays only while
// the token rows are few); above, the quantiser kernel runs first.
#ifndef FP8BQ_FUSED_LINEAR_MAX_M
#define FP8BQ_FUSED_LINEAR_MAX_M 16
#endif
constexpr int64_t kFusedLinearMaxM = FP8BQ_FUSED_LINEAR_MAX_M;

int fp8bq_linear(const void *x, int64_t ldx, const void *w, const float *s_w, const void *bias,
                 void *y, int64_t M, int64_t N, int64_t K, void *ws, size_t ws_bytes,
                 void *stream) {
  if (M == 0) return empty_batch(K, N);
  if (!w || !s_w || !y) return FP8BQ_ERR_NULL;
  RETURN_IF(check_act(x, M, K, ldx, 16));
  RETURN_IF(check_gemm_shape(M, N, K, 16));
  if (!aligned(w, 16) || !aligned(y, 16) || !aligned(s_w, 4) || !aligned(bias, 2))
    return FP8BQ_ERR_ALIGN;
  RETURN_IF(check_ws(ws, ws_bytes, FP8BQ_OP_LINEAR, M, N, K));
  if (M == 0) return FP8BQ_OK;
  DeviceInfo dev;
  RETURN_IF(device_info(&dev));
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (M <= kFusedLinearMaxM) {
    // decode: one launch -- the GEMM's CTAs quantise the activations of
    // their own K range as the stages arrive (same codes and scales as
    // fp8bq_quant_act), with no second kernel and no round trip through the
    // workspace
    GemmArgs a = base_args(kModeBlock, M, N, K, bias, y, ws, FP8BQ_OP_LINEAR);
    a.sw = s_w;
    a.xq = x;
    a.ldxq = ldx;
    cudaError_t e;
    const int r = launch_gemm(a, nullptr, w, dev, st, &e);
    return finish_launch(r, e);
  }
  const WorkspaceLayout L = workspace_layout(FP8BQ_OP_LINEAR, M, N, K);
  uint8_t *q = static_cast<uint8_t *>(ws) + L.q;
  float *s = reinterpret_cast<float *>(static_cast<uint8_t *>(ws) + L.s);
  // row-major scales: each epilogue thread walks its own row's scales, which
  // stay in L1 across consecutive K blocks
  launch_quant_group(x, M, K, ldx, q, s, FP8BQ_SCALE_ROW_MAJOR, dev.num_sms, st);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e);
  return gemm_block_impl(q, s, FP8BQ_SCALE_ROW_MAJOR, w, s_w, bias, y, M, N, K, ws,
                         FP8BQ_OP_LINEAR, st, dev);
}

// ------------------------------------------------------------------ MX path

int fp8bq_mx_quant_act(const void *x, int64_t M, int64_t K, int64_t ldx, void *q, uint8_t *s,
                       void *stream) {
  if (M == 0) return empty_batch(K, 1);
  if (!q || !s) return FP8BQ_ERR_NULL;
  RETURN_IF(check_act(x, M, K, ldx, 32));
  if (!aligned(q, 16)) return FP8BQ_ERR_ALIGN;
  if (M == 0) return FP8BQ_OK;
  DeviceInfo dev;
  RETURN_IF(device_info(&dev));
  launch_quant_mx(x, M, K, ldx, q, s, dev.num_sms, static_cast<cudaStream_t>(stream));
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? FP8BQ_OK : cuda_fail(e);
}

int fp8bq_mx_gemm(const void *q, const uint8_t *s_x, const void *w, const uint8_t *s_w,
                  const void *bias, void *y, int64_t M, int64_t N, int64_t K, void *ws,
                  size_t ws_bytes, void *stream) {
  if (M == 0) return empty_batch(K, N);
  if (!q || !s_x || !w || !s_w || !y) return FP8BQ_ERR_NULL;
  RETURN_IF(check_gemm_shape(M, N, K, 32));
  if (!aligned(q, 16) || !aligned(w, 16) || !aligned(y, 16) || !aligned(bias, 2))
    return FP8BQ_ERR_ALIGN;
  RETURN_IF(check_ws(ws, ws_bytes, FP8BQ_OP_MX_GEMM, M, N, K));
  if (M == 0) return FP8BQ_OK;
  DeviceInfo dev;
  RETURN_IF(device_info(&dev));
  return gemm_mx_impl(q, s_x, w, s_w, bias, y, M, N, K, ws, FP8BQ_OP_MX_GEMM,
                      static_cast<cudaStream_t>(stream), dev);
}

int fp8bq_mx_linear(const void *x, int64_t ldx, const void *w, const uint8_t *s_w,
                    const void *bias, void *y, int64_t M, int64_t N, int64_t K, void *ws,
                    size_t ws_bytes, void *stream) {
  if (M == 0) return empty_batch(K, N);
  if (!w || !s_w || !y) return FP8BQ_ERR_NULL;
  RETURN_IF(check_act(x, M, K, ldx, 32));
  RETURN_IF(check_gemm_shape(M, N, K, 32));
  if (!aligned(w, 16) || !aligned(y, 16) || !aligned(bias, 2)) return FP8BQ_ERR_ALIGN;
  RETURN_IF(check_ws(ws, ws_bytes, FP8BQ_OP_MX_LINEAR, M, N, K));
  if (M == 0) return FP8BQ_OK;
  DeviceInfo dev;
  RETURN_IF(device_info(&dev));
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const WorkspaceLayout L = workspace_layout(FP8BQ_OP_MX_LINEAR, M, N, K);
  uint8_t *q = static_cast<uint8_t *>(ws) + L.q;
  uint8_t *s = static_cast<uint8_t *>(ws) + L.s;
  launch_quant_mx(x, M, K, ldx, q, s, dev.num_sms, st);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e);
  return gemm_mx_impl(q, s, w, s_w, bias, y, M, N, K, ws, FP8BQ_OP_MX_LINEAR, st, dev);
}

// ------------------------------------------------------------------ static path

// ------------------------------------------------------------------ residual add + RMSNorm

namespace {

constexpr int64_t kNormMaxK = 16384;

int norm_common(const void *x, int64_t ldx, const void *residual, int64_t ld_res,
                const void *residual_out, const void *gamma, float eps, int64_t M, int64_t K,
                const void *y, const void *q) {
  RETURN_IF(check_act(x, M, K, ldx, 16));
  if (!gamma) return FP8BQ_ERR_NULL;
  if (K > kNormMaxK || !(eps >= 0.0f) || !(eps <= 3.4e38f)) return FP8BQ_ERR_UNSUPPORTED;
  if (residual && (ld_res < K || !aligned(residual, 16) || ld_res % 8 != 0))
    return ld_res < K ? FP8BQ_ERR_SHAPE : FP8BQ_ERR_ALIGN;
  if (residual_out && residual_out == residual && ld_res != K) return FP8BQ_ERR_SHAPE;
  if (!aligned(gamma, 16) || !aligned(residual_out, 16) || !aligned(y, 16) || !aligned(q, 16))
    return FP8BQ_ERR_ALIGN;
  return FP8BQ_OK;
}

}  // namespace

int fp8bq_add_rmsnorm_quant_act(const void *x, int64_t ldx, const void *residual,
                                int64_t ld_res, void *residual_out, const void *gamma, float eps,
                                int64_t M, int64_t K, void *y, void *q, float *s, int s_layout,
                                void *stream) {
  if (M == 0) return empty_batch(K, 1);
  RETURN_IF(norm_common(x, ldx, residual, ld_res, residual_out, gamma, eps, M, K, y, q));
  if (q) {
    if (!s) return FP8BQ_ERR_NULL;
    if (s_layout != FP8BQ_SCALE_ROW_MAJOR && s_layout != FP8BQ_SCALE_COL_MAJOR)
      return FP8BQ_ERR_UNSUPPORTED;
    if (!aligned(s, 4)) return FP8BQ_ERR_ALIGN;
  }
  DeviceInfo dev;
  RETURN_IF(device_info(&dev));
  cudaError_t e = launch_add_rmsnorm(x, ldx, residual, ld_res, residual_out, gamma, eps, M, K,
                                     y, q, s, s_layout, nullptr, dev.num_sms,
                                     static_cast<cudaStream_t>(stream));
  if (e == cudaSuccess) e = cudaGetLastError();
  return e == cudaSuccess ? FP8BQ_OK : cuda_fail(e);
}

int fp8bq_add_rmsnorm_static_quant_act(const void *x, int64_t ldx, const void *residual,
                                       int64_t ld_res, void *residual_out, const void *gamma,
                                       float eps, const float *s_x, int64_t M, int64_t K,
                                       void *y, void *q, void *stream) {
  if (M == 0) return empty_batch(K, 1);
  if (!q || !s_x) return FP8BQ_ERR_NULL;
  RETURN_IF(norm_common(x, ldx, residual, ld_res, residual_out, gamma, eps, M, K, y, q));
  if (!aligned(s_x, 4)) return FP8BQ_ERR_ALIGN;
  DeviceInfo dev;
  RETURN_IF(device_info(&dev));
  cudaError_t e = launch_add_rmsnorm(x, ldx, residual, ld_res, residual_out, gamma, eps, M, K,
                                     y, q, nullptr, FP8BQ_SCALE_ROW_MAJOR, s_x, dev.num_sms,
                                     static_cast<cudaStream_t>(stream));
  if (e == cudaSuccess) e = cudaGetLastError();
  return e == cudaSuccess ? FP8BQ_OK : cuda_fail(e);
}

int fp8bq_static_quant_act(const void *x, int64_t M, int64_t K, int64_t ldx, const float *s_x,
                           void *q, void *stream) {
  if (M == 0) return empty_batch(K, 1);
  if (!q || !s_x) return FP8BQ_ERR_NULL;
  RETURN_IF(check_act(x, M, K, ldx, 16));
  if (!aligned(q, 16) || !aligned(s_x, 4)) return FP8BQ_ERR_ALIGN;
  if (M == 0) return FP8BQ_OK;
  DeviceInfo dev;
  RETURN_IF(device_info(&dev));
  launch_quant_static(x, M, K, ldx, s_x, q, dev.num_sms, static_cast<cudaStream_t>(stream));
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? FP8BQ_OK : cuda_fail(e);
}

int fp8bq_static_gemm(const void *q, const float *s_x, const void *w, const float *s_w_part,
                      const int64_t *part_sizes_host, int n_parts, const void *bias, void *y,
                      int64_t M, int64_t N, int64_t K, void *ws, size_t ws_bytes, void *stream) {
  if (M == 0) return empty_batch(K, N);
  if (!q || !s_x || !w || !s_w_part || !y) return FP8BQ_ERR_NULL;
  RETURN_IF(check_gemm_shape(M, N, K, 16));
  RETURN_IF(check_parts(part_sizes_host, n_parts, N));
  if (!aligned(q, 16) || !aligned(w, 16) || !aligned(y, 16) || !aligned(s_x, 4) ||
      !aligned(s_w_part, 4) || !aligned(bias, 2))
    return FP8BQ_ERR_ALIGN;
  RETURN_IF(check_ws(ws, ws_bytes, FP8BQ_OP_STATIC_GEMM, M, N, K));
  if (M == 0) return FP8BQ_OK;
  DeviceInfo dev;
  RETURN_IF(device_info(&dev));
  return gemm_static_impl(q, s_x, w, s_w_part, part_sizes_host, n_parts, bias, y, M, N, K, ws,
                          FP8BQ_OP_STATIC_GEMM, static_cast<cudaStream_t>(stream), dev);
}

int fp8bq_static_linear(const void *x, int64_t ldx, const float *s_x, const void *w,
                        const float *s_w_part, const int64_t *part_sizes_host, int n_parts,
                        const void *bias, void *y, int64_t M, int64_t N, int64_t K, void *ws,
                        size_t ws_bytes, void *stream) {
  if (M == 0) return empty_batch(K, N);
  if (!s_x || !w || !s_w_part || !y) return FP8BQ_ERR_NULL;
  RETURN_IF(check_act(x, M, K, ldx, 16));
  RETURN_IF(check_gemm_shape(M, N, K, 16));
  RETURN_IF(check_parts(part_sizes_host, n_parts, N));
  if (!aligned(w, 16) || !aligned(y, 16) || !aligned(s_x, 4) || !aligned(s_w_part, 4) ||
      !aligned(bias, 2))
    return FP8BQ_ERR_ALIGN;
  RETURN_IF(check_ws(ws, ws_bytes, FP8BQ_OP_STATIC_LINEAR, M, N, K));
  if (M == 0) return FP8BQ_OK;
  DeviceInfo dev;
  RETURN_IF(device_info(&dev));
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const WorkspaceLayout L = workspace_layout(FP8BQ_OP_STATIC_LINEAR, M, N, K);
  uint8_t *q = static_cast<uint8_t *>(ws) + L.q;
  launch_quant_static(x, M, K, ldx, s_x, q, dev.num_sms, st);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e);
  return gemm_static_impl(q, s_x, w, s_w_part, part_sizes_host, n_parts, bias, y, M, N, K, ws,
                          FP8BQ_OP_STATIC_LINEAR, st, dev);
}

// ------------------------------------------------------------------ set-up helpers

int fp8bq_quant_weight_block(const void *w, int64_t N, int64_t K, int64_t ldw, void *q,
                             float *s_w, void *stream) {
  if (!q || !s_w) return FP8BQ_ERR_NULL;
  RETURN_IF(check_act(w, N, K, ldw, 16));
  if (N < 1) return FP8BQ_ERR_SHAPE;
  if (!aligned(q, 16) || !aligned(s_w, 4)) return FP8BQ_ERR_ALIGN;
  if ((N + 127) / 128 > 65535) return FP8BQ_ERR_SHAPE;
  DeviceInfo dev;
  RETURN_IF(device_info(&dev));
  launch_quant_weight_block(w, N, K, ldw, q, s_w, static_cast<cudaStream_t>(stream));
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? FP8BQ_OK : cuda_fail(e);
}

int fp8bq_absmax_scale(const void *x, int64_t rows, int64_t K, int64_t ldx, float *s,
                       void *stream) {
  if (!s) return FP8BQ_ERR_NULL;
  RETURN_IF(check_act(x, rows, K, ldx, 16));
  if (rows < 1) return FP8BQ_ERR_SHAPE;
  if (!aligned(s, 4)) return FP8BQ_ERR_ALIGN;
  DeviceInfo dev;
  RETURN_IF(device_info(&dev));
  launch_absmax_scale(x, rows, K, ldx, s, dev.num_sms, static_cast<cudaStream_t>(stream));
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? FP8BQ_OK : cuda_fail(e);
}

int fp8bq_check_scales(const float *s, int64_t n, void *scratch, int64_t *counts_host,
                       int64_t *first_bad_host, void *stream) {
  if (!counts_host || !first_bad_host) return FP8BQ_ERR_NULL;
  if (n < 0) return FP8BQ_ERR_SHAPE;
  if (n > 0 && (!s || !scratch)) return FP8BQ_ERR_NULL;
  if (!aligned(s, 4) || !aligned(scratch, 8)) return FP8BQ_ERR_ALIGN;
  if (n == 0) {
    counts_host[0] = counts_host[1] = counts_host[2] = 0;
    *first_bad_host = -1;
    return FP8BQ_OK;
  }
  DeviceInfo dev;
  RETURN_IF(device_info(&dev));
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  unsigned long long *out = static_cast<unsigned long long *>(scratch);
  launch_check_scales(s, n, out, dev.num_sms, st);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e);
  unsigned long long h[4];
  e = cudaMemcpyAsync(h, out, sizeof h, cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_fail(e);
  for (int k = 0; k < 3; ++k) counts_host[k] = static_cast<int64_t>(h[k]);
  *first_bad_host = h[3] < static_cast<unsigned long long>(n) ? static_cast<int64_t>(h[3]) : -1;
  return FP8BQ_OK;
}

int fp8bq_e4m3_from_bits(uint32_t first, int64_t n, uint8_t *codes, void *stream) {
  if (n < 0 || static_cast<uint64_t>(first) + static_cast<uint64_t>(n) > (1ull << 32))
    return FP8BQ_ERR_SHAPE;
  if (n == 0) return FP8BQ_OK;
  if (!codes) return FP8BQ_ERR_NULL;
  if (!aligned(codes, 8)) return FP8BQ_ERR_ALIGN;
  DeviceInfo dev;
  RETURN_IF(device_info(&dev));
  launch_e4m3_bits(first, n, codes, dev.num_sms, static_cast<cudaStream_t>(stream));
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? FP8BQ_OK : cuda_fail(e);
}

// ------------------------------------------------------------------ no-allocation GEMM

// fp8bq_gemm with the library's fixed scratch array in place of a caller
// workspace: same checks, same kernels, same results.  Allocates nothing.
int fp8bq_gemm_noalloc(const void *q, const float *s_x, int s_layout, const void *w,
                       const float *s_w, const void *bias, void *y, int64_t M, int64_t N,
                       int64_t K, void *stream) {
  if (M == 0) return empty_batch(K, N);
  if (!q || !s_x || !w || !s_w || !y) return FP8BQ_ERR_NULL;
  RETURN_IF(check_gemm_shape(M, N, K, 16));
  if (s_layout != FP8BQ_SCALE_ROW_MAJOR && s_layout != FP8BQ_SCALE_COL_MAJOR)
    return FP8BQ_ERR_UNSUPPORTED;
  if (!aligned(q, 16) || !aligned(w, 16) || !aligned(y, 16) || !aligned(s_x, 4) ||
      !aligned(s_w, 4) || !aligned(bias, 2))
    return FP8BQ_ERR_ALIGN;
  // the scratch is laid out like an fp8bq_gemm workspace of this shape without
  // the split tail tiles' partials (those tiles then run whole)
  const WorkspaceLayout L = workspace_layout(FP8BQ_OP_GEMM, M, N, K, false);
  if (L.total > static_cast<size_t>(FP8BQ_NOALLOC_SCRATCH_BYTES)) return FP8BQ_ERR_WORKSPACE;
  DeviceInfo dev;
  RETURN_IF(device_info(&dev));
  int d = 0;
  cudaError_t e = cudaGetDevice(&d);
  if (e != cudaSuccess) return cuda_fail(e);
  void *scratch = nullptr;
  RETURN_IF(noalloc_scratch(d, &scratch));
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // The status word, the tile counters and the decode tiles' partial slots
  // must start at zero; a previous call whose bounded wait ran out may have
  // left them set.
  e = cudaMemsetAsync(scratch, 0, L.partials, st);
  if (e != cudaSuccess) return cuda_fail(e);
  int kps = 0;
  const int splits = M <= 64 ? decode_splits(N, K, dev.num_sms, &kps) : 1;
  if (splits > 1) {
    const size_t slot = static_cast<size_t>((M + 3) / 4 * 4) * static_cast<size_t>(N) * 4;
    e = cudaMemsetAsync(static_cast<uint8_t *>(scratch) + L.partials, 0,
                        static_cast<size_t>(splits) * slot, st);
    if (e != cudaSuccess) return cuda_fail(e);
  }
  return gemm_block_impl(q, s_x, s_layout, w, s_w, bias, y, M, N, K, scratch, FP8BQ_OP_GEMM, st,
                         dev, false);
}


// The status word of the scratch array on the current device: read after the
// stream's work has finished, then cleared (like fp8bq_poll_status).
int fp8bq_noalloc_poll_status(void *stream) {
  DeviceInfo dev;
  RETURN_IF(device_info(&dev));
  int d = 0;
  cudaError_t e = cudaGetDevice(&d);
  if (e != cudaSuccess) return cuda_fail(e);
  void *scratch = nullptr;
  RETURN_IF(noalloc_scratch(d, &scratch));
  return fp8bq_poll_status(scratch, stream);
}

// ------------------------------------------------------------------ channelwise path

int fp8bq_channel_quant_act(const void *x, int64_t M, int64_t K, int64_t ldx, void *q, float *s,
                            void *stream) {
  if (M == 0) return empty_batch(K, 1);
  if (!q || !s) return FP8BQ_ERR_NULL;
  RETURN_IF(check_act(x, M, K, ldx, 16));
  if (!aligned(q, 16) || !aligned(s, 4)) return FP8BQ_ERR_ALIGN;
  DeviceInfo dev;
  RETURN_IF(device_info(&dev));
  launch_quant_token(x, M, K, ldx, q, s, dev.num_sms, static_cast<cudaStream_t>(stream));
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? FP8BQ_OK : cuda_fail(e);
}

int fp8bq_channel_gemm(const void *q, const float *s_x, const void *w, const float *s_w,
                       const void *bias, void *y, int64_t M, int64_t N, int64_t K, void *ws,
                       size_t ws_bytes, void *stream) {
  if (M == 0) return empty_batch(K, N);
  if (!q || !s_x || !w || !s_w || !y) return FP8BQ_ERR_NULL;
  RETURN_IF(check_gemm_shape(M, N, K, 16));
  if (!aligned(q, 16) || !aligned(w, 16) || !aligned(y, 16) || !aligned(s_x, 4) ||
      !aligned(s_w, 4) || !aligned(bias, 2))
    return FP8BQ_ERR_ALIGN;
  RETURN_IF(check_ws(ws, ws_bytes, FP8BQ_OP_CHANNEL_GEMM, M, N, K));
  DeviceInfo dev;
  RETURN_IF(device_info(&dev));
  return gemm_channel_impl(q, s_x, w, s_w, bias, y, M, N, K, ws, FP8BQ_OP_CHANNEL_GEMM,
                           static_cast<cudaStream_t>(stream), dev);
}

int fp8bq_channel_linear(const void *x, int64_t ldx, const void *w, const float *s_w,
                         const void *bias, void *y, int64_t M, int64_t N, int64_t K, void *ws,
                         size_t ws_bytes, void *stream) {
  if (M == 0) return empty_batch(K, N);
  if (!w || !s_w || !y) return FP8BQ_ERR_NULL;
  RETURN_IF(check_act(x, M, K, ldx, 16));
  RETURN_IF(check_gemm_shape(M, N, K, 16));
  if (!aligned(w, 16) || !aligned(y, 16) || !aligned(s_w, 4) || !aligned(bias, 2))
    return FP8BQ_ERR_ALIGN;
  RETURN_IF(check_ws(ws, ws_bytes, FP8BQ_OP_CHANNEL_LINEAR, M, N, K));
  DeviceInfo dev;
  RETURN_IF(device_info(&dev));
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const WorkspaceLayout L = workspace_layout(FP8BQ_OP_CHANNEL_LINEAR, M, N, K);
  uint8_t *q = static_cast<uint8_t *>(ws) + L.q;
  float *s = reinterpret_cast<float *>(static_cast<uint8_t *>(ws) + L.s);
  launch_quant_token(x, M, K, ldx, q, s, dev.num_sms, st);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e);
  return gemm_channel_impl(q, s, w, s_w, bias, y, M, N, K, ws, FP8BQ_OP_CHANNEL_LINEAR, st, dev);
}

// ------------------------------------------------------------------ block FP8 with UE8M0 scales

int fp8bq_quant_act_ue8m0(const void *x, int64_t M, int64_t K, int64_t ldx, void *q, uint8_t *u,
                          void *stream) {
  if (M == 0) return empty_batch(K, 1);
  if (!q || !u) return FP8BQ_ERR_NULL;
  RETURN_IF(check_act(x, M, K, ldx, 16));
  if (!aligned(q, 16)) return FP8BQ_ERR_ALIGN;
  DeviceInfo dev;
  RETURN_IF(device_info(&dev));
  launch_quant_group_ue8m0(x, M, K, ldx, q, u, dev.num_sms, static_cast<cudaStream_t>(stream));
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? FP8BQ_OK : cuda_fail(e);
}

int fp8bq_requant_weight_ue8m0(const void *q, const float *s_w, int64_t N, int64_t K, void *q_out,
                               uint8_t *u_w, void *stream) {
  if (!q || !s_w || !q_out || !u_w) return FP8BQ_ERR_NULL;
  if (N < 1 || K < 1 || N > (int64_t(1) << 31) - 1 || K > (int64_t(1) << 30)) return FP8BQ_ERR_SHAPE;
  if (!aligned(s_w, 4)) return FP8BQ_ERR_ALIGN;
  DeviceInfo dev;
  RETURN_IF(device_info(&dev));
  launch_requant_ue8m0(q, s_w, N, K, q_out, u_w, static_cast<cudaStream_t>(stream));
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? FP8BQ_OK : cuda_fail(e);
}

int fp8bq_ue8m0_gemm(const void *q, const uint8_t *u_x, const void *w, const uint8_t *u_w,
                     const void *bias, void *y, int64_t M, int64_t N, int64_t K, void *ws,
                     size_t ws_bytes, void *stream) {
  if (M == 0) return empty_batch(K, N);
  if (!q || !u_x || !w || !u_w || !y) return FP8BQ_ERR_NULL;
  RETURN_IF(check_gemm_shape(M, N, K, 32));
  if (!aligned(q, 16) || !aligned(w, 16) || !aligned(y, 16) || !aligned(bias, 2))
    return FP8BQ_ERR_ALIGN;
  RETURN_IF(check_ws(ws, ws_bytes, FP8BQ_OP_UE8M0_GEMM, M, N, K));
  DeviceInfo dev;
  RETURN_IF(device_info(&dev));
  return gemm_mx_impl(q, u_x, w, u_w, bias, y, M, N, K, ws, FP8BQ_OP_UE8M0_GEMM,
                      static_cast<cudaStream_t>(stream), dev, true);
}

int fp8bq_ue8m0_linear(const void *x, int64_t ldx, const void *w, const uint8_t *u_w,
                       const void *bias, void *y, int64_t M, int64_t N, int64_t K, void *ws,
                       size_t ws_bytes, void *stream) {
  if (M == 0) return empty_batch(K, N);
  if (!w || !u_w || !y) return FP8BQ_ERR_NULL;
  RETURN_IF(check_act(x, M, K, ldx, 32));
  RETURN_IF(check_gemm_shape(M, N, K, 32));
  if (!aligned(w, 16) || !aligned(y, 16) || !aligned(bias, 2)) return FP8BQ_ERR_ALIGN;
  RETURN_IF(check_ws(ws, ws_bytes, FP8BQ_OP_UE8M0_LINEAR, M, N, K));
  DeviceInfo dev;
  RETURN_IF(device_info(&dev));
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const WorkspaceLayout L = workspace_layout(FP8BQ_OP_UE8M0_LINEAR, M, N, K);
  uint8_t *q = static_cast<uint8_t *>(ws) + L.q;
  uint8_t *u = static_cast<uint8_t *>(ws) + L.s;
  launch_quant_group_ue8m0(x, M, K, ldx, q, u, dev.num_sms, st);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e);
  return gemm_mx_impl(q, u, w, u_w, bias, y, M, N, K, ws, FP8BQ_OP_UE8M0_LINEAR, st, dev, true);
}

// ------------------------------------------------------------------ grouped (MoE)

int fp8bq_grouped_gemm(const void *q, const float *s_x, int s_layout, const void *w,
                       const float *s_w, const int32_t *offsets, int64_t E, void *y, int64_t M,
                       int64_t N, int64_t K, void *ws, size_t ws_bytes, void *stream) {
  RETURN_IF(check_grouped(q, s_x, s_layout, w, s_w, offsets, E, M, N, K, E + (M + 127) / 128, y));
  RETURN_IF(check_ws(ws, ws_bytes, FP8BQ_OP_GROUPED_GEMM, M, N, K));
  if (M == 0) return FP8BQ_OK;
  DeviceInfo dev;
  RETURN_IF(device_info(&dev));
  return gemm_grouped_impl(q, s_x, s_layout, w, s_w, offsets, nullptr, E, 0, y, M, N, K, ws,
                           static_cast<cudaStream_t>(stream), dev);
}

int fp8bq_grouped_gemm_masked(const void *q, const float *s_x, int s_layout, const void *w,
                              const float *s_w, const int32_t *masked_m, int64_t E,
                              int64_t max_m, void *y, int64_t N, int64_t K, void *ws,
                              size_t ws_bytes, void *stream) {
  if (max_m < 0 || max_m > ((int64_t(1) << 31) - 1) / (E > 0 ? E : 1)) return FP8BQ_ERR_SHAPE;
  const int64_t M = E * max_m;
  RETURN_IF(check_grouped(q, s_x, s_layout, w, s_w, masked_m, E, M, N, K,
                          E * ((max_m + 127) / 128), y));
  RETURN_IF(check_ws(ws, ws_bytes, FP8BQ_OP_GROUPED_GEMM, M, N, K));
  if (M == 0) return FP8BQ_OK;
  DeviceInfo dev;
  RETURN_IF(device_info(&dev));
  return gemm_grouped_impl(q, s_x, s_layout, w, s_w, nullptr, masked_m, E, max_m, y, M, N, K,
                           ws, static_cast<cudaStream_t>(stream), dev);
}

}  // extern "C"
