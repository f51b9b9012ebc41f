"""Block-wise FP8 W8A8 linear for GB300: Python binding of the C ABI (include/fp8bq.h).

Every function here has the name of the C entry point it calls and does
argument marshalling only: torch tensors become device pointers and sizes, the
current CUDA stream becomes the `stream` argument, and a non-zero status
becomes an :class:`Fp8bqError`.  All computation runs in the CUDA library
``_build/libfp8bq.so`` (build it with ``__graft_entry__.build()``); importing
this package without that library raises ImportError -- there is no fallback.

Tensor conventions: BF16 tensors are ``torch.bfloat16``; E4M3 codes are
``torch.float8_e4m3fn`` or ``torch.uint8``; FP32 scales ``torch.float32``;
UE8M0 scale codes ``torch.uint8``.  Matrices are row-major with unit stride in
the last dimension.
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import _build

__all__ = [
    "Fp8bqError", "SCALE_ROW_MAJOR", "SCALE_COL_MAJOR", "OP_GEMM", "OP_LINEAR",
    "OP_MX_GEMM", "OP_MX_LINEAR", "OP_STATIC_GEMM", "OP_STATIC_LINEAR", "OP_CHANNEL_GEMM",
    "OP_CHANNEL_LINEAR", "fp8bq_channel_quant_act", "fp8bq_channel_gemm", "fp8bq_channel_linear",
    "OP_UE8M0_GEMM", "OP_UE8M0_LINEAR", "fp8bq_quant_act_ue8m0", "fp8bq_requant_weight_ue8m0",
    "fp8bq_ue8m0_gemm", "fp8bq_ue8m0_linear",
    "OP_GROUPED_GEMM", "fp8bq_grouped_gemm", "fp8bq_grouped_gemm_masked",
    "fp8bq_check_scales",
    "library_path",
    "fp8bq_version", "fp8bq_status_string", "fp8bq_last_cuda_error",
    "fp8bq_workspace_bytes", "fp8bq_workspace_init", "fp8bq_poll_status",
    "fp8bq_quant_act", "fp8bq_gemm", "fp8bq_linear", "fp8bq_gemm_noalloc",
    "NOALLOC_SCRATCH_BYTES", "fp8bq_mx_quant_act",
    "fp8bq_mx_gemm", "fp8bq_mx_linear", "fp8bq_static_quant_act", "fp8bq_static_gemm",
    "fp8bq_add_rmsnorm_quant_act", "fp8bq_add_rmsnorm_static_quant_act",
    "fp8bq_static_linear", "fp8bq_quant_weight_block", "fp8bq_absmax_scale",
    "new_workspace",
]

SCALE_ROW_MAJOR, SCALE_COL_MAJOR = 0, 1
(OP_GEMM, OP_LINEAR, OP_MX_GEMM, OP_MX_LINEAR, OP_STATIC_GEMM,
 OP_STATIC_LINEAR, OP_CHANNEL_GEMM, OP_CHANNEL_LINEAR, OP_UE8M0_GEMM,
 OP_UE8M0_LINEAR, OP_GROUPED_GEMM) = range(11)
NOALLOC_SCRATCH_BYTES = 16 * 1024 * 1024      # FP8BQ_NOALLOC_SCRATCH_BYTES

STATUS_NAMES = {0: "FP8BQ_OK", 1: "FP8BQ_ERR_NULL", 2: "FP8BQ_ERR_SHAPE",
                3: "FP8BQ_ERR_ALIGN", 4: "FP8BQ_ERR_UNSUPPORTED", 5: "FP8BQ_ERR_ARCH",
                6: "FP8BQ_ERR_WORKSPACE", 7: "FP8BQ_ERR_CUDA", 8: "FP8BQ_ERR_TIMEOUT"}


class Fp8bqError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        self.name = STATUS_NAMES.get(status, str(status))
        msg = f"{what}: {self.name} ({_lib.fp8bq_status_string(status).decode()})"
        if status == 7:
            msg += f", cudaError {_lib.fp8bq_last_cuda_error()}"
        super().__init__(msg)


def library_path() -> str:
    return _build.LIB


def _load():
    if not os.path.exists(_build.LIB):
        raise ImportError(
            f"CUDA library {_build.LIB} is not built; run __graft_entry__.build() "
            "(there is no CPU fallback)")
    lib = ctypes.CDLL(_build.LIB)
    P, I64, I32, SZ = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_size_t
    F32 = ctypes.c_float
    sigs = {
        "fp8bq_version": (I32, []),
        "fp8bq_status_string": (ctypes.c_char_p, [I32]),
        "fp8bq_last_cuda_error": (I32, []),
        "fp8bq_workspace_bytes": (SZ, [I32, I64, I64, I64]),
        "fp8bq_workspace_init": (I32, [P, SZ, P]),
        "fp8bq_poll_status": (I32, [P, P]),
        "fp8bq_quant_act": (I32, [P, I64, I64, I64, P, P, I32, P]),
        "fp8bq_gemm": (I32, [P, P, I32, P, P, P, P, I64, I64, I64, P, SZ, P]),
        "fp8bq_linear": (I32, [P, I64, P, P, P, P, I64, I64, I64, P, SZ, P]),
        "fp8bq_gemm_noalloc": (I32, [P, P, I32, P, P, P, P, I64, I64, I64, P]),
        "fp8bq_mx_quant_act": (I32, [P, I64, I64, I64, P, P, P]),
        "fp8bq_mx_gemm": (I32, [P, P, P, P, P, P, I64, I64, I64, P, SZ, P]),
        "fp8bq_mx_linear": (I32, [P, I64, P, P, P, P, I64, I64, I64, P, SZ, P]),
        "fp8bq_static_quant_act": (I32, [P, I64, I64, I64, P, P, P]),
        "fp8bq_channel_quant_act": (I32, [P, I64, I64, I64, P, P, P]),
        "fp8bq_quant_act_ue8m0": (I32, [P, I64, I64, I64, P, P, P]),
        "fp8bq_requant_weight_ue8m0": (I32, [P, P, I64, I64, P, P, P]),
        "fp8bq_ue8m0_gemm": (I32, [P, P, P, P, P, P, I64, I64, I64, P, SZ, P]),
        "fp8bq_ue8m0_linear": (I32, [P, I64, P, P, P, P, I64, I64, I64, P, SZ, P]),
        "fp8bq_grouped_gemm": (I32, [P, P, I32, P, P, P, I64, P, I64, I64, I64, P, SZ, P]),
        "fp8bq_check_scales": (I32, [P, I64, P, P, P, P]),
        "fp8bq_grouped_gemm_masked": (I32, [P, P, I32, P, P, P, I64, I64, P, I64, I64, P, SZ,
                                            P]),
        "fp8bq_channel_gemm": (I32, [P, P, P, P, P, P, I64, I64, I64, P, SZ, P]),
        "fp8bq_channel_linear": (I32, [P, I64, P, P, P, P, I64, I64, I64, P, SZ, P]),
        "fp8bq_add_rmsnorm_quant_act": (I32, [P, I64, P, I64, P, P, F32, I64, I64, P, P, P,
                                              I32, P]),
        "fp8bq_add_rmsnorm_static_quant_act": (I32, [P, I64, P, I64, P, P, F32, P, I64, I64,
                                                     P, P, P]),
        "fp8bq_static_gemm": (I32, [P, P, P, P, P, I32, P, P, I64, I64, I64, P, SZ, P]),
        "fp8bq_static_linear": (I32, [P, I64, P, P, P, P, I32, P, P, I64, I64, I64, P, SZ,
                                      P]),
        "fp8bq_quant_weight_block": (I32, [P, I64, I64, I64, P, P, P]),
        "fp8bq_absmax_scale": (I32, [P, I64, I64, I64, P, P]),
    }
    for name, (res, args) in sigs.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


_lib = _load()


# ---------------------------------------------------------------- marshalling

def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return ctypes.c_void_p(t)
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return ctypes.c_void_p(stream)
    return ctypes.c_void_p(stream.cuda_stream)


def _ld(x) -> int:
    if x.dim() != 2 or x.stride(1) != 1:
        raise ValueError("expected a 2-D tensor with unit stride in the last dimension")
    return x.stride(0)


def _nbytes(t) -> int:
    return t.numel() * t.element_size()


def _check(status: int, what: str):
    if status != 0:
        raise Fp8bqError(status, what)


# ---------------------------------------------------------------- utility

def fp8bq_version() -> int:
    return _lib.fp8bq_version()


def fp8bq_status_string(status: int) -> str:
    return _lib.fp8bq_status_string(status).decode()


def fp8bq_last_cuda_error() -> int:
    return _lib.fp8bq_last_cuda_error()


def fp8bq_workspace_bytes(op: int, M: int, N: int, K: int) -> int:
    return _lib.fp8bq_workspace_bytes(op, M, N, K)


def fp8bq_workspace_init(ws, stream=None):
    _check(_lib.fp8bq_workspace_init(_ptr(ws), _nbytes(ws), _stream(stream)),
           "fp8bq_workspace_init")


def fp8bq_poll_status(ws, stream=None) -> int:
    """Synchronises the stream; returns 0, or 8 (FP8BQ_ERR_TIMEOUT)."""
    return _lib.fp8bq_poll_status(_ptr(ws), _stream(stream))


def new_workspace(op: int, M: int, N: int, K: int, device="cuda", stream=None):
    """A zero-initialised workspace (torch-owned device memory) for `op` at this shape."""
    ws = torch.empty(fp8bq_workspace_bytes(op, M, N, K), dtype=torch.uint8, device=device)
    fp8bq_workspace_init(ws, stream)
    return ws


# ---------------------------------------------------------------- block path

def fp8bq_quant_act(x, q, s, s_layout: int = SCALE_ROW_MAJOR, stream=None):
    M, K = x.shape
    _check(_lib.fp8bq_quant_act(_ptr(x), M, K, _ld(x), _ptr(q), _ptr(s), s_layout,
                                _stream(stream)), "fp8bq_quant_act")


def fp8bq_gemm(q, s_x, w, s_w, y, ws, bias=None, s_layout: int = SCALE_ROW_MAJOR,
               stream=None):
    M, K = q.shape
    N = w.shape[0]
    _check(_lib.fp8bq_gemm(_ptr(q), _ptr(s_x), s_layout, _ptr(w), _ptr(s_w), _ptr(bias),
                           _ptr(y), M, N, K, _ptr(ws), _nbytes(ws), _stream(stream)),
           "fp8bq_gemm")


def fp8bq_gemm_noalloc(q, s_x, w, s_w, y, bias=None, s_layout: int = SCALE_ROW_MAJOR,
                       stream=None):
    """fp8bq_gemm on the library's fixed device scratch instead of a workspace
    (for callers that may not allocate device memory); see include/fp8bq.h."""
    M, K = q.shape
    N = w.shape[0]
    _check(_lib.fp8bq_gemm_noalloc(_ptr(q), _ptr(s_x), s_layout, _ptr(w), _ptr(s_w),
                                   _ptr(bias), _ptr(y), M, N, K, _stream(stream)),
           "fp8bq_gemm_noalloc")


def fp8bq_linear(x, w, s_w, y, ws, bias=None, stream=None):
    M, K = x.shape
    N = w.shape[0]
    _check(_lib.fp8bq_linear(_ptr(x), _ld(x), _ptr(w), _ptr(s_w), _ptr(bias), _ptr(y),
                             M, N, K, _ptr(ws), _nbytes(ws), _stream(stream)),
           "fp8bq_linear")


# ---------------------------------------------------------------- MX path

def fp8bq_mx_quant_act(x, q, s, stream=None):
    M, K = x.shape
    _check(_lib.fp8bq_mx_quant_act(_ptr(x), M, K, _ld(x), _ptr(q), _ptr(s),
                                   _stream(stream)), "fp8bq_mx_quant_act")


def fp8bq_mx_gemm(q, s_x, w, s_w, y, ws, bias=None, stream=None):
    M, K = q.shape
    N = w.shape[0]
    _check(_lib.fp8bq_mx_gemm(_ptr(q), _ptr(s_x), _ptr(w), _ptr(s_w), _ptr(bias), _ptr(y),
                              M, N, K, _ptr(ws), _nbytes(ws), _stream(stream)),
           "fp8bq_mx_gemm")


def fp8bq_mx_linear(x, w, s_w, y, ws, bias=None, stream=None):
    M, K = x.shape
    N = w.shape[0]
    _check(_lib.fp8bq_mx_linear(_ptr(x), _ld(x), _ptr(w), _ptr(s_w), _ptr(bias), _ptr(y),
                                M, N, K, _ptr(ws), _nbytes(ws), _stream(stream)),
           "fp8bq_mx_linear")


# ---------------------------------------------------------------- static path

def _parts(part_sizes):
    arr = (ctypes.c_int64 * len(part_sizes))(*[int(p) for p in part_sizes])
    return arr, len(part_sizes)


def fp8bq_static_quant_act(x, s_x, q, stream=None):
    M, K = x.shape
    _check(_lib.fp8bq_static_quant_act(_ptr(x), M, K, _ld(x), _ptr(s_x), _ptr(q),
                                       _stream(stream)), "fp8bq_static_quant_act")


def fp8bq_channel_quant_act(x, q, s, stream=None):
    """One scale per row (per-token activations, or per-channel weights)."""
    M, K = x.shape
    _check(_lib.fp8bq_channel_quant_act(_ptr(x), M, K, _ld(x), _ptr(q), _ptr(s),
                                        _stream(stream)), "fp8bq_channel_quant_act")


def fp8bq_channel_gemm(q, s_x, w, s_w, y, ws, bias=None, stream=None):
    M, K = q.shape
    N = w.shape[0]
    _check(_lib.fp8bq_channel_gemm(_ptr(q), _ptr(s_x), _ptr(w), _ptr(s_w), _ptr(bias), _ptr(y),
                                   M, N, K, _ptr(ws), _nbytes(ws), _stream(stream)),
           "fp8bq_channel_gemm")


def fp8bq_channel_linear(x, w, s_w, y, ws, bias=None, stream=None):
    M, K = x.shape
    N = w.shape[0]
    _check(_lib.fp8bq_channel_linear(_ptr(x), _ld(x), _ptr(w), _ptr(s_w), _ptr(bias), _ptr(y),
                                     M, N, K, _ptr(ws), _nbytes(ws), _stream(stream)),
           "fp8bq_channel_linear")


def fp8bq_quant_act_ue8m0(x, q, u, stream=None):
    """Group-128 quantisation with power-of-two (UE8M0) scales."""
    M, K = x.shape
    _check(_lib.fp8bq_quant_act_ue8m0(_ptr(x), M, K, _ld(x), _ptr(q), _ptr(u), _stream(stream)),
           "fp8bq_quant_act_ue8m0")


def fp8bq_requant_weight_ue8m0(q, s_w, q_out, u_w, stream=None):
    """FP32 128x128 block scales -> UE8M0 (rounded up), codes re-encoded."""
    N, K = q.shape
    _check(_lib.fp8bq_requant_weight_ue8m0(_ptr(q), _ptr(s_w), N, K, _ptr(q_out), _ptr(u_w),
                                           _stream(stream)), "fp8bq_requant_weight_ue8m0")


def fp8bq_ue8m0_gemm(q, u_x, w, u_w, y, ws, bias=None, stream=None):
    M, K = q.shape
    N = w.shape[0]
    _check(_lib.fp8bq_ue8m0_gemm(_ptr(q), _ptr(u_x), _ptr(w), _ptr(u_w), _ptr(bias), _ptr(y),
                                 M, N, K, _ptr(ws), _nbytes(ws), _stream(stream)),
           "fp8bq_ue8m0_gemm")


def fp8bq_ue8m0_linear(x, w, u_w, y, ws, bias=None, stream=None):
    M, K = x.shape
    N = w.shape[0]
    _check(_lib.fp8bq_ue8m0_linear(_ptr(x), _ld(x), _ptr(w), _ptr(u_w), _ptr(bias), _ptr(y),
                                   M, N, K, _ptr(ws), _nbytes(ws), _stream(stream)),
           "fp8bq_ue8m0_linear")


def fp8bq_check_scales(s, scratch=None, stream=None) -> dict:
    """Counts unusable FP32 scales in a device tensor: the unloaded sentinel
    (-FLT_MAX), NaN / inf, other values <= 0; and the first bad flat index."""
    if scratch is None:
        scratch = torch.empty(4, dtype=torch.int64, device=s.device)
    counts = (ctypes.c_int64 * 3)()
    first = ctypes.c_int64()
    _check(_lib.fp8bq_check_scales(_ptr(s), s.numel(), _ptr(scratch),
                                   ctypes.c_void_p(ctypes.addressof(counts)),
                                   ctypes.c_void_p(ctypes.addressof(first)), _stream(stream)),
           "fp8bq_check_scales")
    return {"sentinel": counts[0], "nonfinite": counts[1], "nonpositive": counts[2],
            "first_bad": first.value}


# ---------------------------------------------------------------- grouped (MoE)

def _device_int32(t, n: int, what: str):
    """The segment bounds are read by the kernel: a CUDA int32 tensor of n values."""
    if not (isinstance(t, torch.Tensor) and t.is_cuda and t.dtype == torch.int32
            and t.is_contiguous() and t.numel() == n):
        raise ValueError(f"{what} must be a contiguous CUDA int32 tensor with {n} values")

def fp8bq_grouped_gemm(q, s_x, w, s_w, offsets, y, ws, s_layout: int = SCALE_ROW_MAJOR,
                       stream=None):
    """Rows offsets[e] .. offsets[e+1]-1 of q / y use expert e's weight w[e]
    [N, K] and scale grid s_w[e]; offsets is a device int32 tensor [E+1]."""
    M, K = q.shape
    E, N, _ = w.shape
    _device_int32(offsets, E + 1, "offsets")
    _check(_lib.fp8bq_grouped_gemm(_ptr(q), _ptr(s_x), s_layout, _ptr(w), _ptr(s_w),
                                   _ptr(offsets), E, _ptr(y), M, N, K, _ptr(ws), _nbytes(ws),
                                   _stream(stream)), "fp8bq_grouped_gemm")


def fp8bq_grouped_gemm_masked(q, s_x, w, s_w, masked_m, y, ws, s_layout: int = SCALE_ROW_MAJOR,
                              stream=None):
    """q [E, max_m, K] (or [E*max_m, K]); the first masked_m[e] rows of slot e
    use expert e's weight; masked_m is a device int32 tensor [E]."""
    E, N, K = w.shape
    max_m = q.numel() // (K * E) if E else 0
    _device_int32(masked_m, E, "masked_m")
    _check(_lib.fp8bq_grouped_gemm_masked(_ptr(q), _ptr(s_x), s_layout, _ptr(w), _ptr(s_w),
                                          _ptr(masked_m), E, max_m, _ptr(y), N, K, _ptr(ws),
                                          _nbytes(ws), _stream(stream)),
           "fp8bq_grouped_gemm_masked")


def fp8bq_add_rmsnorm_quant_act(x, gamma, eps: float, residual=None, residual_out=None,
                                y=None, q=None, s=None, s_layout: int = SCALE_ROW_MAJOR,
                                stream=None):
    """Residual add + RMSNorm (+ group-128 quantisation when q is given)."""
    M, K = x.shape
    _check(_lib.fp8bq_add_rmsnorm_quant_act(
        _ptr(x), _ld(x), _ptr(residual), 0 if residual is None else _ld(residual),
        _ptr(residual_out), _ptr(gamma), float(eps), M, K, _ptr(y), _ptr(q), _ptr(s),
        s_layout, _stream(stream)), "fp8bq_add_rmsnorm_quant_act")


def fp8bq_add_rmsnorm_static_quant_act(x, gamma, eps: float, s_x, q, residual=None,
                                       residual_out=None, y=None, stream=None):
    """Residual add + RMSNorm, then static per-tensor quantisation with s_x[0]."""
    M, K = x.shape
    _check(_lib.fp8bq_add_rmsnorm_static_quant_act(
        _ptr(x), _ld(x), _ptr(residual), 0 if residual is None else _ld(residual),
        _ptr(residual_out), _ptr(gamma), float(eps), _ptr(s_x), M, K, _ptr(y), _ptr(q),
        _stream(stream)), "fp8bq_add_rmsnorm_static_quant_act")


def fp8bq_static_gemm(q, s_x, w, s_w_part, part_sizes, y, ws, bias=None, stream=None):
    M, K = q.shape
    N = w.shape[0]
    arr, n = _parts(part_sizes)
    _check(_lib.fp8bq_static_gemm(_ptr(q), _ptr(s_x), _ptr(w), _ptr(s_w_part), arr, n,
                                  _ptr(bias), _ptr(y), M, N, K, _ptr(ws), _nbytes(ws),
                                  _stream(stream)), "fp8bq_static_gemm")


def fp8bq_static_linear(x, s_x, w, s_w_part, part_sizes, y, ws, bias=None, stream=None):
    M, K = x.shape
    N = w.shape[0]
    arr, n = _parts(part_sizes)
    _check(_lib.fp8bq_static_linear(_ptr(x), _ld(x), _ptr(s_x), _ptr(w), _ptr(s_w_part),
                                    arr, n, _ptr(bias), _ptr(y), M, N, K, _ptr(ws),
                                    _nbytes(ws), _stream(stream)), "fp8bq_static_linear")


# ---------------------------------------------------------------- set-up helpers

def fp8bq_quant_weight_block(w, q, s_w, stream=None):
    N, K = w.shape
    _check(_lib.fp8bq_quant_weight_block(_ptr(w), N, K, _ld(w), _ptr(q), _ptr(s_w),
                                         _stream(stream)), "fp8bq_quant_weight_block")


def fp8bq_absmax_scale(x, s, stream=None):
    rows, K = x.shape
    _check(_lib.fp8bq_absmax_scale(_ptr(x), rows, K, _ld(x), _ptr(s), _stream(stream)),
           "fp8bq_absmax_scale")
