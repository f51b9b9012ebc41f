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
    "fp8bq_noalloc_poll_status",
    "NOALLOC_SCRATCH_BYTES", "fp8bq_mx_quant_act",
    "fp8bq_mx_gemm", "fp8bq_mx_linear", "fp8bq_static_quant_act", "fp8bq_static_gemm",
    "fp8bq_add_rmsnorm_quant_act", "fp8bq_add_rmsnorm_static_quant_act",
    "fp8bq_static_linear", "fp8bq_quant_weight_block", "fp8bq_absmax_scale",
    "new_workspace", "fp8bq_e4m3_from_bits",
]

SCALE_ROW_MAJOR, SCALE_COL_MAJOR = 0, 1
(OP_GEMM, OP_LINEAR, OP_MX_GEMM, OP_MX_LINEAR, OP_STATIC_GEMM,
 OP_STATIC_LINEAR, OP_CHANNEL_GEMM, OP_CHANNEL_LINEAR, OP_UE8M0_GEMM,
 OP_UE8M0_LINEAR, OP_GROUPED_GEMM) = range(11)
NOALLOC_SCRATCH_BYTES = 16 * 1024 * 1024      # FP8BQ_NOALLOC_SCRATCH_BYTES

STATUS_NAMES = {0: "FP8BQ_OK", 1: "FP8BQ_ERR_NULL", 2: "FP8BQ_ERR_SHAPE",
                3: "FP8BQ_ERR_ALIGN", 4: "FP8BQ_ERR_UNSUPPORTED", 5: "FP8BQ_ERR_ARCH",
                6: "FP8BQ_ERR_WORKSPACE", 7: "FP8BQ_ERR_CUDA", 8: "FP8BQ_ERR_TIMEOUT",
                9: "FP8BQ_ERR_BOUNDS"}


class Fp8bqError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        self.name = STATUS_NAMES.get(status, str(status))
        msg = f"{what}: {self.name} ({_lib.fp8bq_status_string(status).decode()})"
        if status == 7:
            msg += f", cudaError {_lib.fp8bq_last_cuda_error()}"
        super().__init__(msg)


# FP8BQ_LIBRARY selects another build of the same library, e.g. the debug
# build with device-side bounds checks (_build.build(debug=True))
_LIB_PATH = os.environ.get("FP8BQ_LIBRARY") or _build.LIB


def library_path() -> str:
    return _LIB_PATH


def _load():
    if not os.path.exists(_LIB_PATH):
        raise ImportError(
            f"CUDA library {_LIB_PATH} is not built; run __graft_entry__.build() "
            "(there is no CPU fallback)")
    lib = ctypes.CDLL(_LIB_PATH)
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
        "fp8bq_noalloc_poll_status": (I32, [P]),
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
        "fp8bq_e4m3_from_bits": (I32, [ctypes.c_uint32, I64, P, P]),
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


# ---------------------------------------------------------------- argument checks
#
# The C interface takes raw pointers and sizes, so a tensor of the wrong shape,
# dtype or device would be read or written past its end.  Every wrapper below
# describes each tensor it passes and `_validate` checks all of them against the
# sizes before the C call; a mismatch raises ValueError and nothing is launched.

_BF16 = (torch.bfloat16,)
_E4M3 = (torch.uint8, torch.float8_e4m3fn)
_F32 = (torch.float32,)
_U8 = (torch.uint8,)
_I32 = (torch.int32,)


def _kb(K: int) -> int:
    return -(-K // 128)


def _sx_shape(M: int, K: int, layout: int):
    """Shape of the FP32 activation scales: [M][ceil(K/128)] or [ceil(K/128)][M rounded up to 4]."""
    if layout == SCALE_ROW_MAJOR:
        return (M, _kb(K))
    if layout == SCALE_COL_MAJOR:
        return (_kb(K), -(-M // 4) * 4)
    raise ValueError(f"s_layout must be SCALE_ROW_MAJOR or SCALE_COL_MAJOR, not {layout!r}")


class _Spec:
    """One tensor argument: name, accepted dtypes and what its shape must be.

    kind "contig": contiguous with exactly `shape` (or `numel` elements when
    shape is None); kind "rows": 2-D [shape] with unit stride in the last
    dimension and any row pitch (the C call takes the pitch)."""
    __slots__ = ("name", "t", "dtypes", "shape", "numel", "kind", "optional")

    def __init__(self, name, t, dtypes, shape=None, numel=None, kind="contig", optional=False):
        self.name, self.t, self.dtypes = name, t, dtypes
        self.shape = None if shape is None else tuple(int(v) for v in shape)
        self.numel, self.kind, self.optional = numel, kind, optional


def _validate(what: str, specs, stream=None):
    """Checks every tensor argument of one call before any pointer is taken."""
    present = []
    for sp in specs:
        t = sp.t
        if t is None:
            if sp.optional:
                continue
            raise ValueError(f"{what}: {sp.name} is required")
        if not isinstance(t, torch.Tensor):
            raise ValueError(f"{what}: {sp.name} must be a torch.Tensor, not {type(t).__name__}")
        if sp.dtypes is not None and t.dtype not in sp.dtypes:
            names = " or ".join(str(d).replace("torch.", "") for d in sp.dtypes)
            raise ValueError(f"{what}: {sp.name} must be {names}, not "
                             f"{str(t.dtype).replace('torch.', '')}")
        if sp.kind == "rows":
            if t.dim() != 2 or tuple(t.shape) != sp.shape:
                raise ValueError(f"{what}: {sp.name} must have shape {sp.shape}, "
                                 f"not {tuple(t.shape)}")
            if t.numel() and (t.stride(1) != 1 or t.stride(0) < t.shape[1]):
                raise ValueError(f"{what}: {sp.name} needs unit stride in its last dimension "
                                 f"and a row pitch of at least {t.shape[1]}")
        else:
            if sp.shape is not None and tuple(t.shape) != sp.shape:
                raise ValueError(f"{what}: {sp.name} must have shape {sp.shape}, "
                                 f"not {tuple(t.shape)}")
            if sp.numel is not None and t.numel() != sp.numel:
                raise ValueError(f"{what}: {sp.name} must have {sp.numel} elements, "
                                 f"not {t.numel()}")
            if not t.is_contiguous():
                raise ValueError(f"{what}: {sp.name} must be contiguous")
        present.append(sp)
    # device last, so that shape mistakes are reported even for host tensors
    for sp in present:
        if not sp.t.is_cuda:
            raise ValueError(f"{what}: {sp.name} must be a CUDA tensor, not on {sp.t.device}")
    if present:
        want = _call_device(stream)
        for sp in present:
            if sp.t.device.index != want:
                raise ValueError(f"{what}: {sp.name} is on cuda:{sp.t.device.index} but the "
                                 f"call runs on cuda:{want}")


def _call_device(stream) -> int:
    """The device a call runs on: the stream's, else the current device."""
    if stream is not None and not isinstance(stream, int):
        dev = stream.device
        dev_index = dev.index if isinstance(dev, torch.device) else int(dev)
        if dev_index != torch.cuda.current_device():
            raise ValueError(f"stream is on cuda:{dev_index}, the current device is "
                             f"cuda:{torch.cuda.current_device()}")
        return dev_index
    return torch.cuda.current_device()


def _mat(t, name):
    """(rows, cols) of a 2-D matrix argument whose shape sets the call's sizes."""
    if not isinstance(t, torch.Tensor) or t.dim() != 2:
        raise ValueError(f"{name} must be a 2-D tensor")
    return int(t.shape[0]), int(t.shape[1])


# ---------------------------------------------------------------- utility

def fp8bq_version() -> int:
    return _lib.fp8bq_version()


def fp8bq_status_string(status: int) -> str:
    return _lib.fp8bq_status_string(status).decode()


def fp8bq_last_cuda_error() -> int:
    return _lib.fp8bq_last_cuda_error()


def fp8bq_workspace_bytes(op: int, M: int, N: int, K: int) -> int:
    return _lib.fp8bq_workspace_bytes(op, M, N, K)


def _ws(ws):
    return _Spec("ws", ws, None)


def fp8bq_workspace_init(ws, stream=None):
    _validate("fp8bq_workspace_init", [_ws(ws)], stream)
    _check(_lib.fp8bq_workspace_init(_ptr(ws), _nbytes(ws), _stream(stream)),
           "fp8bq_workspace_init")


def fp8bq_poll_status(ws, stream=None) -> int:
    """Synchronises the stream; returns 0, 8 (FP8BQ_ERR_TIMEOUT) or, from a
    debug build, 9 (FP8BQ_ERR_BOUNDS)."""
    _validate("fp8bq_poll_status", [_ws(ws)], stream)
    return _lib.fp8bq_poll_status(_ptr(ws), _stream(stream))


def new_workspace(op: int, M: int, N: int, K: int, device="cuda", stream=None):
    """A zero-initialised workspace (torch-owned device memory) for `op` at this shape."""
    ws = torch.empty(fp8bq_workspace_bytes(op, M, N, K), dtype=torch.uint8, device=device)
    fp8bq_workspace_init(ws, stream)
    return ws


def _bias(bias, N):
    return _Spec("bias", bias, _BF16, numel=N, optional=True)


# ---------------------------------------------------------------- block path

def fp8bq_quant_act(x, q, s, s_layout: int = SCALE_ROW_MAJOR, stream=None):
    M, K = _mat(x, "x")
    _validate("fp8bq_quant_act", [
        _Spec("x", x, _BF16, (M, K), kind="rows"),
        _Spec("q", q, _E4M3, (M, K)),
        _Spec("s", s, _F32, _sx_shape(M, K, s_layout))], stream)
    _check(_lib.fp8bq_quant_act(_ptr(x), M, K, _ld(x), _ptr(q), _ptr(s), s_layout,
                                _stream(stream)), "fp8bq_quant_act")


def _block_gemm_specs(q, s_x, w, s_w, y, bias, s_layout):
    M, K = _mat(q, "q")
    N = _mat(w, "w")[0]
    return M, N, K, [
        _Spec("q", q, _E4M3, (M, K)),
        _Spec("s_x", s_x, _F32, _sx_shape(M, K, s_layout)),
        _Spec("w", w, _E4M3, (N, K)),
        _Spec("s_w", s_w, _F32, (_kb(N), _kb(K))),
        _Spec("y", y, _BF16, (M, N)),
        _bias(bias, N)]


def fp8bq_gemm(q, s_x, w, s_w, y, ws, bias=None, s_layout: int = SCALE_ROW_MAJOR,
               stream=None):
    M, N, K, specs = _block_gemm_specs(q, s_x, w, s_w, y, bias, s_layout)
    _validate("fp8bq_gemm", specs + [_ws(ws)], stream)
    _check(_lib.fp8bq_gemm(_ptr(q), _ptr(s_x), s_layout, _ptr(w), _ptr(s_w), _ptr(bias),
                           _ptr(y), M, N, K, _ptr(ws), _nbytes(ws), _stream(stream)),
           "fp8bq_gemm")


def fp8bq_gemm_noalloc(q, s_x, w, s_w, y, bias=None, s_layout: int = SCALE_ROW_MAJOR,
                       stream=None):
    """fp8bq_gemm on the library's fixed device scratch instead of a workspace
    (for callers that may not allocate device memory); see include/fp8bq.h."""
    M, N, K, specs = _block_gemm_specs(q, s_x, w, s_w, y, bias, s_layout)
    _validate("fp8bq_gemm_noalloc", specs, stream)
    _check(_lib.fp8bq_gemm_noalloc(_ptr(q), _ptr(s_x), s_layout, _ptr(w), _ptr(s_w),
                                   _ptr(bias), _ptr(y), M, N, K, _stream(stream)),
           "fp8bq_gemm_noalloc")


def _linear_specs(x, w, y, bias):
    M, K = _mat(x, "x")
    N = _mat(w, "w")[0]
    return M, N, K, [
        _Spec("x", x, _BF16, (M, K), kind="rows"),
        _Spec("w", w, _E4M3, (N, K)),
        _Spec("y", y, _BF16, (M, N)),
        _bias(bias, N)]


def fp8bq_noalloc_poll_status(stream=None) -> int:
    """Synchronises the stream; 0, or 8 (FP8BQ_ERR_TIMEOUT) if a wait of an
    fp8bq_gemm_noalloc call on this device ran out."""
    return _lib.fp8bq_noalloc_poll_status(_stream(stream))


def fp8bq_linear(x, w, s_w, y, ws, bias=None, stream=None):
    M, N, K, specs = _linear_specs(x, w, y, bias)
    _validate("fp8bq_linear", specs + [_Spec("s_w", s_w, _F32, (_kb(N), _kb(K))), _ws(ws)],
              stream)
    _check(_lib.fp8bq_linear(_ptr(x), _ld(x), _ptr(w), _ptr(s_w), _ptr(bias), _ptr(y),
                             M, N, K, _ptr(ws), _nbytes(ws), _stream(stream)),
           "fp8bq_linear")


# ---------------------------------------------------------------- MX path

def fp8bq_mx_quant_act(x, q, s, stream=None):
    M, K = _mat(x, "x")
    _validate("fp8bq_mx_quant_act", [
        _Spec("x", x, _BF16, (M, K), kind="rows"),
        _Spec("q", q, _E4M3, (M, K)),
        _Spec("s", s, _U8, (M, K // 32))], stream)
    _check(_lib.fp8bq_mx_quant_act(_ptr(x), M, K, _ld(x), _ptr(q), _ptr(s),
                                   _stream(stream)), "fp8bq_mx_quant_act")


def fp8bq_mx_gemm(q, s_x, w, s_w, y, ws, bias=None, stream=None):
    M, K = _mat(q, "q")
    N = _mat(w, "w")[0]
    _validate("fp8bq_mx_gemm", [
        _Spec("q", q, _E4M3, (M, K)),
        _Spec("s_x", s_x, _U8, (M, K // 32)),
        _Spec("w", w, _E4M3, (N, K)),
        _Spec("s_w", s_w, _U8, (N, K // 32)),
        _Spec("y", y, _BF16, (M, N)), _bias(bias, N), _ws(ws)], stream)
    _check(_lib.fp8bq_mx_gemm(_ptr(q), _ptr(s_x), _ptr(w), _ptr(s_w), _ptr(bias), _ptr(y),
                              M, N, K, _ptr(ws), _nbytes(ws), _stream(stream)),
           "fp8bq_mx_gemm")


def fp8bq_mx_linear(x, w, s_w, y, ws, bias=None, stream=None):
    M, N, K, specs = _linear_specs(x, w, y, bias)
    _validate("fp8bq_mx_linear", specs + [_Spec("s_w", s_w, _U8, (N, K // 32)), _ws(ws)],
              stream)
    _check(_lib.fp8bq_mx_linear(_ptr(x), _ld(x), _ptr(w), _ptr(s_w), _ptr(bias), _ptr(y),
                                M, N, K, _ptr(ws), _nbytes(ws), _stream(stream)),
           "fp8bq_mx_linear")


# ---------------------------------------------------------------- static path

def _parts(part_sizes):
    arr = (ctypes.c_int64 * len(part_sizes))(*[int(p) for p in part_sizes])
    return arr, len(part_sizes)


def fp8bq_static_quant_act(x, s_x, q, stream=None):
    M, K = _mat(x, "x")
    _validate("fp8bq_static_quant_act", [
        _Spec("x", x, _BF16, (M, K), kind="rows"),
        _Spec("s_x", s_x, _F32, numel=1),
        _Spec("q", q, _E4M3, (M, K))], stream)
    _check(_lib.fp8bq_static_quant_act(_ptr(x), M, K, _ld(x), _ptr(s_x), _ptr(q),
                                       _stream(stream)), "fp8bq_static_quant_act")


def fp8bq_channel_quant_act(x, q, s, stream=None):
    """One scale per row (per-token activations, or per-channel weights)."""
    M, K = _mat(x, "x")
    _validate("fp8bq_channel_quant_act", [
        _Spec("x", x, _BF16, (M, K), kind="rows"),
        _Spec("q", q, _E4M3, (M, K)),
        _Spec("s", s, _F32, numel=M)], stream)
    _check(_lib.fp8bq_channel_quant_act(_ptr(x), M, K, _ld(x), _ptr(q), _ptr(s),
                                        _stream(stream)), "fp8bq_channel_quant_act")


def fp8bq_channel_gemm(q, s_x, w, s_w, y, ws, bias=None, stream=None):
    M, K = _mat(q, "q")
    N = _mat(w, "w")[0]
    _validate("fp8bq_channel_gemm", [
        _Spec("q", q, _E4M3, (M, K)),
        _Spec("s_x", s_x, _F32, numel=M),
        _Spec("w", w, _E4M3, (N, K)),
        _Spec("s_w", s_w, _F32, numel=N),
        _Spec("y", y, _BF16, (M, N)), _bias(bias, N), _ws(ws)], stream)
    _check(_lib.fp8bq_channel_gemm(_ptr(q), _ptr(s_x), _ptr(w), _ptr(s_w), _ptr(bias), _ptr(y),
                                   M, N, K, _ptr(ws), _nbytes(ws), _stream(stream)),
           "fp8bq_channel_gemm")


def fp8bq_channel_linear(x, w, s_w, y, ws, bias=None, stream=None):
    M, N, K, specs = _linear_specs(x, w, y, bias)
    _validate("fp8bq_channel_linear", specs + [_Spec("s_w", s_w, _F32, numel=N), _ws(ws)],
              stream)
    _check(_lib.fp8bq_channel_linear(_ptr(x), _ld(x), _ptr(w), _ptr(s_w), _ptr(bias), _ptr(y),
                                     M, N, K, _ptr(ws), _nbytes(ws), _stream(stream)),
           "fp8bq_channel_linear")


def fp8bq_quant_act_ue8m0(x, q, u, stream=None):
    """Group-128 quantisation with power-of-two (UE8M0) scales."""
    M, K = _mat(x, "x")
    _validate("fp8bq_quant_act_ue8m0", [
        _Spec("x", x, _BF16, (M, K), kind="rows"),
        _Spec("q", q, _E4M3, (M, K)),
        _Spec("u", u, _U8, (M, _kb(K)))], stream)
    _check(_lib.fp8bq_quant_act_ue8m0(_ptr(x), M, K, _ld(x), _ptr(q), _ptr(u), _stream(stream)),
           "fp8bq_quant_act_ue8m0")


def fp8bq_requant_weight_ue8m0(q, s_w, q_out, u_w, stream=None):
    """FP32 128x128 block scales -> UE8M0 (rounded up), codes re-encoded."""
    N, K = _mat(q, "q")
    _validate("fp8bq_requant_weight_ue8m0", [
        _Spec("q", q, _E4M3, (N, K)),
        _Spec("s_w", s_w, _F32, (_kb(N), _kb(K))),
        _Spec("q_out", q_out, _E4M3, (N, K)),
        _Spec("u_w", u_w, _U8, (_kb(N), _kb(K)))], stream)
    _check(_lib.fp8bq_requant_weight_ue8m0(_ptr(q), _ptr(s_w), N, K, _ptr(q_out), _ptr(u_w),
                                           _stream(stream)), "fp8bq_requant_weight_ue8m0")


def fp8bq_ue8m0_gemm(q, u_x, w, u_w, y, ws, bias=None, stream=None):
    M, K = _mat(q, "q")
    N = _mat(w, "w")[0]
    _validate("fp8bq_ue8m0_gemm", [
        _Spec("q", q, _E4M3, (M, K)),
        _Spec("u_x", u_x, _U8, (M, _kb(K))),
        _Spec("w", w, _E4M3, (N, K)),
        _Spec("u_w", u_w, _U8, (_kb(N), _kb(K))),
        _Spec("y", y, _BF16, (M, N)), _bias(bias, N), _ws(ws)], stream)
    _check(_lib.fp8bq_ue8m0_gemm(_ptr(q), _ptr(u_x), _ptr(w), _ptr(u_w), _ptr(bias), _ptr(y),
                                 M, N, K, _ptr(ws), _nbytes(ws), _stream(stream)),
           "fp8bq_ue8m0_gemm")


def fp8bq_ue8m0_linear(x, w, u_w, y, ws, bias=None, stream=None):
    M, N, K, specs = _linear_specs(x, w, y, bias)
    _validate("fp8bq_ue8m0_linear",
              specs + [_Spec("u_w", u_w, _U8, (_kb(N), _kb(K))), _ws(ws)], stream)
    _check(_lib.fp8bq_ue8m0_linear(_ptr(x), _ld(x), _ptr(w), _ptr(u_w), _ptr(bias), _ptr(y),
                                   M, N, K, _ptr(ws), _nbytes(ws), _stream(stream)),
           "fp8bq_ue8m0_linear")


def fp8bq_check_scales(s, scratch=None, stream=None) -> dict:
    """Counts unusable FP32 scales in a device tensor: the unloaded sentinel
    (-FLT_MAX), NaN / inf, other values <= 0; and the first bad flat index."""
    if scratch is None and isinstance(s, torch.Tensor):
        scratch = torch.empty(4, dtype=torch.int64, device=s.device)
    _validate("fp8bq_check_scales", [
        _Spec("s", s, _F32, numel=s.numel() if isinstance(s, torch.Tensor) else None),
        _Spec("scratch", scratch, (torch.int64,), numel=4)], stream)
    counts = (ctypes.c_int64 * 3)()
    first = ctypes.c_int64()
    _check(_lib.fp8bq_check_scales(_ptr(s), s.numel(), _ptr(scratch),
                                   ctypes.c_void_p(ctypes.addressof(counts)),
                                   ctypes.c_void_p(ctypes.addressof(first)), _stream(stream)),
           "fp8bq_check_scales")
    return {"sentinel": counts[0], "nonfinite": counts[1], "nonpositive": counts[2],
            "first_bad": first.value}


# ---------------------------------------------------------------- grouped (MoE)

def _experts_w(w):
    if not isinstance(w, torch.Tensor) or w.dim() != 3:
        raise ValueError("w must be a 3-D tensor [E, N, K]")
    return (int(v) for v in w.shape)


def fp8bq_grouped_gemm(q, s_x, w, s_w, offsets, y, ws, s_layout: int = SCALE_ROW_MAJOR,
                       stream=None):
    """Rows offsets[e] .. offsets[e+1]-1 of q / y use expert e's weight w[e]
    [N, K] and scale grid s_w[e]; offsets is a device int32 tensor [E+1]."""
    M, K = _mat(q, "q")
    E, N, Kw = _experts_w(w)
    if Kw != K:
        raise ValueError(f"fp8bq_grouped_gemm: w has K = {Kw}, q has K = {K}")
    _validate("fp8bq_grouped_gemm", [
        _Spec("q", q, _E4M3, (M, K)),
        _Spec("s_x", s_x, _F32, _sx_shape(M, K, s_layout)),
        _Spec("w", w, _E4M3, (E, N, K)),
        _Spec("s_w", s_w, _F32, (E, _kb(N), _kb(K))),
        _Spec("offsets", offsets, _I32, numel=E + 1),
        _Spec("y", y, _BF16, (M, N)), _ws(ws)], stream)
    _check(_lib.fp8bq_grouped_gemm(_ptr(q), _ptr(s_x), s_layout, _ptr(w), _ptr(s_w),
                                   _ptr(offsets), E, _ptr(y), M, N, K, _ptr(ws), _nbytes(ws),
                                   _stream(stream)), "fp8bq_grouped_gemm")


def fp8bq_grouped_gemm_masked(q, s_x, w, s_w, masked_m, y, ws, s_layout: int = SCALE_ROW_MAJOR,
                              stream=None):
    """q [E, max_m, K] (or [E*max_m, K]); the first masked_m[e] rows of slot e
    use expert e's weight; masked_m is a device int32 tensor [E]."""
    E, N, K = _experts_w(w)
    if not isinstance(q, torch.Tensor) or E == 0 or q.numel() % (K * E):
        raise ValueError(f"fp8bq_grouped_gemm_masked: q must hold E * max_m rows of K = {K}")
    max_m = q.numel() // (K * E)
    rows = E * max_m
    _validate("fp8bq_grouped_gemm_masked", [
        _Spec("q", q, _E4M3, numel=rows * K),
        _Spec("s_x", s_x, _F32, numel=_sx_shape(rows, K, s_layout)[0] *
              _sx_shape(rows, K, s_layout)[1]),
        _Spec("w", w, _E4M3, (E, N, K)),
        _Spec("s_w", s_w, _F32, (E, _kb(N), _kb(K))),
        _Spec("masked_m", masked_m, _I32, numel=E),
        _Spec("y", y, _BF16, numel=rows * N), _ws(ws)], stream)
    _check(_lib.fp8bq_grouped_gemm_masked(_ptr(q), _ptr(s_x), s_layout, _ptr(w), _ptr(s_w),
                                          _ptr(masked_m), E, max_m, _ptr(y), N, K, _ptr(ws),
                                          _nbytes(ws), _stream(stream)),
           "fp8bq_grouped_gemm_masked")


# ---------------------------------------------------------------- residual add + RMSNorm

def _norm_specs(x, gamma, residual, residual_out, y):
    M, K = _mat(x, "x")
    return M, K, [
        _Spec("x", x, _BF16, (M, K), kind="rows"),
        _Spec("gamma", gamma, _BF16, numel=K),
        _Spec("residual", residual, _BF16, (M, K), kind="rows", optional=True),
        _Spec("residual_out", residual_out, _BF16, (M, K), optional=True),
        _Spec("y", y, _BF16, (M, K), optional=True)]


def fp8bq_add_rmsnorm_quant_act(x, gamma, eps: float, residual=None, residual_out=None,
                                y=None, q=None, s=None, s_layout: int = SCALE_ROW_MAJOR,
                                stream=None):
    """Residual add + RMSNorm (+ group-128 quantisation when q is given)."""
    M, K, specs = _norm_specs(x, gamma, residual, residual_out, y)
    if q is not None:
        specs += [_Spec("q", q, _E4M3, (M, K)), _Spec("s", s, _F32, _sx_shape(M, K, s_layout))]
    _validate("fp8bq_add_rmsnorm_quant_act", specs, stream)
    _check(_lib.fp8bq_add_rmsnorm_quant_act(
        _ptr(x), _ld(x), _ptr(residual), 0 if residual is None else _ld(residual),
        _ptr(residual_out), _ptr(gamma), float(eps), M, K, _ptr(y), _ptr(q), _ptr(s),
        s_layout, _stream(stream)), "fp8bq_add_rmsnorm_quant_act")


def fp8bq_add_rmsnorm_static_quant_act(x, gamma, eps: float, s_x, q, residual=None,
                                       residual_out=None, y=None, stream=None):
    """Residual add + RMSNorm, then static per-tensor quantisation with s_x[0]."""
    M, K, specs = _norm_specs(x, gamma, residual, residual_out, y)
    specs += [_Spec("s_x", s_x, _F32, numel=1), _Spec("q", q, _E4M3, (M, K))]
    _validate("fp8bq_add_rmsnorm_static_quant_act", specs, stream)
    _check(_lib.fp8bq_add_rmsnorm_static_quant_act(
        _ptr(x), _ld(x), _ptr(residual), 0 if residual is None else _ld(residual),
        _ptr(residual_out), _ptr(gamma), float(eps), _ptr(s_x), M, K, _ptr(y), _ptr(q),
        _stream(stream)), "fp8bq_add_rmsnorm_static_quant_act")


# ---------------------------------------------------------------- static GEMM

def fp8bq_static_gemm(q, s_x, w, s_w_part, part_sizes, y, ws, bias=None, stream=None):
    M, K = _mat(q, "q")
    N = _mat(w, "w")[0]
    arr, n = _parts(part_sizes)
    _validate("fp8bq_static_gemm", [
        _Spec("q", q, _E4M3, (M, K)),
        _Spec("s_x", s_x, _F32, numel=1),
        _Spec("w", w, _E4M3, (N, K)),
        _Spec("s_w_part", s_w_part, _F32, numel=n),
        _Spec("y", y, _BF16, (M, N)), _bias(bias, N), _ws(ws)], stream)
    _check(_lib.fp8bq_static_gemm(_ptr(q), _ptr(s_x), _ptr(w), _ptr(s_w_part), arr, n,
                                  _ptr(bias), _ptr(y), M, N, K, _ptr(ws), _nbytes(ws),
                                  _stream(stream)), "fp8bq_static_gemm")


def fp8bq_static_linear(x, s_x, w, s_w_part, part_sizes, y, ws, bias=None, stream=None):
    M, N, K, specs = _linear_specs(x, w, y, bias)
    arr, n = _parts(part_sizes)
    _validate("fp8bq_static_linear", specs + [
        _Spec("s_x", s_x, _F32, numel=1),
        _Spec("s_w_part", s_w_part, _F32, numel=n), _ws(ws)], stream)
    _check(_lib.fp8bq_static_linear(_ptr(x), _ld(x), _ptr(s_x), _ptr(w), _ptr(s_w_part),
                                    arr, n, _ptr(bias), _ptr(y), M, N, K, _ptr(ws),
                                    _nbytes(ws), _stream(stream)), "fp8bq_static_linear")


# ---------------------------------------------------------------- set-up helpers

def fp8bq_quant_weight_block(w, q, s_w, stream=None):
    N, K = _mat(w, "w")
    _validate("fp8bq_quant_weight_block", [
        _Spec("w", w, _BF16, (N, K), kind="rows"),
        _Spec("q", q, _E4M3, (N, K)),
        _Spec("s_w", s_w, _F32, (_kb(N), _kb(K)))], stream)
    _check(_lib.fp8bq_quant_weight_block(_ptr(w), N, K, _ld(w), _ptr(q), _ptr(s_w),
                                         _stream(stream)), "fp8bq_quant_weight_block")


def fp8bq_absmax_scale(x, s, stream=None):
    rows, K = _mat(x, "x")
    _validate("fp8bq_absmax_scale", [
        _Spec("x", x, _BF16, (rows, K), kind="rows"),
        _Spec("s", s, _F32, numel=1)], stream)
    _check(_lib.fp8bq_absmax_scale(_ptr(x), rows, K, _ld(x), _ptr(s), _stream(stream)),
           "fp8bq_absmax_scale")


def fp8bq_e4m3_from_bits(first: int, codes, stream=None):
    """codes[i] = the quantisers' E4M3 conversion of the binary32 value with bit
    pattern first + i, for every element of the uint8 tensor `codes`."""
    _validate("fp8bq_e4m3_from_bits", [_Spec("codes", codes, _U8, numel=codes.numel()
                                             if isinstance(codes, torch.Tensor) else None)],
              stream)
    _check(_lib.fp8bq_e4m3_from_bits(first, codes.numel(), _ptr(codes), _stream(stream)),
           "fp8bq_e4m3_from_bits")
