"""CPU oracle for the block-wise FP8 W8A8 linear (test infrastructure only).

Only the test-suite, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may import this package.  The CUDA
library never calls it, and it shares no code with the CUDA library: the C
source next to this file (``fp8bq_oracle.c``) restates the pages' definitions
in plain loops, binary32 for the scale and quotient divisions the pages write
down and binary64 for everything after decoding.

BF16 tensors cross this interface as ``numpy.uint16`` bit patterns; E4M3 codes
and UE8M0 scale codes as ``numpy.uint8``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "fp8bq_oracle.c")
_HDR = os.path.join(_HERE, "fp8bq_oracle.h")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB = os.path.join(_OUT_DIR, "liboracle.so")
_CFLAGS = ["-O2", "-ffp-contract=off", "-fno-fast-math", "-std=c11", "-Wall",
           "-fPIC", "-shared"]

_lock = threading.Lock()
_handle = None


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/_build/liboracle.so`` with gcc."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    newest = max(os.path.getmtime(_SRC), os.path.getmtime(_HDR))
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= newest:
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", *_CFLAGS, _SRC, "-o", tmp, "-lpthread", "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_SIGS = {
    "orc_e4m3_encode": (ctypes.c_uint8, [ctypes.c_double]),
    "orc_e4m3_decode": (ctypes.c_double, [ctypes.c_uint8]),
    "orc_e4m3_sig": (ctypes.c_int32, [ctypes.c_uint8]),
    "orc_ue8m0_decode": (ctypes.c_double, [ctypes.c_uint8]),
    "orc_bf16_to_f32": (ctypes.c_float, [ctypes.c_uint16]),
    "orc_e4m3_encode_f32_array": (None, [_P, _I64, _P]),
    "orc_e4m3_decode_array": (None, [_P, _I64, _P]),
    "orc_e4m3_encode_bits_range": (None, [ctypes.c_uint32, _I64, _P, ctypes.c_int]),
    "orc_quant_group": (None, [_P, _I64, _I64, _I64, _I64, _P, _P]),
    "orc_quant_mx": (None, [_P, _I64, _I64, _I64, _P, _P]),
    "orc_quant_static": (None, [_P, _I64, _I64, _I64, ctypes.c_float, _P]),
    "orc_absmax_scale": (ctypes.c_float, [_P, _I64, _I64, _I64, _I64]),
    "orc_quant_weight_block": (None, [_P, _I64, _I64, _I64, _I64, _I64, _P, _P]),
    "orc_quant_weight_static": (None, [_P, _I64, _I64, _I64, _P, ctypes.c_int, _P, _P]),
    "orc_gemm_block": (None, [_P, _P, _P, _P, _P, _I64, _I64, _I64, _I64, _I64, _P,
                              ctypes.c_int]),
    "orc_gemm_block_sampled": (None, [_P, _P, _P, _P, _P, _I64, _I64, _I64, _I64,
                                      _I64, _P, _P, _I64, _P, ctypes.c_int]),
    "orc_gemm_mx": (None, [_P, _P, _P, _P, _P, _I64, _I64, _I64, _P, ctypes.c_int]),
    "orc_gemm_mx_sampled": (None, [_P, _P, _P, _P, _P, _I64, _I64, _I64, _P, _P, _I64,
                                   _P, ctypes.c_int]),
    "orc_gemm_static": (None, [_P, ctypes.c_float, _P, _P, _P, ctypes.c_int, _P, _I64,
                               _I64, _I64, _P, ctypes.c_int]),
    "orc_gemm_static_sampled": (None, [_P, ctypes.c_float, _P, _P, _P, ctypes.c_int, _P,
                                       _I64, _I64, _I64, _P, _P, _I64, _P,
                                       ctypes.c_int]),
    "orc_bf16_from_f64": (ctypes.c_uint16, [ctypes.c_double]),
    "orc_sumsq_f32": (ctypes.c_float, [_P, _I64]),
    "orc_add_rmsnorm": (None, [_P, _I64, _P, _I64, _P, ctypes.c_float, _I64, _I64, _P, _P]),
    "orc_gemm_channel": (None, [_P, _P, _P, _P, _P, _I64, _I64, _I64, _P, ctypes.c_int]),
    "orc_gemm_channel_sampled": (None, [_P, _P, _P, _P, _P, _I64, _I64, _I64, _P, _P, _I64,
                                        _P, ctypes.c_int]),
    "orc_quant_ue8m0": (None, [_P, _I64, _I64, _I64, _I64, _P, _P]),
    "orc_requant_weight_ue8m0": (None, [_P, _P, _I64, _I64, _I64, _I64, _P, _P]),
    "orc_gemm_grouped": (None, [_P, _P, _P, _P, _P, _I64, _I64, _I64, _P, ctypes.c_int]),
    "orc_gemm_grouped_sampled": (None, [_P, _P, _P, _P, _P, _I64, _I64, _I64, _P, _P, _I64,
                                        _P, ctypes.c_int]),
    "orc_e4m3_dot_int": (ctypes.c_int64, [_P, _P, _I64]),
    "orc_e4m3_dot_f64": (ctypes.c_double, [_P, _P, _I64]),
}


def lib():
    global _handle
    with _lock:
        if _handle is None:
            h = ctypes.CDLL(build())
            for name, (res, args) in _SIGS.items():
                fn = getattr(h, name)
                fn.restype = res
                fn.argtypes = args
            _handle = h
    return _handle


def default_threads() -> int:
    return os.cpu_count() or 1


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def _check_samples(rows, cols, M: int, N: int) -> None:
    """The C routines index with the sample coordinates unchecked, so reject
    any outside the [M, N] output before they reach it."""
    if rows.shape != cols.shape:
        raise ValueError(f"rows {rows.shape} and cols {cols.shape} differ")
    if rows.size and (rows.min() < 0 or rows.max() >= M or cols.min() < 0 or cols.max() >= N):
        raise ValueError(f"sample coordinates outside the {M} x {N} output")


# --------------------------------------------------------------------------
# number formats
# --------------------------------------------------------------------------

def e4m3_encode(v) -> np.ndarray:
    """binary32 values -> E4M3 codes (RNE, saturating at +-448)."""
    v = _c(v, np.float32)
    out = np.empty(v.shape, np.uint8)
    lib().orc_e4m3_encode_f32_array(_p(v), v.size, _p(out))
    return out


def e4m3_encode_bits_range(first: int, n: int, threads: int | None = None) -> np.ndarray:
    """Codes of the binary32 values whose bit patterns are first .. first + n - 1."""
    if first < 0 or n < 0 or first + n > 1 << 32:
        raise ValueError("bit patterns outside 0 .. 2^32 - 1")
    out = np.empty(n, np.uint8)
    lib().orc_e4m3_encode_bits_range(first, n, _p(out), threads or default_threads())
    return out


def e4m3_decode(c) -> np.ndarray:
    c = _c(c, np.uint8)
    out = np.empty(c.shape, np.float64)
    lib().orc_e4m3_decode_array(_p(c), c.size, _p(out))
    return out


def e4m3_sig(c: int) -> int:
    return int(lib().orc_e4m3_sig(int(c)))


def ue8m0_decode(u) -> np.ndarray:
    u = np.asarray(u, np.uint8)
    return np.array([lib().orc_ue8m0_decode(int(x)) for x in u.ravel()],
                    np.float64).reshape(u.shape)


def bf16_to_f32(b) -> np.ndarray:
    b = _c(b, np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32)


# --------------------------------------------------------------------------
# quantisers
# --------------------------------------------------------------------------

def quant_group(x, group: int = 128):
    """Per-token group quantisation -> (q [M,K] uint8, s [M,ceil(K/group)] f32)."""
    x = _c(x, np.uint16)
    M, K = x.shape
    G = -(-K // group)
    q = np.empty((M, K), np.uint8)
    s = np.empty((M, G), np.float32)
    lib().orc_quant_group(_p(x), M, K, K, group, _p(q), _p(s))
    return q, s


def quant_mx(x):
    """MXFP8 [1,32] quantisation -> (q [M,K] uint8, u [M,K/32] uint8)."""
    x = _c(x, np.uint16)
    M, K = x.shape
    if K % 32:
        raise ValueError("MXFP8 needs K % 32 == 0")
    q = np.empty((M, K), np.uint8)
    u = np.empty((M, K // 32), np.uint8)
    lib().orc_quant_mx(_p(x), M, K, K, _p(q), _p(u))
    return q, u


def quant_channel(x):
    """Per-token (or, for weights, per-channel) quantisation: one scale per row,
    the group rule with the group spanning the whole row -> (q [M,K], s [M])."""
    x = _c(x, np.uint16)
    q, s = quant_group(x, group=x.shape[1])
    return q, s.reshape(-1)


def quant_static(x, s: float):
    x = _c(x, np.uint16)
    M, K = x.shape
    q = np.empty((M, K), np.uint8)
    lib().orc_quant_static(_p(x), M, K, K, float(np.float32(s)), _p(q))
    return q


def absmax_scale(x, r0: int = 0, r1: int | None = None) -> np.float32:
    x = _c(x, np.uint16)
    M, K = x.shape
    r1 = M if r1 is None else r1
    return np.float32(lib().orc_absmax_scale(_p(x), r0, r1, K, K))


def quant_weight_block(w, bn: int = 128, bk: int = 128):
    """128x128 block quantisation -> (q [N,K] uint8, s [ceil(N/bn),ceil(K/bk)] f32)."""
    w = _c(w, np.uint16)
    N, K = w.shape
    q = np.empty((N, K), np.uint8)
    s = np.empty((-(-N // bn), -(-K // bk)), np.float32)
    lib().orc_quant_weight_block(_p(w), N, K, K, bn, bk, _p(q), _p(s))
    return q, s


def quant_weight_static(w, part_sizes):
    w = _c(w, np.uint16)
    N, K = w.shape
    parts = _c(part_sizes, np.int64)
    if int(parts.sum()) != N:
        raise ValueError("partition sizes must sum to N")
    q = np.empty((N, K), np.uint8)
    s = np.empty(parts.size, np.float32)
    lib().orc_quant_weight_static(_p(w), N, K, K, _p(parts), parts.size, _p(q), _p(s))
    return q, s


# --------------------------------------------------------------------------
# residual add + RMSNorm
# --------------------------------------------------------------------------

def bf16_from_f64(v: float) -> int:
    """binary64 -> BF16 bits (RNE, overflow to infinity)."""
    return int(lib().orc_bf16_from_f64(float(v)))


def sumsq_f32(r) -> np.float32:
    """Sum of squares of a BF16 row (uint16 bits), exact, rounded once to binary32."""
    r = _c(r, np.uint16).ravel()
    return np.float32(lib().orc_sumsq_f32(_p(r), r.size))


def add_rmsnorm(x, gamma, eps: float, residual=None):
    """r = BF16(x + residual), y = BF16(RMSNorm(r) * gamma) -> (r, y), uint16 [M,d]."""
    x = _c(x, np.uint16)
    M, d = x.shape
    g = _c(gamma, np.uint16).ravel()
    if g.size != d:
        raise ValueError("gamma must have d elements")
    res = None if residual is None else _c(residual, np.uint16)
    if res is not None and res.shape != x.shape:
        raise ValueError("residual must match x")
    r = np.empty((M, d), np.uint16)
    y = np.empty((M, d), np.uint16)
    lib().orc_add_rmsnorm(_p(x), d, _p(res), d, _p(g), float(np.float32(eps)), M, d,
                          _p(r), _p(y))
    return r, y


def add_rmsnorm_quant_group(x, gamma, eps: float, residual=None):
    """Residual add + RMSNorm, then group-128 quantisation of the BF16 output:
    -> (r, q, s)."""
    r, y = add_rmsnorm(x, gamma, eps, residual)
    q, s = quant_group(y)
    return r, q, s


def add_rmsnorm_quant_static(x, gamma, eps: float, s_x: float, residual=None):
    """Residual add + RMSNorm, then static per-tensor quantisation: -> (r, q)."""
    r, y = add_rmsnorm(x, gamma, eps, residual)
    return r, quant_static(y, s_x)


# --------------------------------------------------------------------------
# reference GEMMs (binary64 results)
# --------------------------------------------------------------------------

def _bias(bias):
    return None if bias is None else _c(bias, np.uint16)


def gemm_block(qa, sa, qw, sw, bias=None, bn: int = 128, bk: int = 128,
               threads: int | None = None) -> np.ndarray:
    qa, qw = _c(qa, np.uint8), _c(qw, np.uint8)
    sa, sw = _c(sa, np.float32), _c(sw, np.float32)
    M, K = qa.shape
    N = qw.shape[0]
    b = _bias(bias)
    y = np.empty((M, N), np.float64)
    lib().orc_gemm_block(_p(qa), _p(sa), _p(qw), _p(sw), _p(b), M, N, K, bn, bk,
                         _p(y), threads or default_threads())
    return y


def gemm_block_sampled(qa, sa, qw, sw, rows, cols, bias=None, bn: int = 128,
                       bk: int = 128, threads: int | None = None) -> np.ndarray:
    qa, qw = _c(qa, np.uint8), _c(qw, np.uint8)
    sa, sw = _c(sa, np.float32), _c(sw, np.float32)
    rows, cols = _c(rows, np.int64), _c(cols, np.int64)
    M, K = qa.shape
    N = qw.shape[0]
    b = _bias(bias)
    _check_samples(rows, cols, M, N)
    y = np.empty(rows.size, np.float64)
    lib().orc_gemm_block_sampled(_p(qa), _p(sa), _p(qw), _p(sw), _p(b), M, N, K, bn,
                                 bk, _p(rows), _p(cols), rows.size, _p(y),
                                 threads or default_threads())
    return y


def gemm_mx(qa, ua, qw, uw, bias=None, threads: int | None = None) -> np.ndarray:
    qa, qw = _c(qa, np.uint8), _c(qw, np.uint8)
    ua, uw = _c(ua, np.uint8), _c(uw, np.uint8)
    M, K = qa.shape
    N = qw.shape[0]
    b = _bias(bias)
    y = np.empty((M, N), np.float64)
    lib().orc_gemm_mx(_p(qa), _p(ua), _p(qw), _p(uw), _p(b), M, N, K, _p(y),
                      threads or default_threads())
    return y


def gemm_mx_sampled(qa, ua, qw, uw, rows, cols, bias=None,
                    threads: int | None = None) -> np.ndarray:
    qa, qw = _c(qa, np.uint8), _c(qw, np.uint8)
    ua, uw = _c(ua, np.uint8), _c(uw, np.uint8)
    rows, cols = _c(rows, np.int64), _c(cols, np.int64)
    M, K = qa.shape
    N = qw.shape[0]
    b = _bias(bias)
    _check_samples(rows, cols, M, N)
    y = np.empty(rows.size, np.float64)
    lib().orc_gemm_mx_sampled(_p(qa), _p(ua), _p(qw), _p(uw), _p(b), M, N, K,
                              _p(rows), _p(cols), rows.size, _p(y),
                              threads or default_threads())
    return y


def gemm_static(qa, s_x, qw, s_part, part_sizes, bias=None,
                threads: int | None = None) -> np.ndarray:
    qa, qw = _c(qa, np.uint8), _c(qw, np.uint8)
    s_part = _c(s_part, np.float32)
    parts = _c(part_sizes, np.int64)
    M, K = qa.shape
    N = qw.shape[0]
    b = _bias(bias)
    y = np.empty((M, N), np.float64)
    lib().orc_gemm_static(_p(qa), float(np.float32(s_x)), _p(qw), _p(s_part),
                          _p(parts), parts.size, _p(b), M, N, K, _p(y),
                          threads or default_threads())
    return y


def gemm_static_sampled(qa, s_x, qw, s_part, part_sizes, rows, cols, bias=None,
                        threads: int | None = None) -> np.ndarray:
    qa, qw = _c(qa, np.uint8), _c(qw, np.uint8)
    s_part = _c(s_part, np.float32)
    parts = _c(part_sizes, np.int64)
    rows, cols = _c(rows, np.int64), _c(cols, np.int64)
    M, K = qa.shape
    N = qw.shape[0]
    b = _bias(bias)
    _check_samples(rows, cols, M, N)
    y = np.empty(rows.size, np.float64)
    lib().orc_gemm_static_sampled(_p(qa), float(np.float32(s_x)), _p(qw), _p(s_part),
                                  _p(parts), parts.size, _p(b), M, N, K, _p(rows),
                                  _p(cols), rows.size, _p(y),
                                  threads or default_threads())
    return y


def e4m3_dot_int(a, b) -> int:
    a, b = _c(a, np.uint8), _c(b, np.uint8)
    return int(lib().orc_e4m3_dot_int(_p(a), _p(b), a.size))


def e4m3_dot_f64(a, b) -> float:
    a, b = _c(a, np.uint8), _c(b, np.uint8)
    return float(lib().orc_e4m3_dot_f64(_p(a), _p(b), a.size))


def gemm_channel(qa, sa, qw, sw, bias=None, threads: int | None = None) -> np.ndarray:
    """Channelwise GEMM: y[i,j] = (sum_k qa*qw) * sa[i] * sw[j] (+bias), binary64."""
    qa, qw = _c(qa, np.uint8), _c(qw, np.uint8)
    sa, sw = _c(sa, np.float32).ravel(), _c(sw, np.float32).ravel()
    M, K = qa.shape
    N = qw.shape[0]
    if sa.size != M or sw.size != N:
        raise ValueError("one activation scale per row, one weight scale per output channel")
    b = _bias(bias)
    y = np.empty((M, N), np.float64)
    lib().orc_gemm_channel(_p(qa), _p(sa), _p(qw), _p(sw), _p(b), M, N, K, _p(y),
                           threads or default_threads())
    return y


def gemm_channel_sampled(qa, sa, qw, sw, rows, cols, bias=None,
                         threads: int | None = None) -> np.ndarray:
    qa, qw = _c(qa, np.uint8), _c(qw, np.uint8)
    sa, sw = _c(sa, np.float32).ravel(), _c(sw, np.float32).ravel()
    rows, cols = _c(rows, np.int64), _c(cols, np.int64)
    M, K = qa.shape
    N = qw.shape[0]
    b = _bias(bias)
    _check_samples(rows, cols, M, N)
    y = np.empty(rows.size, np.float64)
    lib().orc_gemm_channel_sampled(_p(qa), _p(sa), _p(qw), _p(sw), _p(b), M, N, K, _p(rows),
                                   _p(cols), rows.size, _p(y), threads or default_threads())
    return y


# --------------------------------------------------------------------------
# block FP8 with UE8M0 (power-of-two) scales
# --------------------------------------------------------------------------

def quant_ue8m0(x, group: int = 128):
    """Group quantisation with power-of-two scales -> (q [M,K], u [M,ceil(K/group)])."""
    x = _c(x, np.uint16)
    M, K = x.shape
    G = -(-K // group)
    q = np.empty((M, K), np.uint8)
    u = np.empty((M, G), np.uint8)
    lib().orc_quant_ue8m0(_p(x), M, K, K, group, _p(q), _p(u))
    return q, u


def requant_weight_ue8m0(q, s, bn: int = 128, bk: int = 128):
    """FP32 block scales -> UE8M0 rounded up, codes re-encoded -> (q2 [N,K], u [NB,KB])."""
    q = _c(q, np.uint8)
    s = _c(s, np.float32)
    N, K = q.shape
    q2 = np.empty((N, K), np.uint8)
    u = np.empty(s.shape, np.uint8)
    lib().orc_requant_weight_ue8m0(_p(q), _p(s), N, K, bn, bk, _p(q2), _p(u))
    return q2, u


def ue8m0_to_f32(u) -> np.ndarray:
    """UE8M0 codes 1..254 as the binary32 powers of two they stand for."""
    u = np.asarray(u, np.uint8)
    return ue8m0_decode(u).astype(np.float32)


def gemm_block_ue8m0(qa, ua, qw, uw, bias=None, threads: int | None = None) -> np.ndarray:
    """Block-scaled GEMM whose 128-block scales are powers of two (the block
    definition with s = 2^(u - 127)), binary64."""
    return gemm_block(qa, ue8m0_to_f32(ua), qw, ue8m0_to_f32(uw), bias=bias, threads=threads)


def gemm_block_ue8m0_sampled(qa, ua, qw, uw, rows, cols, bias=None,
                             threads: int | None = None) -> np.ndarray:
    return gemm_block_sampled(qa, ue8m0_to_f32(ua), qw, ue8m0_to_f32(uw), rows, cols,
                              bias=bias, threads=threads)


# --------------------------------------------------------------------------
# grouped (MoE) block-scaled GEMM
# --------------------------------------------------------------------------

def row_expert_contiguous(offsets, T: int) -> np.ndarray:
    """Expert of each row when rows are sorted by expert: rows offsets[e] ..
    offsets[e+1]-1 belong to expert e; rows outside every range get -1."""
    off = np.clip(np.asarray(offsets, np.int64), 0, T)   # bounds outside [0, T] clamp
    r = np.full(T, -1, np.int32)
    for e in range(off.size - 1):
        r[off[e]:off[e + 1]] = e
    return r


def row_expert_masked(masked_m, max_m: int) -> np.ndarray:
    """Expert of each row of the masked layout [E, max_m, K]: the first
    masked_m[e] rows of slot e belong to expert e, the rest to none (-1)."""
    m = np.clip(np.asarray(masked_m, np.int64), 0, max_m)  # counts clamp to [0, max_m]
    r = np.full(m.size * max_m, -1, np.int32)
    for e in range(m.size):
        r[e * max_m:e * max_m + int(m[e])] = e
    return r


def gemm_grouped(qa, sa, qw, sw, row_expert, threads: int | None = None) -> np.ndarray:
    """y[i, j] = block GEMM element of row i with its expert's weight qw[e] [N,K]
    and scale grid sw[e]; rows of no expert are NaN.  binary64."""
    qa, qw = _c(qa, np.uint8), _c(qw, np.uint8)
    sa, sw = _c(sa, np.float32), _c(sw, np.float32)
    re = _c(row_expert, np.int32).ravel()
    M, K = qa.shape
    E, N, K2 = qw.shape
    if K2 != K or re.size != M or sw.shape[0] != E:
        raise ValueError("shape mismatch")
    y = np.empty((M, N), np.float64)
    lib().orc_gemm_grouped(_p(qa), _p(sa), _p(qw), _p(sw), _p(re), M, N, K, _p(y),
                           threads or default_threads())
    return y


def gemm_grouped_sampled(qa, sa, qw, sw, row_expert, rows, cols,
                         threads: int | None = None) -> np.ndarray:
    qa, qw = _c(qa, np.uint8), _c(qw, np.uint8)
    sa, sw = _c(sa, np.float32), _c(sw, np.float32)
    re = _c(row_expert, np.int32).ravel()
    rows, cols = _c(rows, np.int64), _c(cols, np.int64)
    M, K = qa.shape
    E, N, _ = qw.shape
    _check_samples(rows, cols, M, N)
    y = np.empty(rows.size, np.float64)
    lib().orc_gemm_grouped_sampled(_p(qa), _p(sa), _p(qw), _p(sw), _p(re), M, N, K, _p(rows),
                                   _p(cols), rows.size, _p(y), threads or default_threads())
    return y
