"""Seeded synthetic inputs for the block-wise FP8 linear.

This module is the only thing the CUDA path and the CPU oracle share: it draws
BF16 activations, weights and calibration batches and holds none of the
method's arithmetic (no scale, no quantisation, no GEMM).

Recipe (identical on every machine that runs the same numpy):
  * splitmix64 as a counter-based generator: output i of stream s is
    mix64(seed_s + (i + 1) * 0x9E3779B97F4A7C15), seed_s = base_seed + s.
    Streams: 0 = activations X, 1 = weights W, 2 = calibration batch,
    3 = outlier-channel pick, 4 = residual stream, 5 = norm gains,
    6 = MoE routing.
  * uniform u = (z >> 11) * 2^-53; normal by Box-Muller (cosine branch), element
    e using outputs 2e and 2e+1: sqrt(-2 ln(1 - u0)) * cos(2 pi u1).
  * value = sigma * normal, times `outlier_scale` on the outlier channels, then
    rounded binary64 -> binary32 -> BF16 (nearest-even at each step).
  * outlier channels: round(frac * K) channels from a partial Fisher-Yates
    shuffle of 0..K-1 driven by stream 3.
  * residual stream: sigma 4, the outlier channels x20 (the large channels of
    a transformer's residual stream); norm gains: exp(0.5 * normal), a
    positive log-normal spread around 1.
  * MoE routing (rows per local expert): T routed rows each pick expert
    perm[r] with probability proportional to (r + 1)^-skew, r the inverse-CDF
    rank of a stream-6 uniform and perm a Fisher-Yates shuffle of the experts
    driven by the same stream (after the T row draws); skew 0.5 gives hot
    experts at about 3x the mean load and cold ones at about 0.5x.

BF16 tensors are returned as numpy.uint16 bit patterns, row-major.
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)

STREAM_X, STREAM_W, STREAM_CALIB, STREAM_OUTLIER = 0, 1, 2, 3
STREAM_RES, STREAM_GAIN = 4, 5
STREAM_ROUTE = 6


def _mix64(z: np.ndarray) -> np.ndarray:
    """splitmix64's output mix, in place on a uint64 array."""
    with np.errstate(over="ignore"):
        z ^= z >> np.uint64(30)
        z *= _M1
        z ^= z >> np.uint64(27)
        z *= _M2
        z ^= z >> np.uint64(31)
    return z


def splitmix64(seed: int, start: int, count: int) -> np.ndarray:
    """Outputs start .. start+count-1 of the splitmix64 sequence seeded `seed`."""
    z = np.arange(start + 1, start + count + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z *= GOLDEN
        z += np.uint64(seed & 0xFFFFFFFFFFFFFFFF)
    return _mix64(z)


def _uniform(z: np.ndarray) -> np.ndarray:
    return (z >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)


def _normals(seed: int, start: int, count: int) -> np.ndarray:
    z = splitmix64(seed, 2 * start, 2 * count).reshape(count, 2)
    u0 = _uniform(z[:, 0])
    u1 = _uniform(z[:, 1])
    del z
    np.negative(u0, out=u0)
    np.log1p(u0, out=u0)
    u0 *= -2.0
    np.sqrt(u0, out=u0)
    u1 *= 2.0 * np.pi
    np.cos(u1, out=u1)
    u0 *= u1
    return u0


def f32_to_bf16_bits(v: np.ndarray) -> np.ndarray:
    """binary32 -> BF16 bit patterns, round to nearest even (finite inputs)."""
    u = np.ascontiguousarray(v, dtype=np.float32).view(np.uint32)
    r = (u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    return r.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32)
            << np.uint32(16)).view(np.float32)


def outlier_channels(K: int, frac: float = 0.01, base_seed: int = 0) -> np.ndarray:
    """round(frac*K) distinct channels, sorted, from stream 3."""
    n = int(round(frac * K))
    if n <= 0:
        return np.zeros(0, np.int64)
    perm = np.arange(K, dtype=np.int64)
    z = splitmix64(base_seed + STREAM_OUTLIER, 0, n)
    for t in range(n):
        j = t + int(z[t] % np.uint64(K - t))
        perm[t], perm[j] = perm[j], perm[t]
    return np.sort(perm[:n])


def normal_bf16(rows: int, cols: int, sigma: float, stream: int,
                base_seed: int = 0, outlier_cols: np.ndarray | None = None,
                outlier_scale: float = 50.0, row_start: int = 0,
                chunk_elems: int = 1 << 22, threads: int | None = None) -> np.ndarray:
    """[rows, cols] BF16 bit patterns; rows row_start.. of the stream's matrix.

    Chunks are independent slices of the counter-based stream, so the thread
    count never changes the result."""
    out = np.empty((rows, cols), np.uint16)
    seed = base_seed + stream
    rows_per_chunk = max(1, chunk_elems // max(cols, 1))
    mult = None
    if outlier_cols is not None and len(outlier_cols):
        mult = np.ones(cols, np.float64)
        mult[np.asarray(outlier_cols, np.int64)] = outlier_scale

    def fill(r0: int) -> None:
        r1 = min(rows, r0 + rows_per_chunk)
        v = _normals(seed, (row_start + r0) * cols, (r1 - r0) * cols).reshape(r1 - r0, cols)
        v *= sigma
        if mult is not None:
            v *= mult[None, :]
        out[r0:r1] = f32_to_bf16_bits(v.astype(np.float32))

    starts = list(range(0, rows, rows_per_chunk))
    nthreads = threads or min(16, os.cpu_count() or 1)
    if nthreads <= 1 or len(starts) <= 1:
        for r0 in starts:
            fill(r0)
    else:
        with ThreadPoolExecutor(nthreads) as ex:
            list(ex.map(fill, starts))
    return out


# ---------------------------------------------------------------------------
# The workloads: shapes and value distributions of the pages' model layers.
# ---------------------------------------------------------------------------

def activations(M: int, K: int, outliers: bool = True, base_seed: int = 0,
                frac: float = 0.01, outlier_scale: float = 50.0) -> np.ndarray:
    """X ~ N(0,1) [M, K]; with `outliers`, round(1% of K) channels x50."""
    oc = outlier_channels(K, frac, base_seed) if outliers else None
    return normal_bf16(M, K, 1.0, STREAM_X, base_seed, oc, outlier_scale)


def weights(N: int, K: int, sigma: float = 0.02, base_seed: int = 0) -> np.ndarray:
    """W ~ N(0, sigma) [N, K]."""
    return normal_bf16(N, K, sigma, STREAM_W, base_seed)


def calibration(rows: int, K: int, base_seed: int = 0) -> np.ndarray:
    """Calibration batch ~ N(0,1) [rows, K] for a static activation scale."""
    return normal_bf16(rows, K, 1.0, STREAM_CALIB, base_seed)


def residual_stream(M: int, K: int, base_seed: int = 0) -> np.ndarray:
    """Residual stream R ~ N(0, 4^2) [M, K], outlier channels x20."""
    return normal_bf16(M, K, 4.0, STREAM_RES, base_seed, outlier_channels(K, 0.01, base_seed), 20.0)


def norm_gain(K: int, base_seed: int = 0) -> np.ndarray:
    """Per-channel norm gains g = exp(0.5 * N(0,1)) [K] as BF16 bits."""
    z = _normals(base_seed + STREAM_GAIN, 0, K)
    return f32_to_bf16_bits(np.exp(0.5 * z).astype(np.float32))


def expert_counts(T: int, E: int, skew: float = 0.5, base_seed: int = 0) -> np.ndarray:
    """Rows per expert (int64 [E], summing to T) for T routed rows."""
    seed = base_seed + STREAM_ROUTE
    p = np.arange(1, E + 1, dtype=np.float64) ** -skew
    cdf = np.cumsum(p / p.sum())
    u = _uniform(splitmix64(seed, 0, T))
    rank = np.minimum(np.searchsorted(cdf, u, side="right"), E - 1)
    perm = np.arange(E)
    z = splitmix64(seed, T, E)
    for i in range(E - 1, 0, -1):
        j = int(z[i] % np.uint64(i + 1))
        perm[i], perm[j] = perm[j], perm[i]
    return np.bincount(perm[rank], minlength=E).astype(np.int64)


# Shapes of the five workloads.
TINY = dict(M=16, K=256, N=384)
DECODE = dict(K=6144, N=6144, M_list=(1, 8, 32, 64))
PREFILL = dict(M=4096, K=6144, N_list=(6144, 24576))
MXFP8 = dict(M=2048, K=7168, N=4096)
# residual add + RMSNorm + quantisation before the linear: the hidden size
# 6144 (dynamic group-128) and the static workload's 4096 channels
NORM = dict(M_list=(1, 512, 4096), K_list=(6144, 4096), eps=1e-5)
STATIC = dict(M_list=(1, 512, 4096), K=4096, N=14336, parts=(4096, 4096, 6144),
              calib_rows=256)
# grouped (MoE) experts: hidden size H, intermediate size I per expert, E local
# experts (256 routed experts over 8 expert-parallel ranks), T routed rows per
# rank; w13 is [E, 2I, H] (N = 2I, K = H), w2 is [E, H, I] (N = H, K = I)
MOE = dict(E=32, H=7168, I=2048, T=4096, skew=0.5)
