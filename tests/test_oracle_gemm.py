"""Pins for the oracle's reference GEMMs (block-scaled, MXFP8, static).

Independent references: the exact integer significand dot product, special
cases that reduce to a library matmul (unit scales; one K block, where the
pages' outer-product form applies; per-partition scales expanded channelwise),
and exact rational arithmetic (fractions) on tiny ragged inputs with distinct
scales per block, so a swapped index or a dropped block shows up.
"""
from fractions import Fraction

import numpy as np
import pytest

import oracle
import synthetic_inputs as si


def _codes(rng, shape, allowed=None):
    if allowed is None:
        c = rng.integers(0, 256, shape).astype(np.uint8)
        c[(c & 0x7F) == 0x7F] = 0x7E                         # no NaN codes
        return c
    return rng.choice(np.asarray(allowed, np.uint8), shape)


def _dec(c):
    return oracle.e4m3_decode(c)


# ------------------------------------------------------------- inner sums

def test_block_inner_sum_is_exact():
    """Products of two E4M3 values carry at most 8 significant bits over
    2^-18 .. 2^17.8, so 128 of them sum exactly in binary64: the oracle's
    binary64 inner sum equals the integer significand dot times 2^-18."""
    rng = np.random.default_rng(10)
    for _ in range(200):
        a = _codes(rng, 128)
        b = _codes(rng, 128)
        assert oracle.e4m3_dot_f64(a, b) == oracle.e4m3_dot_int(a, b) * 2.0 ** -18
    ext = np.array([0x7E, 0xFE, 0x01, 0x81, 0x08], np.uint8)
    a = np.resize(ext, 128)
    b = np.resize(ext[::-1], 128)
    assert oracle.e4m3_dot_f64(a, b) == oracle.e4m3_dot_int(a, b) * 2.0 ** -18


# ------------------------------------------------------------- block-scaled

# codes for 0, +-0.5, +-1, +-2
SMALL = [0x00, 0x30, 0xB0, 0x38, 0xB8, 0x40, 0xC0]


def test_small_codes_decode_as_expected():
    assert list(_dec(np.array(SMALL, np.uint8))) == [0, 0.5, -0.5, 1, -1, 2, -2]


def test_block_gemm_unit_scales_is_integer_matmul():
    rng = np.random.default_rng(11)
    M, N, K = 9, 260, 384
    qa, qw = _codes(rng, (M, K), SMALL), _codes(rng, (N, K), SMALL)
    sa = np.ones((M, 3), np.float32)
    sw = np.ones((3, 3), np.float32)
    y = oracle.gemm_block(qa, sa, qw, sw)
    ia = (_dec(qa) * 2).astype(np.int64)
    iw = (_dec(qw) * 2).astype(np.int64)
    assert np.array_equal(y * 4, (ia @ iw.T).astype(np.float64))


def test_block_gemm_one_k_block_is_outer_product_scaling():
    """With K = 128 the sum has one term: Y = (Qx Qw^T) * (s_x s_w^T), the
    scaled-GEMM form of the pages, with s_w expanded to rows."""
    rng = np.random.default_rng(12)
    M, N, K = 17, 300, 128
    qa, qw = _codes(rng, (M, K)), _codes(rng, (N, K))
    sa = rng.uniform(0.01, 2, (M, 1)).astype(np.float32)
    sw = rng.uniform(0.01, 2, (3, 1)).astype(np.float32)
    y = oracle.gemm_block(qa, sa, qw, sw)
    sw_rows = np.repeat(sw[:, 0], 128)[:N].astype(np.float64)
    ref = (_dec(qa) @ _dec(qw).T) * np.outer(sa[:, 0].astype(np.float64), sw_rows)
    assert np.allclose(y, ref, rtol=1e-12, atol=1e-300)


def _exact_block(qa, sa, qw, sw, bias=None, bn=128, bk=128):
    M, K = qa.shape
    N = qw.shape[0]
    KB = -(-K // bk)
    A = [[Fraction(float(v)) for v in row] for row in _dec(qa)]
    W = [[Fraction(float(v)) for v in row] for row in _dec(qw)]
    out = np.empty((M, N))
    for i in range(M):
        for j in range(N):
            tot = Fraction(0)
            for b in range(KB):
                p = sum(A[i][k] * W[j][k] for k in range(b * bk, min(K, (b + 1) * bk)))
                tot += p * Fraction(float(sa[i, b])) * Fraction(float(sw[j // bn, b]))
            if bias is not None:
                tot += Fraction(float(si.bf16_bits_to_f32(bias[j:j + 1])[0]))
            out[i, j] = float(tot)
    return out


def test_block_gemm_brute_force_exact_rational():
    """Ragged M, N, K; every block gets a different scale (powers of 2 and 3)
    so a transposed grid or a wrong block index changes the answer."""
    rng = np.random.default_rng(13)
    M, N, K = 3, 130, 260                     # 2 N-blocks, 3 K-blocks, ragged tails
    qa, qw = _codes(rng, (M, K)), _codes(rng, (N, K))
    sa = np.array([[2.0 ** i * 3 ** b for b in range(3)] for i in range(M)], np.float32)
    sw = np.array([[3.0 ** -b * 2 ** (5 * n) for b in range(3)] for n in range(2)],
                  np.float32)
    bias = si.f32_to_bf16_bits(rng.standard_normal(N).astype(np.float32))
    y = oracle.gemm_block(qa, sa, qw, sw, bias=bias)
    ref = _exact_block(qa, sa, qw, sw, bias)
    assert np.allclose(y, ref, rtol=1e-13, atol=0)
    # and the transposed scale grid would not pass
    bad = _exact_block(qa, sa, qw, sw[::-1].copy())
    assert not np.allclose(y - si.bf16_bits_to_f32(bias)[None, :], bad, rtol=1e-6)


def test_block_sampled_matches_full_and_threads():
    rng = np.random.default_rng(14)
    x = si.activations(40, 512)
    qa, sa = oracle.quant_group(x)
    qw, sw = oracle.quant_weight_block(si.weights(300, 512))
    y1 = oracle.gemm_block(qa, sa, qw, sw, threads=1)
    y8 = oracle.gemm_block(qa, sa, qw, sw, threads=8)
    assert np.array_equal(y1, y8)
    rows = rng.integers(0, 40, 500)
    cols = rng.integers(0, 300, 500)
    ys = oracle.gemm_block_sampled(qa, sa, qw, sw, rows, cols, threads=4)
    assert np.array_equal(ys, y1[rows, cols])


# ------------------------------------------------------------- MXFP8

def test_mx_gemm_unit_scales_is_matmul():
    rng = np.random.default_rng(15)
    M, N, K = 5, 70, 96
    qa, qw = _codes(rng, (M, K)), _codes(rng, (N, K))
    ua = np.full((M, 3), 127, np.uint8)
    uw = np.full((N, 3), 127, np.uint8)
    y = oracle.gemm_mx(qa, ua, qw, uw)
    assert np.array_equal(y, _dec(qa) @ _dec(qw).T)      # exact: one 96-term sum


def test_mx_gemm_brute_force_exact_rational():
    rng = np.random.default_rng(16)
    M, N, K = 3, 5, 96
    qa, qw = _codes(rng, (M, K)), _codes(rng, (N, K))
    ua = rng.integers(110, 140, (M, 3)).astype(np.uint8)
    uw = rng.integers(110, 140, (N, 3)).astype(np.uint8)
    y = oracle.gemm_mx(qa, ua, qw, uw)
    A, W = _dec(qa), _dec(qw)
    for i in range(M):
        for j in range(N):
            tot = Fraction(0)
            for g in range(3):
                p = sum(Fraction(float(A[i, k])) * Fraction(float(W[j, k]))
                        for k in range(32 * g, 32 * g + 32))
                tot += p * Fraction(2) ** (int(ua[i, g]) - 127) * \
                    Fraction(2) ** (int(uw[j, g]) - 127)
            assert y[i, j] == pytest.approx(float(tot), rel=1e-14, abs=0)


def test_mx_sampled_matches_full():
    x = si.activations(8, 256)
    qa, ua = oracle.quant_mx(x)
    qw, uw = oracle.quant_mx(si.weights(64, 256))
    y = oracle.gemm_mx(qa, ua, qw, uw)
    rows, cols = np.arange(8).repeat(3), np.tile([0, 31, 63], 8)
    assert np.array_equal(oracle.gemm_mx_sampled(qa, ua, qw, uw, rows, cols), y[rows, cols])


# ------------------------------------------------------------- static per-tensor

def test_static_gemm_is_channelwise_scaled_matmul():
    """Per-partition weight scales expand to one scale per output row
    (convert_to_channelwise); then Y = (Qx Qw^T) * s_x * s_w[row]."""
    rng = np.random.default_rng(17)
    x = si.activations(6, 256, outliers=False)
    s_x = oracle.absmax_scale(si.calibration(64, 256))
    qa = oracle.quant_static(x, s_x)
    parts = [48, 16, 64]
    qw, sp = oracle.quant_weight_static(si.weights(128, 256), parts)
    y = oracle.gemm_static(qa, s_x, qw, sp, parts)
    chan = np.repeat(sp.astype(np.float64), parts)
    ref = (_dec(qa) @ _dec(qw).T) * float(s_x) * chan[None, :]
    assert np.allclose(y, ref, rtol=1e-12, atol=0)
    rows = rng.integers(0, 6, 50)
    cols = rng.integers(0, 128, 50)
    assert np.array_equal(oracle.gemm_static_sampled(qa, s_x, qw, sp, parts, rows, cols),
                          y[rows, cols])



def test_mx_and_static_bias_adds_the_decoded_bf16_per_column():
    """A BF16 bias adds its decoded value to every row of its output column, in
    the MX and static GEMMs alike; the sampled forms carry it too."""
    M, N, K = 4, 96, 128
    bias = si.f32_to_bf16_bits(np.linspace(-3, 3, N).astype(np.float32))
    b = si.bf16_bits_to_f32(bias).astype(np.float64)[None, :]
    rows, cols = np.array([0, 3, 1, 2]), np.array([0, 95, 47, 10])
    qa, ua = oracle.quant_mx(si.activations(M, K))
    qw, uw = oracle.quant_mx(si.weights(N, K))
    y0, y1 = oracle.gemm_mx(qa, ua, qw, uw), oracle.gemm_mx(qa, ua, qw, uw, bias=bias)
    np.testing.assert_allclose(y1 - y0, np.broadcast_to(b, (M, N)), rtol=0, atol=1e-12)
    assert np.array_equal(oracle.gemm_mx_sampled(qa, ua, qw, uw, rows, cols, bias=bias),
                          y1[rows, cols])
    s_x = oracle.absmax_scale(si.calibration(32, K))
    qs = oracle.quant_static(si.activations(M, K, outliers=False), s_x)
    parts = [64, 32]
    qws, sp = oracle.quant_weight_static(si.weights(N, K), parts)
    z0 = oracle.gemm_static(qs, s_x, qws, sp, parts)
    z1 = oracle.gemm_static(qs, s_x, qws, sp, parts, bias=bias)
    np.testing.assert_allclose(z1 - z0, np.broadcast_to(b, (M, N)), rtol=0, atol=1e-12)
    assert np.array_equal(oracle.gemm_static_sampled(qs, s_x, qws, sp, parts, rows, cols,
                                                     bias=bias), z1[rows, cols])

def test_sampled_rejects_coordinates_outside_the_output():
    qa, sa = oracle.quant_group(si.activations(3, 128))
    qw, sw = oracle.quant_weight_block(si.weights(130, 128))
    for rows, cols in (([3], [0]), ([0], [130]), ([-1], [0]), ([0, 1], [0])):
        with pytest.raises(ValueError):
            oracle.gemm_block_sampled(qa, sa, qw, sw, np.array(rows), np.array(cols))
