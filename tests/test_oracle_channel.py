"""Pins of the channelwise (per-token activation x per-channel weight) oracle
("SGLang 源码完全拆解(十九)", §一条 GEMM 的三种缩放组合: for per-token +
per-channel the output scale is the M x N outer product s_x[i] * s_w[j];
§装载后的三个分支: the weight scale is the group rule with group = K)."""
import numpy as np
import pytest

import oracle
import synthetic_inputs as si


def _codes(rng, shape):
    c = rng.integers(0, 0x7F, shape).astype(np.uint8)       # no NaN codes
    c |= (rng.integers(0, 2, shape).astype(np.uint8) << 7)
    c[c == 0xFF] = 0xFE
    c[c == 0x7F] = 0x7E
    return c


@pytest.mark.parametrize("M,N,K", [(3, 5, 40), (7, 2, 257), (1, 9, 1024)])
def test_gemm_channel_equals_decoded_matmul(M, N, K):
    """Exact: E4M3 products have at most 8 significant bits and span 2^-18..2^18,
    so the float64 sums are exact in any order; the two scale products are
    rounded in the same order on both sides."""
    rng = np.random.default_rng(M * 100 + N)
    qa, qw = _codes(rng, (M, K)), _codes(rng, (N, K))
    sa = np.exp2(rng.integers(-8, 8, M)).astype(np.float32) * rng.uniform(0.5, 1, M).astype(np.float32)
    sw = np.exp2(rng.integers(-8, 8, N)).astype(np.float32) * rng.uniform(0.5, 1, N).astype(np.float32)
    ref = oracle.e4m3_decode(qa) @ oracle.e4m3_decode(qw).T
    ref = ref * sa.astype(np.float64)[:, None] * sw.astype(np.float64)[None, :]
    np.testing.assert_array_equal(oracle.gemm_channel(qa, sa, qw, sw), ref)


def test_gemm_channel_scales_are_not_transposed():
    """Row i carries sa[i], column j sw[j]: distinct powers of two per row and
    column locate each factor."""
    M, N, K = 4, 6, 64
    rng = np.random.default_rng(3)
    qa, qw = _codes(rng, (M, K)), _codes(rng, (N, K))
    one_a, one_w = np.ones(M, np.float32), np.ones(N, np.float32)
    base = oracle.gemm_channel(qa, one_a, qw, one_w)
    sa = np.exp2(np.arange(M)).astype(np.float32)
    sw = np.exp2(-np.arange(N) * 3.0).astype(np.float32)
    got = oracle.gemm_channel(qa, sa, qw, sw)
    np.testing.assert_array_equal(got, base * np.exp2(np.arange(M))[:, None]
                                  * np.exp2(-np.arange(N) * 3.0)[None, :])


def test_gemm_channel_reduces_to_per_partition_with_one_row_partitions():
    """A constant activation scale and one-row partitions give the static form."""
    M, N, K = 5, 7, 96
    rng = np.random.default_rng(4)
    qa, qw = _codes(rng, (M, K)), _codes(rng, (N, K))
    sw = rng.uniform(0.001, 0.01, N).astype(np.float32)
    c = np.float32(0.0371)
    got = oracle.gemm_channel(qa, np.full(M, c, np.float32), qw, sw)
    ref = oracle.gemm_static(qa, c, qw, sw, np.ones(N, np.int64))
    np.testing.assert_array_equal(got, ref)


def test_gemm_channel_bias_and_sampled():
    M, N, K = 6, 10, 128
    rng = np.random.default_rng(5)
    qa, qw = _codes(rng, (M, K)), _codes(rng, (N, K))
    sa = rng.uniform(0.01, 0.1, M).astype(np.float32)
    sw = rng.uniform(0.001, 0.01, N).astype(np.float32)
    bias = si.f32_to_bf16_bits(np.linspace(-1, 1, N).astype(np.float32))
    full = oracle.gemm_channel(qa, sa, qw, sw, bias=bias)
    nob = oracle.gemm_channel(qa, sa, qw, sw)
    np.testing.assert_allclose(full - nob, np.broadcast_to(
        oracle.bf16_to_f32(bias).astype(np.float64)[None, :], (M, N)), rtol=0, atol=1e-12)
    rows = np.array([0, 5, 3, 2], np.int64)
    cols = np.array([9, 0, 4, 4], np.int64)
    np.testing.assert_array_equal(oracle.gemm_channel_sampled(qa, sa, qw, sw, rows, cols, bias=bias),
                                  full[rows, cols])


def test_quant_channel_is_one_scale_per_row():
    """s_i = max|x_i| / 448 (binary32 division) and q = RNE_sat(x / s_i)."""
    x = si.activations(9, 320)
    q, s = oracle.quant_channel(x)
    xf = oracle.bf16_to_f32(x)
    amax = np.maximum(np.abs(xf).max(axis=1), np.float32(1e-10)).astype(np.float32)
    s_ref = (amax / np.float32(448.0)).astype(np.float32)
    np.testing.assert_array_equal(s, s_ref)
    np.testing.assert_array_equal(q, oracle.e4m3_encode((xf / s_ref[:, None]).astype(np.float32)))
    # the largest magnitude of every row maps to +-448 (code 0x7E)
    assert np.all((q & 0x7F).max(axis=1) == 0x7E)
