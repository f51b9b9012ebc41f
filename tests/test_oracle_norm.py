"""Pins of the residual-add + RMSNorm oracle against facts fixed outside it:
torch's BF16 addition, exact rational arithmetic (Python fractions), a float64
RMSNorm, and closed forms ("GLM-5.3 推理全链路(十七)", §第1站 RMSNorm 的两个出口:
r = x + residual in BF16, y = r / sqrt(mean(r^2) + eps) * g with the sums and
the root in FP32, BF16 out)."""
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def _bf16_bits(a: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(torch.bfloat16).view(
        torch.int16).numpy().view(np.uint16)


def _bits_to_f64(b: np.ndarray) -> np.ndarray:
    return oracle.bf16_to_f32(b).astype(np.float64)


def _wide_bf16(rng, shape, lo=-30, hi=30) -> np.ndarray:
    """BF16 values with random signs, significands and exponents in [lo, hi]."""
    sig = 1.0 + rng.integers(0, 128, shape) / 128.0
    exp = rng.integers(lo, hi + 1, shape)
    sign = rng.choice([-1.0, 1.0], shape)
    return _bf16_bits((sign * np.ldexp(sig, exp)).astype(np.float32))


# ------------------------------------------------------------------ BF16 rounding

def test_bf16_from_f64_ties_and_overflow():
    one = 0x3F80
    assert oracle.bf16_from_f64(1.0) == one
    assert oracle.bf16_from_f64(1.0 + 2.0 ** -8) == one            # tie -> even (down)
    assert oracle.bf16_from_f64(1.0 + 3 * 2.0 ** -8) == one + 2    # tie -> even (up)
    assert oracle.bf16_from_f64(1.0 + 2.0 ** -8 + 2.0 ** -40) == one + 1
    assert oracle.bf16_from_f64(-0.0) == 0x8000
    big = float(np.ldexp(255.0 / 128.0, 127))                      # largest finite BF16
    assert oracle.bf16_from_f64(big) == 0x7F7F
    assert oracle.bf16_from_f64(big + 2.0 ** 119) == 0x7F80        # halfway -> infinity
    assert oracle.bf16_from_f64(2.0 ** -133) == 0x0001              # smallest subnormal
    assert oracle.bf16_from_f64(2.0 ** -134) == 0x0000              # tie -> even (zero)


def test_bf16_from_f64_matches_torch():
    """Rounding binary32 values to BF16 agrees with torch's conversion."""
    rng = np.random.default_rng(1)
    f = (rng.standard_normal(20000) * np.exp2(rng.integers(-40, 40, 20000))).astype(np.float32)
    ref = _bf16_bits(f)
    got = np.array([oracle.bf16_from_f64(float(v)) for v in f], np.uint16)
    np.testing.assert_array_equal(got, ref)


def test_residual_add_matches_torch_bf16_add():
    rng = np.random.default_rng(2)
    M, d = 16, 256
    x = _wide_bf16(rng, (M, d), -20, 20)
    res = _wide_bf16(rng, (M, d), -20, 20)
    res[0, :8] = x[0, :8] ^ 0x8000                    # exact cancellation -> +0
    r, _ = oracle.add_rmsnorm(x, np.full(d, 0x3F80, np.uint16), 1e-6, residual=res)
    tx = torch.from_numpy(x.view(np.int16)).view(torch.bfloat16)
    tr = torch.from_numpy(res.view(np.int16)).view(torch.bfloat16)
    ref = (tx + tr).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(r, ref)


# ------------------------------------------------------------------ exact sum of squares

def _check_correctly_rounded(bits: np.ndarray, s: np.float32):
    exact = sum((Fraction(float(v)) ** 2 for v in _bits_to_f64(bits)), Fraction(0))
    assert np.isfinite(s)
    here = Fraction(float(s))
    up = Fraction(float(np.nextafter(s, np.float32(np.inf))))
    dn = Fraction(float(np.nextafter(s, np.float32(-np.inf)))) if s > 0 else Fraction(0)
    err = abs(here - exact)
    assert err <= abs(up - exact) and err <= abs(dn - exact), (float(s), float(exact))
    if err == abs(up - exact) or (s > 0 and err == abs(dn - exact)):
        assert int(np.float32(s).view(np.uint32)) % 2 == 0  # a tie goes to the even significand


@pytest.mark.parametrize("lo,hi", [(-3, 3), (-40, 40), (-126, -100), (-133, 60)])
def test_sumsq_is_correctly_rounded(lo, hi):
    rng = np.random.default_rng(300 + hi)
    for trial in range(25):
        d = int(rng.integers(1, 300))
        bits = _wide_bf16(rng, d, max(lo, -126), hi)
        if lo < -126:                                 # some BF16 subnormals
            bits[: d // 3] = rng.integers(1, 128, d // 3).astype(np.uint16)
        _check_correctly_rounded(bits, oracle.sumsq_f32(bits))


def test_sumsq_ties_round_to_even():
    # 1 + 2^-24 is a binary32 tie (the sum is exact): nearest even is 1
    one, tiny = 0x3F80, int(_bf16_bits(np.float32(2.0 ** -12)).ravel()[0])  # tiny^2 = 2^-24
    assert oracle.sumsq_f32(np.array([one, tiny], np.uint16)) == np.float32(1.0)
    # 1 + 2^-24 + 2^-48 is above the tie: rounds up
    tinier = int(_bf16_bits(np.float32(2.0 ** -24)).ravel()[0])
    s = oracle.sumsq_f32(np.array([one, tiny, tinier], np.uint16))
    assert s == np.nextafter(np.float32(1.0), np.float32(2.0))


def test_sumsq_closed_forms_and_specials():
    assert oracle.sumsq_f32(np.full(6144, 0x3F80, np.uint16)) == np.float32(6144.0)
    assert oracle.sumsq_f32(_bf16_bits(np.array([3.0, 4.0], np.float32))) == np.float32(25.0)
    assert oracle.sumsq_f32(np.zeros(7, np.uint16)) == np.float32(0.0)
    big = _bf16_bits(np.array([2.0 ** 100, 2.0 ** 100], np.float32))
    assert np.isinf(oracle.sumsq_f32(big))                       # 2^201 overflows
    assert np.isnan(oracle.sumsq_f32(np.array([0x3F80, 0x7FC0, 0x7F80], np.uint16)))
    assert np.isposinf(oracle.sumsq_f32(np.array([0x3F80, 0xFF80], np.uint16)))


# ------------------------------------------------------------------ RMSNorm

def test_rmsnorm_closed_form_constant_row():
    """A constant row c with g = 1 and eps = 0 normalises to sign(c) exactly."""
    d = 64
    for c in (3.0, -0.375, 96.0):
        x = np.full((1, d), int(_bf16_bits(np.float32(c)).ravel()[0]), np.uint16)
        _, y = oracle.add_rmsnorm(x, np.full(d, 0x3F80, np.uint16), 0.0)
        np.testing.assert_array_equal(oracle.bf16_to_f32(y), np.full((1, d), np.sign(c), np.float32))


def test_rmsnorm_zero_row_with_eps_is_zero():
    d = 128
    x = np.zeros((2, d), np.uint16)
    _, y = oracle.add_rmsnorm(x, np.full(d, 0x4000, np.uint16), 1e-6)
    assert np.all(oracle.bf16_to_f32(y) == 0.0)


@pytest.mark.parametrize("eps", [1e-6, 1e-5, 0.5])
def test_rmsnorm_within_one_bf16_ulp_of_float64(eps):
    """The FP32 steps stay within an ulp of the float64 norm; the BF16 output is
    the float64 value rounded, or its neighbour when that lies near a midpoint."""
    rng = np.random.default_rng(7)
    M, d = 24, 1024
    x = _bf16_bits(rng.standard_normal((M, d)).astype(np.float32) * 3)
    res = _bf16_bits(rng.standard_normal((M, d)).astype(np.float32))
    g = _bf16_bits(rng.uniform(0.25, 4.0, d).astype(np.float32) * rng.choice([-1, 1], d))
    r, y = oracle.add_rmsnorm(x, g, eps, residual=res)
    rf = _bits_to_f64(r)
    y64 = rf / np.sqrt((rf * rf).mean(axis=1, keepdims=True) + np.float64(np.float32(eps)))
    y64 = y64 * _bits_to_f64(g)[None, :]
    got = _bits_to_f64(y)
    ulp = np.exp2(np.floor(np.log2(np.abs(y64))) - 7)
    assert np.all(np.abs(got - y64) <= ulp * 1.01)
    # at least nine in ten land on the nearest BF16 of the float64 value
    nearest = _bits_to_f64(_bf16_bits(y64.astype(np.float32)))
    assert np.mean(got == nearest) > 0.9


def test_rmsnorm_gamma_is_per_channel():
    """Distinct per-channel gains on a constant row: y_k = g_k exactly, so a
    shifted or transposed gain index fails."""
    d = 256
    x = np.full((3, d), 0x4040, np.uint16)                        # 3.0
    g = _bf16_bits(np.linspace(-2.0, 2.0, d).astype(np.float32))
    _, y = oracle.add_rmsnorm(x, g, 0.0)
    for i in range(3):
        np.testing.assert_array_equal(y[i], g)


def test_plain_rmsnorm_without_residual_passes_x_through():
    rng = np.random.default_rng(9)
    x = _bf16_bits(rng.standard_normal((4, 96)).astype(np.float32))
    r, _ = oracle.add_rmsnorm(x, np.full(96, 0x3F80, np.uint16), 1e-6)
    np.testing.assert_array_equal(r, x)


def test_norm_quant_is_the_composition():
    """The fused outputs are the quantisers applied to the BF16 norm output."""
    rng = np.random.default_rng(11)
    x = _bf16_bits(rng.standard_normal((5, 384)).astype(np.float32))
    g = _bf16_bits(rng.uniform(0.5, 2, 384).astype(np.float32))
    r, q, s = oracle.add_rmsnorm_quant_group(x, g, 1e-6)
    _, y = oracle.add_rmsnorm(x, g, 1e-6)
    q2, s2 = oracle.quant_group(y)
    np.testing.assert_array_equal(q, q2)
    np.testing.assert_array_equal(s, s2)
    # group scales follow the normalised rows: |y| <= 448 s per group
    yf = np.abs(oracle.bf16_to_f32(y)).reshape(5, 3, 128).max(axis=2)
    np.testing.assert_array_equal(s, np.maximum(yf, np.float32(1e-10)) / np.float32(448))
