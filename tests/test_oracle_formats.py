"""Pins for the oracle's number formats (E4M3, UE8M0, BF16) and the input generator.

Each check compares the oracle with something that is not the oracle: numbers
printed on the pages (tests/golden), PyTorch's own float8_e4m3fn / bfloat16
conversions (library routines), or a brute-force nearest-value search.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import synthetic_inputs as si


def _all_codes():
    return np.arange(256, dtype=np.uint8)


def _finite_codes():
    c = _all_codes()
    return c[(c & 0x7F) != 0x7F]


def _torch_decode(codes):
    return torch.from_numpy(np.asarray(codes, np.uint8)).view(torch.float8_e4m3fn) \
        .to(torch.float32).numpy().astype(np.float64)


def _torch_encode(v):
    return torch.from_numpy(np.asarray(v, np.float32)).to(torch.float8_e4m3fn) \
        .view(torch.uint8).numpy()


# ---------------------------------------------------------------- E4M3 decode

def test_e4m3_page_constants(golden):
    d = oracle.e4m3_decode(_all_codes())
    assert d[0x7E] == golden["e4m3_max"]["value"]
    assert d[0xFE] == -golden["e4m3_max"]["value"]
    assert np.nanmax(np.abs(d)) == golden["e4m3_max"]["value"]
    assert d[0x08] == 2.0 ** golden["e4m3_min_normal_log2"]["value"]
    # the smallest normal is the smallest code with a non-zero exponent field
    assert d[0x07] < d[0x08] and d[0x07] == 7 * 2.0 ** -9
    assert d[0x01] == 2.0 ** -9
    assert np.isnan(d[0x7F]) and np.isnan(d[0xFF])
    assert np.count_nonzero(np.isfinite(d)) == 254
    assert d[0x00] == 0.0 and not math.copysign(1.0, d[0x00]) < 0
    assert d[0x80] == 0.0 and math.copysign(1.0, d[0x80]) < 0


def test_e4m3_decode_monotone_and_symmetric():
    d = oracle.e4m3_decode(_all_codes())
    pos = d[0x00:0x7F]
    assert np.all(np.diff(pos) > 0)
    assert np.array_equal(d[0x80:0xFF], -pos)


def test_e4m3_decode_matches_torch():
    c = _finite_codes()
    assert np.array_equal(oracle.e4m3_decode(c), _torch_decode(c))


def test_e4m3_sig_is_value_times_2_pow_9():
    c = _finite_codes()
    sig = np.array([oracle.e4m3_sig(int(x)) for x in c], np.float64)
    assert np.array_equal(sig, oracle.e4m3_decode(c) * 512.0)


# ---------------------------------------------------------------- E4M3 encode

def _probe_values(rng):
    pos = oracle.e4m3_decode(np.arange(0, 0x7F, dtype=np.uint8))   # 0 .. 448
    mids = (pos[:-1] + pos[1:]) / 2                                 # every tie
    mids32 = mids.astype(np.float32)
    assert np.array_equal(mids32.astype(np.float64), mids)          # ties are exact in fp32
    up = np.nextafter(mids32, np.float32(np.inf))
    dn = np.nextafter(mids32, np.float32(0))
    logu = np.exp2(rng.uniform(-14, math.log2(448.0), 200000)).astype(np.float32)
    lin = rng.uniform(0, 448, 100000).astype(np.float32)
    v = np.concatenate([pos.astype(np.float32), mids32, up, dn, logu, lin])
    v = v[v <= 448]
    return np.concatenate([v, -v])


def test_e4m3_encode_matches_torch_in_range():
    """PyTorch's float8_e4m3fn cast rounds to nearest even; inside +-448 it
    must agree with the oracle code for code (incl. every tie and its
    neighbours, and the sign of zero)."""
    v = _probe_values(np.random.default_rng(1))
    assert np.array_equal(oracle.e4m3_encode(v), _torch_encode(v))


def test_e4m3_encode_brute_force_nearest():
    """Nearest of the 254 finite codes by exhaustive search, ties to the code
    with an even mantissa, saturating beyond 448."""
    rng = np.random.default_rng(2)
    v = _probe_values(rng)[::7]
    v = np.concatenate([v, np.float32([460.0, 464.0, 500.0, 1e6, 3e38, -470.0, -1e30])])
    codes = np.arange(0, 0x7F, dtype=np.uint8)
    vals = oracle.e4m3_decode(codes)
    a = np.minimum(np.abs(v.astype(np.float64)), 448.0)   # clamp(., -448, 448)
    dist = np.abs(a[:, None] - vals[None, :])
    best = dist.min(axis=1, keepdims=True)
    cand = dist == best
    # among equally near codes take the one with an even mantissa field
    even = (codes[None, :] & 1) == 0
    pick_even = cand & even
    idx = np.where(pick_even.any(axis=1), pick_even.argmax(axis=1), cand.argmax(axis=1))
    expect = codes[idx] | np.where(np.signbit(v), 0x80, 0).astype(np.uint8)
    assert np.array_equal(oracle.e4m3_encode(v), expect)


def test_e4m3_saturation_and_nan():
    v = np.float32([448.0, 449.0, 463.9, 464.0, 1e10, np.finfo(np.float32).max])
    assert np.all(oracle.e4m3_encode(v) == 0x7E)
    assert np.all(oracle.e4m3_encode(-v) == 0xFE)
    assert oracle.e4m3_encode(np.float32([np.nan]))[0] == 0x7F


def test_e4m3_round_trip():
    c = _finite_codes()
    d = oracle.e4m3_decode(c).astype(np.float32)
    assert np.array_equal(oracle.e4m3_encode(d), c)


def test_e4m3_error_bound(golden):
    """Relative rounding error at most 2^-4 in the normal range (the pages'
    bound); at most half the subnormal step 2^-10 below 2^-6."""
    rng = np.random.default_rng(3)
    v = np.exp2(rng.uniform(-6, math.log2(448.0), 400000)).astype(np.float32)
    err = np.abs(oracle.e4m3_decode(oracle.e4m3_encode(v)) - v) / v
    bound = golden["e4m3_max_rel_rounding_error"]["value"]
    assert err.max() <= bound
    assert err.max() > 0.9 * (1 / 17)         # sup is 1/17 at 2^e * 17/16
    s = rng.uniform(0, 2 ** -6, 100000).astype(np.float32)
    assert np.abs(oracle.e4m3_decode(oracle.e4m3_encode(s)) - s).max() <= 2 ** -10


def test_e4m3_rms_error_uniform_binade(golden):
    """Uniform values in one binade [2^e, 2^(e+1)): the rounding error is
    uniform on +-2^(e-4), so its RMS is 2^(e-4)/sqrt(3), which is the pages'
    2^-5/sqrt(3) relative to the top of the binade."""
    rng = np.random.default_rng(4)
    for e in (-3, 0, 5):
        v = rng.uniform(2.0 ** e, 2.0 ** (e + 1), 400000).astype(np.float32)
        err = oracle.e4m3_decode(oracle.e4m3_encode(v)) - v
        rms = math.sqrt(np.mean(err ** 2)) / 2.0 ** (e + 1)
        assert abs(rms / golden["e4m3_rms_rel_error_uniform"]["value"] - 1) < 0.01


# ---------------------------------------------------------------- UE8M0 / BF16

def test_ue8m0_decode(golden):
    u = np.arange(255, dtype=np.uint8)
    d = oracle.ue8m0_decode(u)
    assert np.array_equal(d, np.ldexp(1.0, u.astype(np.int64) - 127))
    assert d[0] == 2.0 ** golden["ue8m0_range_log2"]["min"]
    assert d[254] == 2.0 ** golden["ue8m0_range_log2"]["max"]
    assert np.isnan(oracle.ue8m0_decode(np.uint8([255]))[0])


def test_bf16_decode_matches_torch():
    b = np.random.default_rng(5).integers(0, 1 << 16, 50000).astype(np.uint16)
    b = b[((b >> 7) & 0xFF) != 0xFF]                 # finite patterns only
    t = torch.from_numpy(b.view(np.int16)).view(torch.bfloat16).to(torch.float32).numpy()
    assert np.array_equal(oracle.bf16_to_f32(b), t)
    assert all(oracle.lib().orc_bf16_to_f32(int(x)) == float(y) for x, y in zip(b[:100], t[:100]))


# ---------------------------------------------------------------- input generator

def test_splitmix64_reference_vector():
    # splitmix64 seeded with 0: first outputs of the published generator
    z = si.splitmix64(0, 0, 2)
    assert int(z[0]) == 0xE220A8397B1DCDAF
    assert int(z[1]) == 0x6E789E6AA1B965F4


def test_generator_bf16_rounding_matches_torch():
    v = np.random.default_rng(6).standard_normal(100000).astype(np.float32) * 7
    t = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(si.f32_to_bf16_bits(v), t)


def test_generator_distributions():
    x = si.bf16_bits_to_f32(si.activations(64, 6144, outliers=False))
    assert abs(x.mean()) < 0.01 and abs(x.std() - 1) < 0.01
    w = si.bf16_bits_to_f32(si.weights(256, 1024))
    assert abs(w.std() / 0.02 - 1) < 0.01
    oc = si.outlier_channels(6144)
    assert len(oc) == 61 and len(np.unique(oc)) == 61
    assert len(si.outlier_channels(7168)) == 72
    xo = si.bf16_bits_to_f32(si.activations(64, 6144))
    ratio = xo[:, oc].std() / np.delete(xo, oc, axis=1).std()
    assert 45 < ratio < 55
    # a row slice of a stream equals the same rows of the full matrix
    assert np.array_equal(si.normal_bf16(3, 100, 1.0, 0, row_start=5),
                          si.normal_bf16(8, 100, 1.0, 0)[5:])


@pytest.mark.parametrize("threads", [1, 3])
def test_generator_thread_invariance(threads):
    a = si.normal_bf16(300, 1000, 0.02, 1, chunk_elems=20000, threads=threads)
    b = si.normal_bf16(300, 1000, 0.02, 1, chunk_elems=1 << 22, threads=1)
    assert np.array_equal(a, b)


def test_encode_bits_range_is_the_encoder_on_each_pattern():
    """The range encoder used by the exhaustive GPU sweep is the pinned
    encoder applied to consecutive binary32 bit patterns: around the subnormal
    and normal boundaries, the saturation threshold, infinities and NaNs, and
    at the ends of the 32-bit range; the thread count does not matter."""
    for first, n in ((0, 4096), (0x3A7F_F000, 8192), (0x43DF_F000, 8192),
                     (0x7F7F_FF00, 0x200), (0xFF7F_FF00, 0x100), ((1 << 32) - 300, 300)):
        bits = (np.uint64(first) + np.arange(n, dtype=np.uint64)).astype(np.uint32)
        ref = oracle.e4m3_encode(bits.view(np.float32))
        for threads in (1, 3):
            assert np.array_equal(oracle.e4m3_encode_bits_range(first, n, threads=threads), ref)
    with pytest.raises(ValueError):
        oracle.e4m3_encode_bits_range((1 << 32) - 2, 3)
