"""Pins for the oracle's quantisers (group-128, MXFP8 [1,32], static, weight blocks).

Independent references used here: the pages' printed byte counts and grid
shapes, closed forms (power-of-two scales, exactly representable groups,
all-zero groups), and a second implementation from numpy binary32 arithmetic
plus PyTorch's float8_e4m3fn cast.
"""
import numpy as np
import pytest
import torch

import oracle
import synthetic_inputs as si

F32_FLOOR = np.float32(1e-10)
F448 = np.float32(448.0)


def _torch_e4m3(v32):
    return torch.from_numpy(np.ascontiguousarray(v32, np.float32)) \
        .to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def _bf16(v):
    return si.f32_to_bf16_bits(np.asarray(v, np.float32))


def _independent_group_quant(x_bits, group):
    """numpy float32 division + torch RNE cast (values never exceed 448 here)."""
    x = si.bf16_bits_to_f32(x_bits)
    M, K = x.shape
    G = -(-K // group)
    q = np.empty((M, K), np.uint8)
    s = np.empty((M, G), np.float32)
    for g in range(G):
        sl = slice(g * group, min(K, (g + 1) * group))
        amax = np.maximum(np.abs(x[:, sl]).max(axis=1), F32_FLOOR)
        sg = (amax / F448).astype(np.float32)
        s[:, g] = sg
        q[:, sl] = _torch_e4m3((x[:, sl] / sg[:, None]).astype(np.float32))
    return q, s


# ------------------------------------------------------------- byte accounting

def test_row_6144_bytes(golden):
    g = golden["row_6144"]
    x = si.activations(2, g["hidden"])
    q, s = oracle.quant_group(x, 128)
    assert s.shape[1] == g["groups"]
    assert q[0].nbytes == g["fp8_bytes"] and s[0].nbytes == g["scale_bytes"]
    assert q[0].nbytes + s[0].nbytes == g["total_bytes"]
    assert x[0].nbytes == g["bf16_bytes"]
    assert round(4 / 128, 3) == golden["scale_overhead_fp32_group128"]["value"]
    d = golden["dispatch_scale_bytes"]
    assert s[0].nbytes == d["fp32_bytes"] and s.shape[1] * 1 == d["ue8m0_bytes"]
    assert round(d["fp32_bytes"] / g["fp8_bytes"], 2) == d["fp32_frac"]
    assert round(d["ue8m0_bytes"] / g["fp8_bytes"], 3) == d["ue8m0_frac"]


# ------------------------------------------------------------- group quant

def test_group_quant_matches_independent_impl():
    x = si.activations(7, 6144)
    q, s = oracle.quant_group(x, 128)
    q2, s2 = _independent_group_quant(x, 128)
    assert np.array_equal(s.view(np.uint32), s2.view(np.uint32))
    assert np.array_equal(q, q2)


def test_group_quant_ragged_tail():
    x = si.activations(5, 208)                # 128 + 80
    q, s = oracle.quant_group(x, 128)
    assert s.shape == (5, 2)
    q2, s2 = _independent_group_quant(x, 128)
    assert np.array_equal(q, q2) and np.array_equal(s, s2)
    xf = si.bf16_bits_to_f32(x)
    assert np.array_equal(s[:, 1], (np.abs(xf[:, 128:]).max(1) / F448).astype(np.float32))


def test_group_max_element_maps_to_448():
    """In every group the element of largest magnitude lands on +-448:
    fl(amax / fl(amax/448)) is within an ulp of 448 and rounds there."""
    x = si.activations(32, 6144)
    q, _ = oracle.quant_group(x, 128)
    xf = si.bf16_bits_to_f32(x).reshape(32, 48, 128)
    qq = q.reshape(32, 48, 128)
    idx = np.abs(xf).argmax(axis=2)
    top = np.take_along_axis(qq, idx[..., None], axis=2)[..., 0]
    assert np.all((top == 0x7E) | (top == 0xFE))
    assert not np.any((q & 0x7F) == 0x7F)             # never NaN


def test_group_power_of_two_scale_closed_form():
    """amax = 448 * 2^k gives s = 2^k exactly; inputs that are E4M3 values
    times 2^k then quantise to exactly those codes."""
    codes = np.arange(0, 0x7F, dtype=np.uint8)
    vals = oracle.e4m3_decode(codes)
    rng = np.random.default_rng(7)
    for k in (-5, 0, 3):
        pick = rng.choice(codes, 127)
        sign = rng.integers(0, 2, 127).astype(np.uint8) << 7
        c = np.concatenate([[0x7E], pick]) | np.concatenate([[0], sign]).astype(np.uint8)
        x = (oracle.e4m3_decode(c) * 2.0 ** k).astype(np.float32)
        xb = _bf16(x)
        assert np.array_equal(si.bf16_bits_to_f32(xb), x)      # exact in bf16
        q, s = oracle.quant_group(xb[None, :], 128)
        assert s[0, 0] == np.float32(2.0 ** k)
        expect = np.where(oracle.e4m3_decode(c) == 0, c & 0x80 | 0, c)
        assert np.array_equal(q[0], expect)
    del vals


def test_group_zero_group():
    x = np.zeros((2, 256), np.uint16)
    x[1, :128] = 0x8000                                   # -0.0
    x[1, 128:] = _bf16(np.linspace(-3, 3, 128))
    q, s = oracle.quant_group(x, 128)
    assert s[0, 0] == s[0, 1] == s[1, 0] == np.float32(F32_FLOOR / F448)
    assert np.all(q[0] == 0) and np.all(q[1, :128] == 0x80)
    assert s[1, 1] == np.float32(np.float32(3.0) / F448)


def test_group_size_is_a_parameter():
    """group = K gives one scale per token (the per-token special case)."""
    x = si.activations(4, 512)
    q, s = oracle.quant_group(x, 512)
    q2, s2 = _independent_group_quant(x, 512)
    assert s.shape == (4, 1) and np.array_equal(q, q2) and np.array_equal(s, s2)


# ------------------------------------------------------------- weight blocks

def test_weight_grid_shapes(golden):
    g = golden["weight_grid_7168x2048"]
    q, s = oracle.quant_weight_block(np.zeros((g["N"], g["K"]), np.uint16))
    assert list(s.shape) == g["grid"] and s.size == g["count"]
    r = golden["weight_grid_ragged_11008"]
    _, s = oracle.quant_weight_block(np.zeros((r["N"], 128), np.uint16))
    assert s.shape[0] == r["blocks"]
    _, s = oracle.quant_weight_block(si.weights(384, 256))
    assert s.shape == (3, 2)
    m = golden["moe_scales"]
    _, s13 = oracle.quant_weight_block(np.zeros((2 * m["I_p"], m["H"]), np.uint16))
    _, s2 = oracle.quant_weight_block(np.zeros((m["H"], m["I_p"]), np.uint16))
    assert list(s13.shape) == m["w13_grid"] and s13.size == m["w13_per_expert"]
    assert list(s2.shape) == m["w2_grid"] and s2.size == m["w2_per_expert"]
    assert s13.size + s2.size == m["per_expert"]
    assert m["experts"] * m["per_expert"] == m["total"]
    assert round(m["total"] * 4 / 1e6, 2) == m["total_mb"]        # decimal MB


def test_weight_block_quant_matches_independent_impl():
    w = si.weights(200, 208)                          # ragged in both dims
    q, s = oracle.quant_weight_block(w)
    wf = si.bf16_bits_to_f32(w)
    assert s.shape == (2, 2)
    for nb in range(2):
        for kb in range(2):
            blk = wf[nb * 128:(nb + 1) * 128, kb * 128:(kb + 1) * 128]
            sb = np.float32(np.maximum(np.abs(blk).max(), F32_FLOOR) / F448)
            assert s[nb, kb] == sb
            qb = q[nb * 128:(nb + 1) * 128, kb * 128:(kb + 1) * 128]
            assert np.array_equal(qb, _torch_e4m3((blk / sb).astype(np.float32)))


# ------------------------------------------------------------- MXFP8

def _independent_mx(x_bits):
    x = si.bf16_bits_to_f32(x_bits)
    M, K = x.shape
    xr = x.reshape(M, K // 32, 32)
    amax = np.maximum(np.abs(xr).max(axis=2), F32_FLOOR)
    r = (amax / F448).astype(np.float32)
    m, e = np.frexp(r.astype(np.float64))               # r = m 2^e, m in [0.5, 1)
    ceil_e = np.where(m == 0.5, e - 1, e)
    u = (ceil_e + 127).astype(np.uint8)
    v = np.ldexp(xr.astype(np.float64), -ceil_e[..., None]).astype(np.float32)
    return _torch_e4m3(v.reshape(M, K)), u


def test_mx_matches_independent_impl(golden):
    assert golden["mxfp8_block"]["value"] == [1, 32]
    x = si.activations(9, 7168)
    q, u = oracle.quant_mx(x)
    q2, u2 = _independent_mx(x)
    assert u.shape == (9, 224)
    assert np.array_equal(u, u2) and np.array_equal(q, q2)


def test_mx_no_overflow_and_power_of_two():
    """Rounding the exponent up keeps every |x| * 2^-e <= 448, and the scale
    is at most a factor 2 above amax/448."""
    x = si.activations(16, 7168)
    _, u = oracle.quant_mx(x)
    xf = np.abs(si.bf16_bits_to_f32(x)).reshape(16, 224, 32).max(axis=2)
    scale = np.ldexp(1.0, u.astype(np.int64) - 127)
    assert np.all(xf / scale <= 448.0)
    assert np.all(xf / scale > 224.0)


@pytest.mark.parametrize("k", [-20, -3, 0, 4, 30])
def test_mx_ceil_rule_closed_form(k):
    # amax = 448 * 2^k exactly -> u = k + 127 and the max element encodes to 448
    row = np.zeros(32, np.float32)
    row[5] = 448.0 * 2.0 ** k
    row[9] = -1.5 * 2.0 ** k
    q, u = oracle.quant_mx(_bf16(row)[None, :])
    assert u[0, 0] == k + 127 and q[0, 5] == 0x7E
    # next BF16 value above: 450 * 2^k -> u = k + 128 and 225 rounds to 224 (0x76)
    row[5] = 450.0 * 2.0 ** k
    q, u = oracle.quant_mx(_bf16(row)[None, :])
    assert u[0, 0] == k + 128 and q[0, 5] == 0x76


def test_mx_zero_group():
    q, u = oracle.quant_mx(np.zeros((1, 64), np.uint16))
    # ceil(log2(fl(1e-10)/448)) = -42
    assert np.all(u == 85) and np.all(q == 0)


# ------------------------------------------------------------- static

def test_static_scale_and_quant():
    calib = si.calibration(256, 4096)
    s = oracle.absmax_scale(calib)
    cf = si.bf16_bits_to_f32(calib)
    assert s == np.float32(np.abs(cf).max() / F448)
    x = si.activations(3, 4096, outliers=False)
    q = oracle.quant_static(x, s)
    xf = si.bf16_bits_to_f32(x)
    t = (xf / s).astype(np.float32)
    assert np.array_equal(q, _torch_e4m3(np.clip(t, -448, 448)))
    # inputs above the calibration range saturate instead of overflowing
    big = _bf16(np.float32([1e3, -1e3, 0.5]) * s * 2)
    qb = oracle.quant_static(big[None, :], s)
    assert list(qb[0][:2]) == [0x7E, 0xFE]


def test_static_weight_partitions():
    w = si.weights(300, 256)
    parts = [100, 72, 128]
    q, sp = oracle.quant_weight_static(w, parts)
    wf = si.bf16_bits_to_f32(w)
    r0 = 0
    for p, n in enumerate(parts):
        blk = wf[r0:r0 + n]
        assert sp[p] == np.float32(np.abs(blk).max() / F448)
        assert np.array_equal(q[r0:r0 + n], _torch_e4m3((blk / sp[p]).astype(np.float32)))
        r0 += n
