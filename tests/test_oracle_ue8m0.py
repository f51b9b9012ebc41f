"""Pins of the block-FP8-with-UE8M0 oracle ("SGLang 源码完全拆解(十九)",
§分块 GEMM 的后端分派: act_scale_ue8m0 limits the per-token-group scale to a
power of two; §分块路径的后处理: FP32 block
scales requantised to power-of-two UE8M0 for the SM100 runner)."""
import numpy as np
import pytest

import oracle
import synthetic_inputs as si


def test_quant_ue8m0_group32_equals_mx_quantiser():
    """The same rule at group 32 is the MXFP8 quantiser (a separate routine)."""
    x = si.activations(7, 224)
    q, u = oracle.quant_ue8m0(x, group=32)
    q_mx, u_mx = oracle.quant_mx(x)
    np.testing.assert_array_equal(u, u_mx)
    np.testing.assert_array_equal(q, q_mx)


@pytest.mark.parametrize("K", [256, 200, 6144])
def test_quant_ue8m0_tight_power_of_two(K):
    """2^e is the smallest power of two with amax / 2^e <= 448, and every code is
    the E4M3 rounding of the exactly scaled value."""
    x = si.activations(5, K)
    q, u = oracle.quant_ue8m0(x, group=128)
    xf = oracle.bf16_to_f32(x)
    G = -(-K // 128)
    assert u.shape == (5, G)
    for i in range(5):
        for g in range(G):
            blk = xf[i, g * 128:(g + 1) * 128]
            e = int(u[i, g]) - 127
            amax = float(np.abs(blk).max())
            assert amax <= 448.0 * 2.0 ** e
            assert amax > 448.0 * 2.0 ** (e - 1) or amax < 1e-10 * 2
            ref = oracle.e4m3_encode(np.ldexp(blk.astype(np.float64), -e).astype(np.float32))
            np.testing.assert_array_equal(q[i, g * 128:(g + 1) * 128], ref)


def test_requant_identity_for_power_of_two_scales():
    qw, sw = oracle.quant_weight_block(si.weights(256, 384))
    sw_p2 = np.exp2(np.ceil(np.log2(sw.astype(np.float64)))).astype(np.float32)
    q2, u = oracle.requant_weight_ue8m0(qw, sw_p2)
    # codes stay: m = s / s' = 1
    np.testing.assert_array_equal(q2, qw)
    np.testing.assert_array_equal(oracle.ue8m0_to_f32(u), sw_p2)


def test_requant_rule_and_bounds():
    """s' = 2^ceil(log2 s) (from frexp), q' = RNE_sat(dec(q) * s / s'), and the
    requantised values stay within half an E4M3 step of the originals."""
    N, K = 300, 520
    qw, sw = oracle.quant_weight_block(si.weights(N, K))
    q2, u = oracle.requant_weight_ue8m0(qw, sw)
    m, ex = np.frexp(sw.astype(np.float64))
    e = np.where(m == 0.5, ex - 1, ex)
    np.testing.assert_array_equal(u.astype(np.int64), e + 127)
    sp = np.exp2(e.astype(np.float64))
    assert np.all(sp >= sw) and np.all(sp < 2 * sw.astype(np.float64))
    enc = oracle.lib().orc_e4m3_encode
    dq = oracle.e4m3_decode(qw)
    dq2 = oracle.e4m3_decode(q2)
    for nb in range(sw.shape[0]):
        for kb in range(sw.shape[1]):
            rs, cs = slice(nb * 128, (nb + 1) * 128), slice(kb * 128, (kb + 1) * 128)
            ratio = float(sw[nb, kb]) / sp[nb, kb]
            blk = dq[rs, cs]
            ref = np.array([enc(float(v) * ratio) for v in blk.ravel()], np.uint8).reshape(blk.shape)
            np.testing.assert_array_equal(q2[rs, cs], ref)
            # |dec(q') s' - dec(q) s| <= half an E4M3 step of the new code, times s'
            old = blk * float(sw[nb, kb])
            new = dq2[rs, cs] * sp[nb, kb]
            step = np.exp2(np.floor(np.log2(np.maximum(np.abs(dq2[rs, cs]), 2.0 ** -6))) - 3)
            assert np.all(np.abs(new - old) <= 0.5 * step * sp[nb, kb] * (1 + 1e-12))


def test_gemm_block_ue8m0_equals_mx_gemm_on_replicated_scales():
    """A 128-group power-of-two scale is four identical 32-group scales: the block
    definition and the MXFP8 definition (separate routines) agree."""
    M, N, K = 9, 260, 384
    qa, ua = oracle.quant_ue8m0(si.activations(M, K), group=128)
    qw, sw = oracle.quant_weight_block(si.weights(N, K))
    qw2, uw = oracle.requant_weight_ue8m0(qw, sw)
    y = oracle.gemm_block_ue8m0(qa, ua, qw2, uw)
    ua32 = np.repeat(ua, 4, axis=1)
    uw32 = np.repeat(np.repeat(uw, 128, axis=0)[:N], 4, axis=1)
    y_mx = oracle.gemm_mx(qa, ua32, qw2, uw32)
    np.testing.assert_allclose(y, y_mx, rtol=1e-12, atol=1e-12)
