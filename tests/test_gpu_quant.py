"""GPU parity of the quantisation kernels against the CPU oracle: E4M3 codes and
scales must be bit-identical, on the five workloads' shapes, ragged K, both
scale layouts, a row pitch wider than K, and every finite BF16 input."""
import numpy as np
import pytest
import torch

import block_wise_fp8_gb300 as fb
import oracle
import synthetic_inputs as si
from gpu_util import Guarded, dev, host

pytestmark = pytest.mark.gpu


def _gpu_quant_group(x, layout=fb.SCALE_ROW_MAJOR, ldx_pad=0):
    M, K = x.shape
    xd = dev(x)
    if ldx_pad:
        wide = torch.zeros(M, K + ldx_pad, dtype=torch.bfloat16, device="cuda")
        wide[:, :K] = xd
        xd = wide[:, :K]
    G = -(-K // 128)
    q = Guarded((M, K), torch.uint8)
    shape = (M, G) if layout == fb.SCALE_ROW_MAJOR else (G, -(-M // 4) * 4)
    s = Guarded(shape, torch.float32, fill=-1.0)
    fb.fp8bq_quant_act(xd, q.t, s.t, layout)
    torch.cuda.synchronize()
    q.check(f"codes {M}x{K}")
    s.check(f"scales {M}x{K} layout {layout}")
    return host(q.t), host(s.t)


@pytest.mark.parametrize("M,K", [(16, 256), (5, 208), (1, 6144), (8, 6144), (32, 6144),
                                 (64, 6144), (4096, 6144), (2048, 7168), (4096, 4096),
                                 (3, 16), (7, 144)])
def test_quant_group_bit_exact(M, K):
    x = si.activations(M, K)
    q, s = _gpu_quant_group(x)
    qr, sr = oracle.quant_group(x)
    assert np.array_equal(s.view(np.uint32), sr.view(np.uint32))
    assert np.array_equal(q, qr)


def test_quant_group_col_major_and_pitch():
    M, K = 37, 6144
    x = si.activations(M, K)
    q, s = _gpu_quant_group(x, fb.SCALE_COL_MAJOR, ldx_pad=64)
    qr, sr = oracle.quant_group(x)
    assert np.array_equal(q, qr)
    assert np.array_equal(s[:, :M].view(np.uint32), sr.T.view(np.uint32))


def test_quant_group_special_values():
    """zero groups, negative zero, tiny and subnormal BF16 values, exact powers."""
    K = 512
    x = np.zeros((4, K), np.uint16)
    x[1, :128] = 0x8000                                              # -0.0
    x[1, 128:256] = si.f32_to_bf16_bits(np.linspace(-1e-38, 1e-38, 128).astype(np.float32))
    x[2] = si.f32_to_bf16_bits((np.arange(K) - 256).astype(np.float32) * 2.0 ** -20)
    x[3] = np.arange(K, dtype=np.uint16) * 127                        # assorted patterns
    x[3][((x[3] >> 7) & 0xFF) == 0xFF] = 0                            # no inf/nan
    q, s = _gpu_quant_group(x)
    qr, sr = oracle.quant_group(x)
    assert np.array_equal(s.view(np.uint32), sr.view(np.uint32))
    assert np.array_equal(q, qr)


@pytest.mark.parametrize("amax", [3.0, 5.0, 7.0, 100.5, 0.3, 1e-30, 2.5e36])
def test_quant_group_every_bf16_below_amax(amax):
    """Every group has max |x| = amax (so the same non-power-of-two scale) and the
    other 127 slots sweep every BF16 value of smaller magnitude, both signs: all
    reachable quotients x / s, including those next to E4M3 rounding ties, must
    give the codes of an IEEE binary32 division."""
    a_bits = si.f32_to_bf16_bits(np.float32([amax]))[0]
    a = si.bf16_bits_to_f32(np.array([a_bits]))[0]
    pats = np.arange(1 << 15, dtype=np.uint32).astype(np.uint16)     # positive patterns
    vals = si.bf16_bits_to_f32(pats)
    pats = pats[np.isfinite(vals) & (vals <= a)]
    pats = np.concatenate([pats, pats | 0x8000])
    n_groups = -(-len(pats) // 127)
    body = np.zeros(n_groups * 127, np.uint16)
    body[:len(pats)] = pats
    x = np.empty((n_groups, 128), np.uint16)
    x[:, 0] = a_bits
    x[:, 1:] = body.reshape(n_groups, 127)
    x = x.reshape(-1, 1024) if n_groups % 8 == 0 else x
    q, s = _gpu_quant_group(x)
    qr, sr = oracle.quant_group(x)
    assert np.array_equal(s.view(np.uint32), sr.view(np.uint32))
    assert np.array_equal(q, qr)


@pytest.mark.parametrize("scale", [1.0, 0.0137, 3.3])
def test_static_quant_every_finite_bf16_value(scale):
    """q = RNE_sat(x / s) for all 2^16 BF16 patterns except Inf/NaN.  With s = 1 this
    checks the hardware conversion (saturation, subnormals, ties, signed zero)
    against the oracle's encoder exhaustively over BF16 inputs; the other scales
    check every quotient the division can produce."""
    pats = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    pats = pats[((pats >> 7) & 0xFF) != 0xFF]
    pats = np.concatenate([pats, np.zeros((-len(pats)) % 16, np.uint16)])
    x = pats.reshape(-1, 16 * 64) if len(pats) % (16 * 64) == 0 else pats.reshape(-1, 16)
    sx = torch.full((1,), scale, dtype=torch.float32, device="cuda")
    q = Guarded(x.shape, torch.uint8)
    fb.fp8bq_static_quant_act(dev(x), sx, q.t)
    torch.cuda.synchronize()
    q.check("static codes")
    assert np.array_equal(host(q.t), oracle.quant_static(x, np.float32(scale)))


@pytest.mark.parametrize("M,K", [(2048, 7168), (5, 96), (64, 7168), (1, 32)])
def test_quant_mx_bit_exact(M, K):
    x = si.activations(M, K)
    q = Guarded((M, K), torch.uint8)
    s = Guarded((M, K // 32), torch.uint8)
    fb.fp8bq_mx_quant_act(dev(x), q.t, s.t)
    torch.cuda.synchronize()
    q.check("mx codes")
    s.check("mx scale codes")
    qr, ur = oracle.quant_mx(x)
    assert np.array_equal(host(s.t), ur)
    assert np.array_equal(host(q.t), qr)


def test_quant_mx_special_groups():
    row = np.zeros((3, 64), np.float32)
    row[1, 5] = 448.0 * 2.0 ** -7
    row[1, 40] = 450.0 * 2.0 ** 9
    row[2] = np.linspace(-3e-39, 3e-39, 64)
    x = si.f32_to_bf16_bits(row)
    q = torch.empty(3, 64, dtype=torch.uint8, device="cuda")
    s = torch.empty(3, 2, dtype=torch.uint8, device="cuda")
    fb.fp8bq_mx_quant_act(dev(x), q, s)
    torch.cuda.synchronize()
    qr, ur = oracle.quant_mx(x)
    assert np.array_equal(host(s), ur) and np.array_equal(host(q), qr)


@pytest.mark.parametrize("M", [1, 512, 4096])
def test_static_scale_and_quant_bit_exact(M):
    K = 4096
    calib = si.calibration(256, K)
    s_gpu = torch.empty(1, dtype=torch.float32, device="cuda")
    fb.fp8bq_absmax_scale(dev(calib), s_gpu)
    s_ref = oracle.absmax_scale(calib)
    torch.cuda.synchronize()
    assert host(s_gpu).view(np.uint32)[0] == np.float32(s_ref).view(np.uint32)
    x = si.activations(M, K)              # outlier channels exceed the calibration range
    q = torch.empty(M, K, dtype=torch.uint8, device="cuda")
    fb.fp8bq_static_quant_act(dev(x), s_gpu, q)
    torch.cuda.synchronize()
    qr = oracle.quant_static(x, s_ref)
    assert np.array_equal(host(q), qr)
    if M > 1:
        assert np.any(qr == 0x7E)          # saturation is exercised


@pytest.mark.parametrize("N,K", [(384, 256), (200, 208), (6144, 6144), (130, 16)])
def test_weight_block_quant_bit_exact(N, K):
    w = si.weights(N, K)
    q = Guarded((N, K), torch.uint8)
    s = Guarded((-(-N // 128), -(-K // 128)), torch.float32)
    fb.fp8bq_quant_weight_block(dev(w), q.t, s.t)
    torch.cuda.synchronize()
    q.check("weight codes")
    s.check("weight block scales")
    qr, sr = oracle.quant_weight_block(w)
    assert np.array_equal(host(s.t).view(np.uint32), sr.view(np.uint32))
    assert np.array_equal(host(q.t), qr)


def test_weight_partition_scales_bit_exact():
    w = si.weights(14336, 4096)
    parts = [4096, 4096, 6144]
    qr, spr = oracle.quant_weight_static(w, parts)
    wd = dev(w)
    sp = torch.empty(3, dtype=torch.float32, device="cuda")
    q = torch.empty(14336, 4096, dtype=torch.uint8, device="cuda")
    r0 = 0
    for p, n in enumerate(parts):
        fb.fp8bq_absmax_scale(wd[r0:r0 + n], sp[p:p + 1])
        fb.fp8bq_static_quant_act(wd[r0:r0 + n], sp[p:p + 1], q[r0:r0 + n])
        r0 += n
    torch.cuda.synchronize()
    assert np.array_equal(host(sp).view(np.uint32), spr.view(np.uint32))
    assert np.array_equal(host(q), qr)


def test_empty_batch_is_a_no_op():
    x = torch.empty(0, 256, dtype=torch.bfloat16, device="cuda")
    q = torch.empty(0, 256, dtype=torch.uint8, device="cuda")
    s = torch.empty(0, 2, dtype=torch.float32, device="cuda")
    fb.fp8bq_quant_act(x, q, s)
    fb.fp8bq_mx_quant_act(x, q, s.view(torch.uint8))
