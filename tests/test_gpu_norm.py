"""GPU parity of the fused residual add + RMSNorm + quantisation against the CPU
oracle: the residual stream, the BF16 norm output, the E4M3 codes and the group
scales must be bit-identical ("GLM-5.3 推理全链路(十七)", §第1站 RMSNorm 的两个出口)."""
import numpy as np
import pytest
import torch

import block_wise_fp8_gb300 as fb
import oracle
import synthetic_inputs as si
from gpu_util import Guarded, dev

pytestmark = pytest.mark.gpu

EPS = si.NORM["eps"]


def _bits(t):
    return t.detach().cpu().view(torch.int16).numpy().view(np.uint16)


def _u8(t):
    return t.detach().cpu().view(torch.uint8).numpy()


def _inputs(M, K, seed=0):
    x = si.activations(M, K, base_seed=seed)
    res = si.residual_stream(M, K, base_seed=seed)
    g = si.norm_gain(K, base_seed=seed)
    return x, res, g


def _run_group(x, g, res=None, s_layout=fb.SCALE_ROW_MAJOR, in_place=False):
    M, K = x.shape
    dx = dev(x)
    dres = None if res is None else dev(res)
    # every output between canary bands
    g_r = None if in_place else Guarded((M, K), torch.bfloat16)
    r_out = dres if in_place else g_r.t
    g_y = Guarded((M, K), torch.bfloat16)
    g_q = Guarded((M, K), torch.uint8)
    G = (K + 127) // 128
    g_s = Guarded((M, G) if s_layout == fb.SCALE_ROW_MAJOR else (G, (M + 3) // 4 * 4),
                  torch.float32)
    y, q, s = g_y.t, g_q.t, g_s.t
    fb.fp8bq_add_rmsnorm_quant_act(dx, dev(g), EPS, residual=dres, residual_out=r_out, y=y,
                                   q=q, s=s, s_layout=s_layout)
    torch.cuda.synchronize()
    for name, gb in (("residual_out", g_r), ("y", g_y), ("q", g_q), ("s", g_s)):
        if gb is not None:
            gb.check(f"norm {name} {M}x{K}")
    s_h = s.cpu().numpy()
    if s_layout != fb.SCALE_ROW_MAJOR:
        s_h = s_h[:, :M].T
    return _bits(r_out), _bits(y), _u8(q), s_h


@pytest.mark.parametrize("M,K", [(1, 6144), (3, 208), (5, 4096), (130, 6144), (64, 2064),
                                 (7, 16), (9, 16384), (33, 10240)])
def test_group_quant_small_shapes(M, K):
    x, res, g = _inputs(M, K)
    r, y, q, s = _run_group(x, g, res)
    r_ref, y_ref = oracle.add_rmsnorm(x, g, EPS, residual=res)
    q_ref, s_ref = oracle.quant_group(y_ref)
    np.testing.assert_array_equal(r, r_ref)
    np.testing.assert_array_equal(y, y_ref)
    np.testing.assert_array_equal(q, q_ref)
    np.testing.assert_array_equal(s, s_ref)


def test_no_residual_and_col_major_scales():
    x, _, g = _inputs(37, 6144, seed=3)
    r, y, q, s = _run_group(x, g, None, s_layout=fb.SCALE_COL_MAJOR)
    _, y_ref = oracle.add_rmsnorm(x, g, EPS)
    q_ref, s_ref = oracle.quant_group(y_ref)
    np.testing.assert_array_equal(r, x)
    np.testing.assert_array_equal(y, y_ref)
    np.testing.assert_array_equal(q, q_ref)
    np.testing.assert_array_equal(s, s_ref)


def test_in_place_residual():
    x, res, g = _inputs(20, 4096, seed=5)
    r, y, q, _ = _run_group(x, g, res, in_place=True)
    r_ref, y_ref = oracle.add_rmsnorm(x, g, EPS, residual=res)
    np.testing.assert_array_equal(r, r_ref)
    np.testing.assert_array_equal(y, y_ref)


def test_edge_rows():
    """Zero row (eps alone), tiny subnormal row, rows whose sum of squares
    overflows or sits near binary32 rounding ties, a constant row."""
    K = 512
    rng = np.random.default_rng(17)
    x = np.zeros((6, K), np.uint16)
    x[1] = rng.integers(1, 128, K).astype(np.uint16)                       # BF16 subnormals
    x[2] = si.f32_to_bf16_bits(np.full(K, 2.0 ** 70, np.float32))          # S overflows
    x[3, 0] = 0x3F80                                                       # 1 and tiny terms
    x[3, 1:] = si.f32_to_bf16_bits(np.full(K - 1, 2.0 ** -13, np.float32))
    x[4] = si.f32_to_bf16_bits(np.full(K, -3.0, np.float32))               # constant
    x[5] = si.f32_to_bf16_bits((rng.standard_normal(K) * np.exp2(rng.integers(-60, 60, K)))
                               .astype(np.float32))                        # wide exponents
    g = si.norm_gain(K)
    _, y, q, s = _run_group(x, g)
    _, y_ref = oracle.add_rmsnorm(x, g, EPS)
    q_ref, s_ref = oracle.quant_group(y_ref)
    np.testing.assert_array_equal(y, y_ref)
    np.testing.assert_array_equal(q, q_ref)
    np.testing.assert_array_equal(s, s_ref)


def test_sum_of_squares_rounding_against_exact_oracle():
    """Rows built so that the sum of squares needs the sticky bit and the tie
    rule: one large term plus many terms far below it."""
    K = 1024
    rows = []
    for big_e in (0, 5, -20):
        for small_e in (-12, -13, -40, -70):
            r = np.zeros(K, np.float32)
            r[::2] = 2.0 ** big_e
            r[1::2] = 2.0 ** (big_e + small_e)
            rows.append(si.f32_to_bf16_bits(r))
    x = np.stack(rows)
    g = np.full(K, 0x3F80, np.uint16)
    _, y, _, _ = _run_group(x, g)
    _, y_ref = oracle.add_rmsnorm(x, g, EPS)
    np.testing.assert_array_equal(y, y_ref)


def test_norm_only_mode():
    x, res, g = _inputs(11, 6144, seed=9)
    M, K = x.shape
    y = torch.empty(M, K, dtype=torch.bfloat16, device="cuda")
    r_out = torch.empty_like(y)
    fb.fp8bq_add_rmsnorm_quant_act(dev(x), dev(g), EPS, residual=dev(res), residual_out=r_out,
                                   y=y)
    torch.cuda.synchronize()
    r_ref, y_ref = oracle.add_rmsnorm(x, g, EPS, residual=res)
    np.testing.assert_array_equal(_bits(r_out), r_ref)
    np.testing.assert_array_equal(_bits(y), y_ref)


@pytest.mark.parametrize("M", [1, 130, 512])
@pytest.mark.parametrize("s_val", [None, 0.0137, 3.3])
def test_static_quant(M, s_val):
    K = si.STATIC["K"]
    x, res, g = _inputs(M, K, seed=11)
    if s_val is None:  # calibrated on a batch of normalised rows
        _, yc = oracle.add_rmsnorm(*_inputs(64, K, seed=12)[:1], g, EPS)
        s_val = float(oracle.absmax_scale(yc))
    s_x = torch.tensor([s_val], dtype=torch.float32, device="cuda")
    gq = Guarded((M, K), torch.uint8)
    gy = Guarded((M, K), torch.bfloat16)
    gr = Guarded((M, K), torch.bfloat16)
    q, y, r_out = gq.t, gy.t, gr.t
    fb.fp8bq_add_rmsnorm_static_quant_act(dev(x), dev(g), EPS, s_x, q, residual=dev(res),
                                          residual_out=r_out, y=y)
    torch.cuda.synchronize()
    for name, gb in (("q", gq), ("y", gy), ("residual_out", gr)):
        gb.check(f"static norm {name} M={M}")
    r_ref, y_ref = oracle.add_rmsnorm(x, g, EPS, residual=res)
    np.testing.assert_array_equal(_bits(r_out), r_ref)
    np.testing.assert_array_equal(_bits(y), y_ref)
    np.testing.assert_array_equal(_u8(q), oracle.quant_static(y_ref, np.float32(s_val)))


@pytest.mark.parametrize("M,K", [(4096, 6144), (4096, 4096)])
def test_full_size_every_row(M, K):
    """The full-size launch (persistent CTAs over all rows), every output row
    checked bit for bit against the oracle."""
    x, res, g = _inputs(M, K, seed=21)
    r, y, q, s = _run_group(x, g, res)
    r_ref, y_ref = oracle.add_rmsnorm(x, g, EPS, residual=res)
    q_ref, s_ref = oracle.quant_group(y_ref)
    np.testing.assert_array_equal(r, r_ref)
    np.testing.assert_array_equal(y, y_ref)
    np.testing.assert_array_equal(q, q_ref)
    np.testing.assert_array_equal(s, s_ref)


def test_validation():
    x = torch.zeros(4, 64, dtype=torch.bfloat16, device="cuda")
    g = torch.ones(64, dtype=torch.bfloat16, device="cuda")
    q = torch.empty(4, 64, dtype=torch.uint8, device="cuda")
    with pytest.raises(fb.Fp8bqError) as e:
        fb.fp8bq_add_rmsnorm_quant_act(x, g, -1.0, q=q, s=torch.empty(4, 1, device="cuda"))
    assert e.value.name == "FP8BQ_ERR_UNSUPPORTED"
    with pytest.raises(ValueError):
        fb.fp8bq_add_rmsnorm_quant_act(x, g, 1e-5, q=q)             # s missing (binding)
    st = fb._lib.fp8bq_add_rmsnorm_quant_act(                       # s missing (C ABI)
        fb._ptr(x), 64, None, 0, None, fb._ptr(g), 1e-5, 4, 64, None, fb._ptr(q), None, 0,
        fb._stream(None))
    assert st == 1                                                  # FP8BQ_ERR_NULL
    x2 = torch.zeros(4, 40, dtype=torch.bfloat16, device="cuda")    # K % 16 != 0
    with pytest.raises(fb.Fp8bqError) as e:
        fb.fp8bq_add_rmsnorm_quant_act(x2, torch.ones(40, dtype=torch.bfloat16, device="cuda"),
                                       1e-5)
    assert e.value.name == "FP8BQ_ERR_ALIGN"
