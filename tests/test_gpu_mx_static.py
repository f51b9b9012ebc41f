"""GPU parity of the MXFP8 ([1,32], UE8M0) and static per-tensor GEMMs and
linears against the CPU oracle (binary64 on the same quantised inputs)."""
import numpy as np
import pytest
import torch

import block_wise_fp8_gb300 as fb
import oracle
import synthetic_inputs as si
from gpu_util import Guarded, assert_covers_every_block, check_close, dev, host, sample_indices

pytestmark = pytest.mark.gpu


# ------------------------------------------------------------------ MXFP8

def _mx_gemm(qa, ua, qw, uw, bias=None):
    M, K = qa.shape
    N = qw.shape[0]
    y = Guarded((M, N), torch.bfloat16, fill=float("nan"))
    ws = Guarded((fb.fp8bq_workspace_bytes(fb.OP_MX_GEMM, M, N, K),), torch.uint8)
    fb.fp8bq_workspace_init(ws.t)
    fb.fp8bq_mx_gemm(dev(qa), dev(ua), dev(qw), dev(uw), y.t, ws.t,
                     bias=None if bias is None else dev(bias))
    assert fb.fp8bq_poll_status(ws.t) == 0
    y.check(f"mx y {M}x{N}x{K}")
    ws.check(f"mx workspace {M}x{N}x{K}")
    return host(y.t)


def test_mx_gemm_unit_scales():
    """All scale codes 127 (factor 1): the block-scaled MMA is a plain FP8 GEMM."""
    rng = np.random.default_rng(5)
    M, N, K = 128, 128, 128
    qa = rng.integers(0, 0x7E, (M, K)).astype(np.uint8)
    qw = rng.integers(0, 0x7E, (N, K)).astype(np.uint8)
    ua = np.full((M, K // 32), 127, np.uint8)
    uw = np.full((N, K // 32), 127, np.uint8)
    check_close(_mx_gemm(qa, ua, qw, uw), oracle.gemm_mx(qa, ua, qw, uw), "mx unit scales")


def test_mx_gemm_scale_layout():
    """Distinct power-of-two scales per row and per 32-group on each side locate
    every scale factor: a wrong row, group or operand assignment fails."""
    rng = np.random.default_rng(6)
    M, N, K = 256, 256, 256
    qa = rng.integers(0, 0x7E, (M, K)).astype(np.uint8)
    qw = rng.integers(0, 0x7E, (N, K)).astype(np.uint8)
    ua = (120 + (np.arange(M)[:, None] * 3 + np.arange(K // 32)[None, :]) % 15).astype(np.uint8)
    uw = (118 + (np.arange(N)[:, None] * 5 + 2 * np.arange(K // 32)[None, :]) % 17).astype(np.uint8)
    check_close(_mx_gemm(qa, ua, qw, uw), oracle.gemm_mx(qa, ua, qw, uw), "mx scale layout")


@pytest.mark.parametrize("M,N,K", [(16, 384, 256), (5, 200, 96), (130, 136, 224),
                                   (257, 232, 128), (300, 520, 416), (512, 1024, 7168)])
def test_mx_gemm_shapes(M, N, K):
    qa, ua = oracle.quant_mx(si.activations(M, K))
    qw, uw = oracle.quant_mx(si.weights(N, K))
    check_close(_mx_gemm(qa, ua, qw, uw), oracle.gemm_mx(qa, ua, qw, uw), f"mx {M}x{N}x{K}")


def test_mx_gemm_workload_sampled():
    M, N, K = si.MXFP8["M"], si.MXFP8["N"], si.MXFP8["K"]
    qa, ua = oracle.quant_mx(si.activations(M, K))
    qw, uw = oracle.quant_mx(si.weights(N, K))
    y = _mx_gemm(qa, ua, qw, uw)
    rows, cols = sample_indices(M, N)
    assert_covers_every_block(rows, cols, M, N)
    check_close(y[rows, cols], oracle.gemm_mx_sampled(qa, ua, qw, uw, rows, cols),
                "mx 2048x4096x7168")
    assert np.all(np.isfinite(y))


def test_mx_linear_and_bias():
    M, N, K = 72, 256, 512
    x = si.activations(M, K)
    qw, uw = oracle.quant_mx(si.weights(N, K))
    bias = si.f32_to_bf16_bits(np.linspace(-2, 2, N).astype(np.float32))
    y = Guarded((M, N), torch.bfloat16)
    ws = Guarded((fb.fp8bq_workspace_bytes(fb.OP_MX_LINEAR, M, N, K),), torch.uint8)
    fb.fp8bq_workspace_init(ws.t)
    fb.fp8bq_mx_linear(dev(x), dev(qw), dev(uw), y.t, ws.t, bias=dev(bias))
    assert fb.fp8bq_poll_status(ws.t) == 0
    y.check("mx linear y")
    ws.check("mx linear workspace")
    qa, ua = oracle.quant_mx(x)
    check_close(host(y.t), oracle.gemm_mx(qa, ua, qw, uw, bias=bias), "mx linear")


# ------------------------------------------------------------------ static per-tensor

PARTS = list(si.STATIC["parts"])


@pytest.fixture(scope="module")
def static_weights():
    K, N = si.STATIC["K"], si.STATIC["N"]
    qw, sp = oracle.quant_weight_static(si.weights(N, K), PARTS)
    s_x = oracle.absmax_scale(si.calibration(si.STATIC["calib_rows"], K))
    return qw, sp, s_x


def _static_gemm(qa, s_x, qw, sp, parts, bias=None):
    M, K = qa.shape
    N = qw.shape[0]
    y = Guarded((M, N), torch.bfloat16, fill=float("nan"))
    ws = Guarded((fb.fp8bq_workspace_bytes(fb.OP_STATIC_GEMM, M, N, K),), torch.uint8)
    fb.fp8bq_workspace_init(ws.t)
    sxd = torch.tensor([s_x], dtype=torch.float32, device="cuda")
    fb.fp8bq_static_gemm(dev(qa), sxd, dev(qw), dev(sp), parts, y.t, ws.t,
                         bias=None if bias is None else dev(bias))
    assert fb.fp8bq_poll_status(ws.t) == 0
    y.check(f"static y {M}x{N}x{K}")
    ws.check(f"static workspace {M}x{N}x{K}")
    return host(y.t)


@pytest.mark.parametrize("M", [1, 512, 4096])
def test_static_gemm_workload(static_weights, M):
    qw, sp, s_x = static_weights
    K, N = si.STATIC["K"], si.STATIC["N"]
    qa = oracle.quant_static(si.activations(M, K, outliers=False), s_x)
    y = _static_gemm(qa, s_x, qw, sp, PARTS)
    if M == 1:
        check_close(y, oracle.gemm_static(qa, s_x, qw, sp, PARTS), "static M=1")
    else:
        rows, cols = sample_indices(M, N)
        assert_covers_every_block(rows, cols, M, N)
        # columns on both sides of each partition boundary
        edge = np.array([4095, 4096, 8191, 8192, 14335], np.int64)
        rows = np.concatenate([rows, np.zeros(5, np.int64), np.full(5, M - 1)])
        cols = np.concatenate([cols, edge, edge])
        check_close(y[rows, cols], oracle.gemm_static_sampled(qa, s_x, qw, sp, PARTS, rows,
                                                              cols), f"static M={M}")


@pytest.mark.parametrize("M,N,K,parts", [(3, 200, 208, [72, 128]), (150, 384, 256, [100, 284]),
                                         (64, 256, 4096, [256]), (5, 9728, 768, [4864, 4864])])
def test_static_gemm_small(M, N, K, parts):
    qw, sp = oracle.quant_weight_static(si.weights(N, K), parts)
    s_x = oracle.absmax_scale(si.calibration(32, K))
    qa = oracle.quant_static(si.activations(M, K), s_x)
    bias = si.f32_to_bf16_bits(np.linspace(-1, 1, N).astype(np.float32))
    y = _static_gemm(qa, s_x, qw, sp, parts, bias=bias)
    check_close(y, oracle.gemm_static(qa, s_x, qw, sp, parts, bias=bias), f"static {M}x{N}x{K}")


def test_static_linear(static_weights):
    qw, sp, s_x = static_weights
    M, K, N = 33, si.STATIC["K"], si.STATIC["N"]
    x = si.activations(M, K)
    y = Guarded((M, N), torch.bfloat16)
    ws = Guarded((fb.fp8bq_workspace_bytes(fb.OP_STATIC_LINEAR, M, N, K),), torch.uint8)
    fb.fp8bq_workspace_init(ws.t)
    sxd = torch.tensor([s_x], dtype=torch.float32, device="cuda")
    fb.fp8bq_static_linear(dev(x), sxd, dev(qw), dev(sp), PARTS, y.t, ws.t)
    assert fb.fp8bq_poll_status(ws.t) == 0
    y.check("static linear y")
    ws.check("static linear workspace")
    qa = oracle.quant_static(x, s_x)
    check_close(host(y.t), oracle.gemm_static(qa, s_x, qw, sp, PARTS), "static linear")
