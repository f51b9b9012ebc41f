"""GPU parity of block FP8 with UE8M0 (power-of-two) scales against the CPU
oracle: the power-of-two activation quantiser and the FP32 -> UE8M0 weight
requantisation bit-exact, the GEMM (an MXFP8 view on the block-scaled MMA)
within the GEMM tolerance of gpu_util."""
import numpy as np
import pytest
import torch

import block_wise_fp8_gb300 as fb
import oracle
import synthetic_inputs as si
from gpu_util import Guarded, assert_covers_every_block, check_close, dev, host, sample_indices

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("M,K", [(1, 6144), (5, 208), (130, 4096), (3, 16), (4096, 6144)])
def test_quant_ue8m0_bit_exact(M, K):
    x = si.activations(M, K)
    q = Guarded((M, K), torch.uint8)
    u = Guarded((M, (K + 127) // 128), torch.uint8)
    fb.fp8bq_quant_act_ue8m0(dev(x), q.t, u.t)
    torch.cuda.synchronize()
    q.check("ue8m0 codes")
    u.check("ue8m0 scale codes")
    q_ref, u_ref = oracle.quant_ue8m0(x, group=128)
    np.testing.assert_array_equal(u.t.cpu().numpy(), u_ref)
    np.testing.assert_array_equal(q.t.cpu().numpy(), q_ref)


def _requant(qw, sw, in_place=False):
    N, K = qw.shape
    dq = dev(qw)
    g_out = None if in_place else Guarded(tuple(dq.shape), torch.uint8)
    out = dq if in_place else g_out.t
    u = Guarded(tuple(sw.shape), torch.uint8)
    fb.fp8bq_requant_weight_ue8m0(dq, dev(sw), out, u.t)
    torch.cuda.synchronize()
    u.check("requant scale codes")
    if g_out is not None:
        g_out.check("requant codes")
    return out.cpu().numpy(), u.t.cpu().numpy()


@pytest.mark.parametrize("N,K", [(300, 520), (128, 128), (6144, 6144)])
def test_requant_weight_bit_exact(N, K):
    qw, sw = oracle.quant_weight_block(si.weights(N, K))
    q2, u = _requant(qw, sw)
    q2_ref, u_ref = oracle.requant_weight_ue8m0(qw, sw)
    np.testing.assert_array_equal(u, u_ref)
    np.testing.assert_array_equal(q2, q2_ref)


def test_requant_in_place():
    qw, sw = oracle.quant_weight_block(si.weights(260, 384, base_seed=4))
    q2, u = _requant(qw, sw, in_place=True)
    q2_ref, u_ref = oracle.requant_weight_ue8m0(qw, sw)
    np.testing.assert_array_equal(q2, q2_ref)
    np.testing.assert_array_equal(u, u_ref)


def _operands(M, N, K, seed=0):
    qa, ua = oracle.quant_ue8m0(si.activations(M, K, base_seed=seed), group=128)
    qw, sw = oracle.quant_weight_block(si.weights(N, K, base_seed=seed))
    qw2, uw = oracle.requant_weight_ue8m0(qw, sw)
    return qa, ua, qw2, uw


def _gemm(qa, ua, qw, uw, bias=None):
    M, K = qa.shape
    N = qw.shape[0]
    y = Guarded((M, N), torch.bfloat16, fill=float("nan"))
    ws = Guarded((fb.fp8bq_workspace_bytes(fb.OP_UE8M0_GEMM, M, N, K),), torch.uint8)
    fb.fp8bq_workspace_init(ws.t)
    fb.fp8bq_ue8m0_gemm(dev(qa), dev(ua), dev(qw), dev(uw), y.t, ws.t,
                        bias=None if bias is None else dev(bias))
    assert fb.fp8bq_poll_status(ws.t) == 0
    y.check(f"ue8m0 y {M}x{N}x{K}")
    ws.check(f"ue8m0 workspace {M}x{N}x{K}")
    return host(y.t)


@pytest.mark.parametrize("M,N,K", [(16, 384, 256), (5, 200, 96), (130, 136, 224),
                                   (257, 300, 416), (300, 520, 1024), (64, 256, 6144)])
def test_ue8m0_gemm_small_shapes(M, N, K):
    qa, ua, qw, uw = _operands(M, N, K)
    check_close(_gemm(qa, ua, qw, uw), oracle.gemm_block_ue8m0(qa, ua, qw, uw),
                f"ue8m0 {M}x{N}x{K}")


def test_ue8m0_gemm_scale_layout():
    """Distinct power-of-two codes per row block and K block on both sides."""
    M, N, K = 256, 384, 512
    rng = np.random.default_rng(8)
    qa = rng.integers(0, 0x7E, (M, K)).astype(np.uint8)
    qw = rng.integers(0, 0x7E, (N, K)).astype(np.uint8)
    ua = (120 + (np.arange(M)[:, None] * 3 + np.arange(4)[None, :]) % 15).astype(np.uint8)
    uw = (118 + (np.arange(3)[:, None] * 5 + 2 * np.arange(4)[None, :]) % 17).astype(np.uint8)
    check_close(_gemm(qa, ua, qw, uw), oracle.gemm_block_ue8m0(qa, ua, qw, uw), "ue8m0 layout")


@pytest.mark.parametrize("N", si.PREFILL["N_list"])
def test_ue8m0_gemm_prefill_sampled(N):
    M, K = si.PREFILL["M"], si.PREFILL["K"]
    qa, ua, qw, uw = _operands(M, N, K, seed=5)
    y = _gemm(qa, ua, qw, uw)
    rows, cols = sample_indices(M, N)
    assert_covers_every_block(rows, cols, M, N)
    check_close(y[rows, cols], oracle.gemm_block_ue8m0_sampled(qa, ua, qw, uw, rows, cols),
                "ue8m0 prefill")
    assert np.all(np.isfinite(y))


def test_ue8m0_linear_with_bias():
    M, N, K = 200, 256, 512
    x = si.activations(M, K)
    qw, sw = oracle.quant_weight_block(si.weights(N, K))
    qw2, uw = oracle.requant_weight_ue8m0(qw, sw)
    bias = si.f32_to_bf16_bits(np.linspace(-2, 2, N).astype(np.float32))
    y = Guarded((M, N), torch.bfloat16)
    ws = Guarded((fb.fp8bq_workspace_bytes(fb.OP_UE8M0_LINEAR, M, N, K),), torch.uint8)
    fb.fp8bq_workspace_init(ws.t)
    fb.fp8bq_ue8m0_linear(dev(x), dev(qw2), dev(uw), y.t, ws.t, bias=dev(bias))
    assert fb.fp8bq_poll_status(ws.t) == 0
    y.check("ue8m0 linear y")
    ws.check("ue8m0 linear workspace")
    qa, ua = oracle.quant_ue8m0(x, group=128)
    check_close(host(y.t), oracle.gemm_block_ue8m0(qa, ua, qw2, uw, bias=bias), "ue8m0 linear")
