"""GPU parity of the channelwise W8A8 path (per-token activation scales, per-
channel weight scales) against the CPU oracle: codes and scales bit-exact, the
GEMM within the GEMM tolerance of gpu_util."""
import numpy as np
import pytest
import torch

import block_wise_fp8_gb300 as fb
import oracle
import synthetic_inputs as si
from gpu_util import Guarded, assert_covers_every_block, check_close, dev, host, sample_indices

pytestmark = pytest.mark.gpu


def _quant(x):
    M, K = x.shape
    q = Guarded((M, K), torch.uint8)
    s = Guarded((M,), torch.float32)
    fb.fp8bq_channel_quant_act(dev(x), q.t, s.t)
    torch.cuda.synchronize()
    q.check("per-token codes")
    s.check("per-token scales")
    return q.t.cpu().numpy(), s.t.cpu().numpy()


@pytest.mark.parametrize("M,K", [(1, 6144), (5, 208), (130, 4096), (3, 16), (2, 20480),
                                 (4096, 6144)])
def test_channel_quant_bit_exact(M, K):
    x = si.activations(M, K)
    q, s = _quant(x)
    q_ref, s_ref = oracle.quant_channel(x)
    np.testing.assert_array_equal(s, s_ref)
    np.testing.assert_array_equal(q, q_ref)


def test_channel_quant_zero_rows():
    x = np.zeros((4, 256), np.uint16)
    x[2] = si.activations(1, 256)[0]
    q, s = _quant(x)
    q_ref, s_ref = oracle.quant_channel(x)
    np.testing.assert_array_equal(s, s_ref)
    np.testing.assert_array_equal(q, q_ref)


def _gemm(qa, sa, qw, sw, bias=None):
    M, K = qa.shape
    N = qw.shape[0]
    y = Guarded((M, N), torch.bfloat16, fill=float("nan"))
    ws = Guarded((fb.fp8bq_workspace_bytes(fb.OP_CHANNEL_GEMM, M, N, K),), torch.uint8)
    fb.fp8bq_workspace_init(ws.t)
    fb.fp8bq_channel_gemm(dev(qa), dev(sa), dev(qw), dev(sw), y.t, ws.t,
                          bias=None if bias is None else dev(bias))
    assert fb.fp8bq_poll_status(ws.t) == 0
    y.check(f"channel y {M}x{N}x{K}")
    ws.check(f"channel workspace {M}x{N}x{K}")
    return host(y.t)


def _operands(M, N, K, seed=0):
    qa, sa = oracle.quant_channel(si.activations(M, K, base_seed=seed))
    qw, sw = oracle.quant_channel(si.weights(N, K, base_seed=seed))
    return qa, sa, qw, sw


# (8, 9728, 768) and (3, 6400, 768): decode tiles whose splits hold 3 and 2 K
# blocks, so only some of the four MMA issuers' accumulators receive any
@pytest.mark.parametrize("M,N,K", [(16, 384, 256), (5, 200, 208), (130, 136, 224),
                                   (257, 300, 512), (520, 392, 512), (64, 640, 1024),
                                   (1, 128, 128), (8, 9728, 768), (3, 6400, 768)])
def test_channel_gemm_small_shapes(M, N, K):
    qa, sa, qw, sw = _operands(M, N, K)
    check_close(_gemm(qa, sa, qw, sw), oracle.gemm_channel(qa, sa, qw, sw), f"channel {M}x{N}x{K}")


def test_channel_gemm_row_and_column_scales_located():
    """Distinct powers of two per token and per channel: a transposed or shifted
    scale index fails."""
    M, N, K = 40, 300, 256
    qa, _, qw, _ = _operands(M, N, K, seed=3)
    sa = np.exp2(-(np.arange(M) % 7)).astype(np.float32) * np.float32(0.01)
    sw = np.exp2(-(np.arange(N) % 11)).astype(np.float32) * np.float32(0.002)
    check_close(_gemm(qa, sa, qw, sw), oracle.gemm_channel(qa, sa, qw, sw), "channel scales")


@pytest.mark.parametrize("M", si.DECODE["M_list"])
def test_channel_gemm_decode_sampled(M):
    K = N = si.DECODE["K"]
    qa, sa, qw, sw = _operands(M, N, K, seed=7)
    y = _gemm(qa, sa, qw, sw)
    rows, cols = sample_indices(M, N, per_block=32)
    assert_covers_every_block(rows, cols, M, N)
    check_close(y[rows, cols], oracle.gemm_channel_sampled(qa, sa, qw, sw, rows, cols),
                f"channel decode M={M}")
    assert np.all(np.isfinite(y))


@pytest.mark.parametrize("N", si.PREFILL["N_list"])
def test_channel_gemm_prefill_sampled(N):
    M, K = si.PREFILL["M"], si.PREFILL["K"]
    qa, sa, qw, sw = _operands(M, N, K, seed=9)
    y = _gemm(qa, sa, qw, sw)
    rows, cols = sample_indices(M, N)
    assert_covers_every_block(rows, cols, M, N)
    check_close(y[rows, cols], oracle.gemm_channel_sampled(qa, sa, qw, sw, rows, cols),
                "channel prefill")
    assert np.all(np.isfinite(y))


@pytest.mark.parametrize("M", [3, 300])
def test_channel_linear_with_bias(M):
    N, K = 256, 512
    x = si.activations(M, K)
    qw, sw = oracle.quant_channel(si.weights(N, K))
    bias = si.f32_to_bf16_bits(np.linspace(-2, 2, N).astype(np.float32))
    y = Guarded((M, N), torch.bfloat16)
    ws = Guarded((fb.fp8bq_workspace_bytes(fb.OP_CHANNEL_LINEAR, M, N, K),), torch.uint8)
    fb.fp8bq_workspace_init(ws.t)
    fb.fp8bq_channel_linear(dev(x), dev(qw), dev(sw), y.t, ws.t, bias=dev(bias))
    assert fb.fp8bq_poll_status(ws.t) == 0
    y.check("channel linear y")
    ws.check("channel linear workspace")
    qa, sa = oracle.quant_channel(x)
    check_close(host(y.t), oracle.gemm_channel(qa, sa, qw, sw, bias=bias), f"channel linear M={M}")
