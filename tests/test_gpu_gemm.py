"""GPU parity of the block-scaled FP8 GEMM and the fused linear against the CPU
oracle's binary64 result on the same quantised inputs.

Tolerance (per element |y - ref| <= 1e-2 max(1,|ref|), relative Frobenius
<= 4e-3) at sizes the oracle computes in full; at the prefill sizes on sampled
outputs.  Covers both tile orientations (decode M <= 64 swaps operands and
splits K), ragged M/N/K, both activation-scale layouts, bias, pitch > K,
determinism of the split-K reduction and an exactly representable case."""
import numpy as np
import pytest
import torch

import block_wise_fp8_gb300 as fb
import oracle
import synthetic_inputs as si
from gpu_util import Guarded, assert_covers_every_block, check_close, dev, host, sample_indices

pytestmark = pytest.mark.gpu


def _weights(N, K):
    return oracle.quant_weight_block(si.weights(N, K))


def _gemm(qa, sa, qw, sw, bias=None, layout=fb.SCALE_ROW_MAJOR, ws=None):
    M, K = qa.shape
    N = qw.shape[0]
    if layout == fb.SCALE_COL_MAJOR:
        M4 = -(-M // 4) * 4
        sa_dev = np.zeros((sa.shape[1], M4), np.float32)
        sa_dev[:, :M] = sa.T
    else:
        sa_dev = sa
    # the output and a fresh workspace sit between canary bands: a write past
    # either end fails the call
    y = Guarded((M, N), torch.bfloat16, fill=float("nan"))
    g_ws = None
    if ws is None:
        g_ws = Guarded((fb.fp8bq_workspace_bytes(fb.OP_GEMM, M, N, K),), torch.uint8)
        ws = g_ws.t
        fb.fp8bq_workspace_init(ws)
    fb.fp8bq_gemm(dev(qa), dev(sa_dev), dev(qw), dev(sw), y.t, ws,
                  bias=None if bias is None else dev(bias), s_layout=layout)
    assert fb.fp8bq_poll_status(ws) == 0
    y.check(f"y {M}x{N}x{K}")
    if g_ws is not None:
        g_ws.check(f"workspace {M}x{N}x{K}")
    return host(y.t)


@pytest.mark.parametrize("M,N,K", [(16, 384, 256), (5, 200, 208), (1, 128, 128),
                                   (64, 384, 1024), (128, 256, 128), (200, 520, 384),
                                   (256, 512, 2048), (131, 257 * 8, 144), (65, 136, 16),
                                   (130, 203, 256), (257, 300, 512), (300, 640, 1024),
                                   (520, 392, 512)])
@pytest.mark.parametrize("layout", [fb.SCALE_ROW_MAJOR, fb.SCALE_COL_MAJOR])
def test_gemm_small_shapes(M, N, K, layout):
    qa, sa = oracle.quant_group(si.activations(M, K))
    qw, sw = _weights(N, K)
    y = _gemm(qa, sa, qw, sw, layout=layout)
    check_close(y, oracle.gemm_block(qa, sa, qw, sw), f"gemm {M}x{N}x{K}")


@pytest.mark.parametrize("M", [1, 8, 32, 64])
def test_gemm_decode_full(M):
    K = N = 6144
    qa, sa = oracle.quant_group(si.activations(M, K))
    qw, sw = _weights(N, K)
    y = _gemm(qa, sa, qw, sw)
    check_close(y, oracle.gemm_block(qa, sa, qw, sw), f"decode M={M}")


@pytest.mark.parametrize("N", [6144, 24576])
def test_gemm_prefill_sampled(N):
    M, K = 4096, 6144
    qa, sa = oracle.quant_group(si.activations(M, K))
    qw, sw = _weights(N, K)
    y = _gemm(qa, sa, qw, sw)
    # every 128 x 128 output block: its corners and 4 random elements
    rows, cols = sample_indices(M, N)
    assert_covers_every_block(rows, cols, M, N)
    ref = oracle.gemm_block_sampled(qa, sa, qw, sw, rows, cols)
    check_close(y[rows, cols], ref, f"prefill N={N}")
    assert np.all(np.isfinite(y))


@pytest.mark.parametrize("M,N,K", [(1200, 3400, 1040), (2048, 4864, 6016)])
@pytest.mark.parametrize("layout", [fb.SCALE_ROW_MAJOR, fb.SCALE_COL_MAJOR])
def test_gemm_prefill_ragged_waves(M, N, K, layout):
    """Pair tiles over more than one wave of clusters, with ragged M (five
    m-tiles at 1200 rows, the last one short), ragged N and K, and a split
    tail.  Every 128 x 128 output block is sampled, with a bias, and the output
    and the workspace sit between canary bands."""
    qa, sa = oracle.quant_group(si.activations(M, K, base_seed=M + 1))
    qw, sw = _weights(N, K)
    bias = si.f32_to_bf16_bits(np.linspace(-2, 2, N).astype(np.float32))
    y = _gemm(qa, sa, qw, sw, bias=bias, layout=layout)
    rows, cols = sample_indices(M, N)
    assert_covers_every_block(rows, cols, M, N)
    ref = oracle.gemm_block_sampled(qa, sa, qw, sw, rows, cols, bias=bias)
    check_close(y[rows, cols], ref, f"prefill ragged {M}x{N}x{K}")
    assert np.all(np.isfinite(y))


def test_gemm_bias():
    M, N, K = 48, 256, 384
    qa, sa = oracle.quant_group(si.activations(M, K))
    qw, sw = _weights(N, K)
    bias = si.f32_to_bf16_bits(np.linspace(-4, 4, N).astype(np.float32))
    for m in (48, 160):  # both orientations
        qa_m, sa_m = oracle.quant_group(si.activations(m, K))
        y = _gemm(qa_m, sa_m, qw, sw, bias=bias)
        check_close(y, oracle.gemm_block(qa_m, sa_m, qw, sw, bias=bias), f"bias M={m}")
    del qa, sa


def test_gemm_integer_case_is_exact():
    """Unit scales and codes in {0, +-0.5, +-1, +-2}: every partial sum is a
    multiple of 1/4 below 2^10, exact in FP32, so the output must be exactly the
    round-to-nearest-even BF16 value of the oracle's result."""
    rng = np.random.default_rng(3)
    small = np.array([0x00, 0x30, 0xB0, 0x38, 0xB8, 0x40, 0xC0], np.uint8)
    for M in (7, 192):
        N, K = 256, 256
        qa = rng.choice(small, (M, K))
        qw = rng.choice(small, (N, K))
        sa = np.ones((M, 2), np.float32)
        sw = np.ones((2, 2), np.float32)
        y = _gemm(qa, sa, qw, sw)
        ref = oracle.gemm_block(qa, sa, qw, sw)
        assert np.all(np.abs(ref) <= 256)
        ref_bf16 = torch.from_numpy(ref).to(torch.bfloat16).double().numpy()
        assert np.array_equal(y, ref_bf16)


def test_split_k_reduction_is_deterministic():
    M, N, K = 8, 6144, 6144
    qa, sa = oracle.quant_group(si.activations(M, K))
    qw, sw = _weights(N, K)
    ws = fb.new_workspace(fb.OP_GEMM, M, N, K)
    ys = [_gemm(qa, sa, qw, sw, ws=ws) for _ in range(3)]
    assert np.array_equal(ys[0], ys[1]) and np.array_equal(ys[1], ys[2])


@pytest.mark.parametrize("M,N,K", [(300, 1000, 6016), (512, 768, 1152), (256, 512, 2048)])
@pytest.mark.parametrize("layout", [fb.SCALE_ROW_MAJOR, fb.SCALE_COL_MAJOR])
def test_gemm_split_tail_tiles(M, N, K, layout):
    """Few pair tiles against many clusters: the tiles are split into K ranges
    (47 K blocks in 4 ranges with a short last one; 9 in ranges of 8 and 1) and
    the last range to finish sums the promoted partials.  With a bias, which
    only the summing range adds; three calls on one workspace agree bit for bit
    (the sum runs in range order)."""
    qa, sa = oracle.quant_group(si.activations(M, K, base_seed=M))
    qw, sw = _weights(N, K)
    bias = si.f32_to_bf16_bits(np.linspace(-3, 3, N).astype(np.float32))
    ws = fb.new_workspace(fb.OP_GEMM, M, N, K)
    ys = [_gemm(qa, sa, qw, sw, bias=bias, layout=layout, ws=ws) for _ in range(3)]
    ref = oracle.gemm_block(qa, sa, qw, sw, bias=bias)
    check_close(ys[0], ref, f"split tail {M}x{N}x{K}")
    assert np.array_equal(ys[0], ys[1]) and np.array_equal(ys[1], ys[2])
    # the no-allocation entry point has no room for the partials and runs the
    # tiles whole: the same result within the tolerance, a different FP32
    # summation order (so the split path did run)
    if layout == fb.SCALE_ROW_MAJOR:
        y1 = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
        fb.fp8bq_gemm_noalloc(dev(qa), dev(sa), dev(qw), dev(sw), y1, bias=dev(bias))
        torch.cuda.synchronize()
        y_whole = host(y1)
        check_close(y_whole, ref, f"whole tiles {M}x{N}x{K}")
        assert not np.array_equal(y_whole, ys[0])


@pytest.mark.parametrize("M,N,K", [(16, 384, 256), (1, 6144, 6144), (64, 6144, 6144),
                                   (300, 384, 256), (4096, 6144, 6144)])
def test_linear_matches_oracle(M, N, K):
    x = si.activations(M, K)
    qw, sw = _weights(N, K)
    qa, sa = oracle.quant_group(x)
    xd = dev(x)
    y = Guarded((M, N), torch.bfloat16)
    g_ws = Guarded((fb.fp8bq_workspace_bytes(fb.OP_LINEAR, M, N, K),), torch.uint8)
    fb.fp8bq_workspace_init(g_ws.t)
    fb.fp8bq_linear(xd, dev(qw), dev(sw), y.t, g_ws.t)
    assert fb.fp8bq_poll_status(g_ws.t) == 0
    y.check("linear y")
    g_ws.check("linear workspace")
    yh = host(y.t)
    if M * N * K <= 64 * 6144 * 6144:
        check_close(yh, oracle.gemm_block(qa, sa, qw, sw), f"linear {M}x{N}x{K}")
    else:
        rows, cols = sample_indices(M, N)
        check_close(yh[rows, cols], oracle.gemm_block_sampled(qa, sa, qw, sw, rows, cols),
                    f"linear {M}x{N}x{K}")


def test_linear_with_pitch_and_bias():
    M, N, K = 40, 256, 512
    x = si.activations(M, K)
    qw, sw = _weights(N, K)
    bias = si.f32_to_bf16_bits(np.linspace(-1, 1, N).astype(np.float32))
    wide = torch.zeros(M, K + 128, dtype=torch.bfloat16, device="cuda")
    wide[:, :K] = dev(x)
    y = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    ws = fb.new_workspace(fb.OP_LINEAR, M, N, K)
    fb.fp8bq_linear(wide[:, :K], dev(qw), dev(sw), y, ws, bias=dev(bias))
    assert fb.fp8bq_poll_status(ws) == 0
    qa, sa = oracle.quant_group(x)
    check_close(host(y), oracle.gemm_block(qa, sa, qw, sw, bias=bias), "linear pitch+bias")


def test_empty_batch():
    ws = fb.new_workspace(fb.OP_GEMM, 0, 256, 256)
    y = torch.empty(0, 256, dtype=torch.bfloat16, device="cuda")
    q = torch.empty(0, 256, dtype=torch.uint8, device="cuda")
    s = torch.empty(0, 2, dtype=torch.float32, device="cuda")
    w = torch.zeros(256, 256, dtype=torch.uint8, device="cuda")
    sw = torch.ones(2, 2, dtype=torch.float32, device="cuda")
    fb.fp8bq_gemm(q, s, w, sw, y, ws)
    torch.cuda.synchronize()


@pytest.mark.parametrize("M,N,K", [(1, 6144, 6144), (4, 1024, 6144), (5, 200, 208), (9, 384, 4000),
                                   (16, 384, 256), (17, 640, 1040), (33, 1000, 2048), (64, 6144, 6144),
                                   (8, 24576, 6144)])
def test_decode_linear_fuses_quantisation_bit_exactly(M, N, K):
    """Up to 16 tokens fp8bq_linear is one launch: the GEMM's CTAs quantise their
    own K range of X as the stages arrive, the quantiser warps in groups that
    take the stages in turn (one warp per stage up to 4 tokens, two up to 8,
    four up to 16).  Its output must be bit for bit that of the quantiser
    followed by the GEMM (the same codes, scales, MMAs and promotion order),
    with the bias and a row pitch wider than K, and within the GEMM tolerance
    of the oracle.  Above 16 tokens the linear is the two launches themselves."""
    x = si.activations(M, K, base_seed=M + K)
    qw, sw = _weights(N, K)
    bias = si.f32_to_bf16_bits(np.linspace(-2, 2, N).astype(np.float32))
    wide = torch.zeros(M, K + 64, dtype=torch.bfloat16, device="cuda")
    wide[:, :K] = dev(x)
    xd = wide[:, :K]
    y = Guarded((M, N), torch.bfloat16, fill=float("nan"))
    g_ws = Guarded((fb.fp8bq_workspace_bytes(fb.OP_LINEAR, M, N, K),), torch.uint8)
    fb.fp8bq_workspace_init(g_ws.t)
    fb.fp8bq_linear(xd, dev(qw), dev(sw), y.t, g_ws.t, bias=dev(bias))
    assert fb.fp8bq_poll_status(g_ws.t) == 0
    y.check("fused linear y")
    g_ws.check("fused linear workspace")
    q = torch.empty(M, K, dtype=torch.uint8, device="cuda")
    s = torch.empty(M, -(-K // 128), dtype=torch.float32, device="cuda")
    fb.fp8bq_quant_act(xd, q, s)
    y2 = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    ws2 = fb.new_workspace(fb.OP_GEMM, M, N, K)
    fb.fp8bq_gemm(q, s, dev(qw), dev(sw), y2, ws2, bias=dev(bias))
    assert fb.fp8bq_poll_status(ws2) == 0
    assert torch.equal(y.t.view(torch.int16), y2.view(torch.int16))
    qa, sa = oracle.quant_group(x)
    rows, cols = sample_indices(M, N, per_block=16)
    check_close(host(y.t)[rows, cols],
                oracle.gemm_block_sampled(qa, sa, qw, sw, rows, cols, bias=bias),
                f"fused linear {M}x{N}x{K}")
