"""fp8bq_gemm_noalloc, called through the C ABI, against fp8bq_gemm.

The entry point is for callers that cannot give the library device memory: an
operator with a fixed argument list that has no place for a workspace, or a
runtime that plans all device memory ahead and allows no allocation inside its
operators.  It runs the GEMM of fp8bq_gemm on a fixed scratch array inside the
library instead of a caller workspace, so its output must match fp8bq_gemm's
within the GEMM tolerance of the other tests, call after call, although every
call reuses the scratch the previous one left behind.

The file name makes pytest collect it last, after every other test has used
the library; it must also pass on its own in a fresh process."""
import ctypes

import pytest
import torch

import block_wise_fp8_gb300 as fb
import synthetic_inputs as si
from gpu_util import check_close, dev, host

pytestmark = pytest.mark.gpu

LIB = fb._lib
P = ctypes.c_void_p


def _p(t):
    return None if t is None else P(t.data_ptr())


def _operands(M, N, K, seed, with_bias):
    """E4M3 activations and weights with their FP32 scales, quantised on the GPU."""
    x = dev(si.activations(M, K, base_seed=seed))
    w = dev(si.weights(N, K, base_seed=seed))
    q = torch.empty(M, K, dtype=torch.uint8, device="cuda")
    s_x = torch.empty(M, -(-K // 128), dtype=torch.float32, device="cuda")
    qw = torch.empty(N, K, dtype=torch.uint8, device="cuda")
    s_w = torch.empty(-(-N // 128), -(-K // 128), dtype=torch.float32, device="cuda")
    fb.fp8bq_quant_act(x, q, s_x)
    fb.fp8bq_quant_weight_block(w, qw, s_w)
    bias = None
    if with_bias:
        bias = dev(si.activations(1, N, outliers=False, base_seed=seed + 7).reshape(N))
    return q, s_x, qw, s_w, bias


def _noalloc(q, s_x, qw, s_w, bias, stream):
    M, K = q.shape
    N = qw.shape[0]
    y = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    st = P(stream.cuda_stream)
    status = LIB.fp8bq_gemm_noalloc(_p(q), _p(s_x), fb.SCALE_ROW_MAJOR, _p(qw), _p(s_w),
                                    _p(bias), _p(y), M, N, K, st)
    assert status == 0, fb.fp8bq_status_string(status)
    return y


def _with_workspace(q, s_x, qw, s_w, bias):
    M, K = q.shape
    N = qw.shape[0]
    y = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    ws = fb.new_workspace(fb.OP_GEMM, M, N, K)
    fb.fp8bq_gemm(q, s_x, qw, s_w, y, ws, bias=bias)
    assert fb.fp8bq_poll_status(ws) == 0
    return y


# (M, N, K, bias): decode shapes take the split-K tiles, whose FP32 partials and
# tile counters live in the scratch; the last one takes the 2-CTA prefill tiles
# with ragged M, N and K.
SEQUENCE = [(64, 6144, 6144, True), (64, 6144, 6144, False), (1, 6144, 6144, True),
            (300, 704, 1040, True)]


def test_noalloc_matches_workspace_gemm_on_consecutive_calls():
    stream = torch.cuda.Stream()
    for i, (M, N, K, with_bias) in enumerate(SEQUENCE):
        ops = _operands(M, N, K, seed=100 + i, with_bias=with_bias)
        torch.cuda.synchronize()
        with torch.cuda.stream(stream):
            y = _noalloc(*ops, stream)
        # no wait of the call ran out (the status word of the scratch array)
        assert LIB.fp8bq_noalloc_poll_status(P(stream.cuda_stream)) == 0
        ref = _with_workspace(*ops)
        torch.cuda.synchronize()
        check_close(host(y), host(ref), f"call {i}: M={M} N={N} K={K}")


def test_noalloc_rejects_shapes_beyond_its_scratch():
    """M=64, N=24576 would need 50 MB of split-K partials: rejected on the host
    with FP8BQ_ERR_WORKSPACE, nothing launched, the output left untouched."""
    M, N, K = 64, 24576, 6144
    assert fb.fp8bq_workspace_bytes(fb.OP_GEMM, M, N, K) > fb.NOALLOC_SCRATCH_BYTES
    q = torch.zeros(M, K, dtype=torch.uint8, device="cuda")
    s_x = torch.ones(M, K // 128, dtype=torch.float32, device="cuda")
    qw = torch.zeros(N, K, dtype=torch.uint8, device="cuda")
    s_w = torch.ones(N // 128, K // 128, dtype=torch.float32, device="cuda")
    y = torch.full((M, N), 7.0, dtype=torch.bfloat16, device="cuda")
    status = LIB.fp8bq_gemm_noalloc(_p(q), _p(s_x), fb.SCALE_ROW_MAJOR, _p(qw), _p(s_w), None,
                                    _p(y), M, N, K, None)
    torch.cuda.synchronize()
    assert status == 6
    assert bool(torch.all(y == 7.0))
    # the largest decode width that fits still runs and matches
    ops = _operands(16, N, K, seed=200, with_bias=False)
    torch.cuda.synchronize()
    y16 = _noalloc(*ops, torch.cuda.current_stream())
    torch.cuda.synchronize()
    check_close(host(y16), host(_with_workspace(*ops)), "M=16 N=24576")
