"""The Python binding checks every tensor argument against the call's sizes
before it takes a pointer: a wrong shape, dtype, layout or device raises
ValueError and nothing reaches the C library.  These tests need no GPU: tensors
of the right shape on the host fail only the device check, which comes last, so
each case below shows which check fired."""
import pytest
import torch

import block_wise_fp8_gb300 as fb

BF16, U8, F32, I32 = torch.bfloat16, torch.uint8, torch.float32, torch.int32


def z(*shape, dtype=U8):
    return torch.zeros(*shape, dtype=dtype)


def gemm_args(M=40, N=300, K=256):
    KB, NB = -(-K // 128), -(-N // 128)
    return dict(q=z(M, K), s_x=z(M, KB, dtype=F32), w=z(N, K), s_w=z(NB, KB, dtype=F32),
                y=z(M, N, dtype=BF16), ws=z(1024))


def call_gemm(**kw):
    a = gemm_args()
    a.update(kw)
    bias = a.pop("bias", None)
    layout = a.pop("s_layout", fb.SCALE_ROW_MAJOR)
    fb.fp8bq_gemm(a["q"], a["s_x"], a["w"], a["s_w"], a["y"], a["ws"], bias=bias,
                  s_layout=layout)


def raises(match, fn, *a, **kw):
    with pytest.raises(ValueError, match=match):
        fn(*a, **kw)


def test_well_formed_host_tensors_fail_only_on_the_device():
    raises("must be a CUDA tensor", call_gemm)


def test_gemm_output_too_small_is_rejected():
    raises(r"y must have shape \(40, 300\)", call_gemm, y=z(39, 300, dtype=BF16))
    raises(r"y must have shape", call_gemm, y=z(40 * 300 - 1, dtype=BF16))


def test_gemm_wrong_dtypes():
    raises("y must be bfloat16", call_gemm, y=z(40, 300, dtype=F32))
    raises("s_x must be float32", call_gemm, s_x=z(40, 2, dtype=BF16))
    raises("q must be uint8 or float8_e4m3fn", call_gemm, q=z(40, 256, dtype=BF16))


def test_gemm_scale_shapes_follow_the_layout():
    raises(r"s_x must have shape \(40, 2\)", call_gemm, s_x=z(2, 40, dtype=F32))
    # column-major: [ceil(K/128)][M rounded up to 4]
    raises(r"s_x must have shape \(2, 40\)", call_gemm, s_x=z(40, 2, dtype=F32),
           s_layout=fb.SCALE_COL_MAJOR)
    raises("must be a CUDA tensor", call_gemm, s_x=z(2, 40, dtype=F32),
           s_layout=fb.SCALE_COL_MAJOR)
    raises(r"s_w must have shape \(3, 2\)", call_gemm, s_w=z(2, 3, dtype=F32))
    raises("s_layout must be", call_gemm, s_layout=7)


def test_gemm_bias_and_contiguity():
    raises("bias must have 300 elements", call_gemm, bias=z(299, dtype=BF16))
    raises("must be a CUDA tensor", call_gemm, bias=z(300, dtype=BF16))
    raises("q must be contiguous", call_gemm, q=z(256, 40).t())
    raises("ws must be contiguous", call_gemm, ws=z(1024, 2)[:, 0])


def test_linear_input_pitch():
    M, N, K = 8, 256, 512
    w, s_w, y, ws = z(N, K), z(2, 4, dtype=F32), z(M, N, dtype=BF16), z(256)
    wide = z(M, K + 64, dtype=BF16)
    raises("must be a CUDA tensor", fb.fp8bq_linear, wide[:, :K], w, s_w, y, ws)
    raises("unit stride", fb.fp8bq_linear, z(K, M, dtype=BF16).t(), w, s_w, y, ws)
    raises(r"w must have shape \(256, 512\)", fb.fp8bq_linear, wide[:, :K], z(N, K - 16), s_w,
           y, ws)


def test_quantiser_outputs():
    x = z(5, 208, dtype=BF16)
    raises(r"q must have shape \(5, 208\)", fb.fp8bq_quant_act, x, z(5, 200), z(5, 2, dtype=F32))
    raises(r"s must have shape \(2, 8\)", fb.fp8bq_quant_act, x, z(5, 208), z(5, 2, dtype=F32),
           fb.SCALE_COL_MAJOR)
    raises(r"s must have shape \(5, 6\)", fb.fp8bq_mx_quant_act, z(5, 192, dtype=BF16),
           z(5, 192), z(5, 5))
    raises("s_x must have 1 elements", fb.fp8bq_static_quant_act, x, z(2, dtype=F32), z(5, 208))
    raises("s must have 5 elements", fb.fp8bq_channel_quant_act, x, z(5, 208), z(4, dtype=F32))
    raises(r"u must have shape \(5, 2\)", fb.fp8bq_quant_act_ue8m0, x, z(5, 208), z(5, 1))


def test_other_gemms():
    M, N, K = 16, 384, 256
    q, w, y, ws = z(M, K), z(N, K), z(M, N, dtype=BF16), z(256)
    raises(r"s_w must have shape \(384, 8\)", fb.fp8bq_mx_gemm, q, z(M, 8), w, z(N, 4), y, ws)
    raises("s_w must have 384 elements", fb.fp8bq_channel_gemm, q, z(M, dtype=F32), w,
           z(N - 1, dtype=F32), y, ws)
    raises(r"u_w must have shape \(3, 2\)", fb.fp8bq_ue8m0_gemm, q, z(M, 2), w, z(2, 3), y, ws)
    raises("s_w_part must have 2 elements", fb.fp8bq_static_gemm, q, z(1, dtype=F32), w,
           z(3, dtype=F32), [128, 256], y, ws)


def test_grouped_gemms():
    E, T, N, K = 3, 40, 256, 128
    q, s_x, w = z(T, K), z(T, 1, dtype=F32), z(E, N, K)
    s_w, y, ws = z(E, 2, 1, dtype=F32), z(T, N, dtype=BF16), z(256)
    raises("offsets must have 4 elements", fb.fp8bq_grouped_gemm, q, s_x, w, s_w,
           z(3, dtype=I32), y, ws)
    raises("offsets must be int32", fb.fp8bq_grouped_gemm, q, s_x, w, s_w,
           z(4, dtype=torch.int64), y, ws)
    raises(r"s_w must have shape \(3, 2, 1\)", fb.fp8bq_grouped_gemm, q, s_x, w,
           z(E, 1, 2, dtype=F32), z(4, dtype=I32), y, ws)
    raises("3-D", fb.fp8bq_grouped_gemm, q, s_x, z(N, K), s_w, z(4, dtype=I32), y, ws)
    raises("E \\* max_m rows", fb.fp8bq_grouped_gemm_masked, z(41, K), s_x, w, s_w,
           z(E, dtype=I32), y, ws)
    raises("y must have 10752 elements", fb.fp8bq_grouped_gemm_masked, z(E, 14, K),
           z(E * 14, 1, dtype=F32), w, s_w, z(E, dtype=I32), z(E * 14, N - 1, dtype=BF16), ws)


def test_norm_outputs():
    M, K = 4, 256
    x, g = z(M, K, dtype=BF16), z(K, dtype=BF16)
    raises(r"residual_out must have shape \(4, 256\)", fb.fp8bq_add_rmsnorm_quant_act, x, g,
           1e-5, residual_out=z(M, K - 8, dtype=BF16))
    raises("gamma must have 256 elements", fb.fp8bq_add_rmsnorm_quant_act, x, z(K // 2,
           dtype=BF16), 1e-5)
    raises("s is required", fb.fp8bq_add_rmsnorm_quant_act, x, g, 1e-5, q=z(M, K))
    raises(r"q must have shape \(4, 256\)", fb.fp8bq_add_rmsnorm_static_quant_act, x, g, 1e-5,
           z(1, dtype=F32), z(M, K // 2))


def test_setup_helpers():
    raises(r"s_w must have shape \(2, 2\)", fb.fp8bq_quant_weight_block, z(200, 208, dtype=BF16),
           z(200, 208), z(2, 1, dtype=F32))
    raises("s must have 1 elements", fb.fp8bq_absmax_scale, z(8, 64, dtype=BF16),
           z(2, dtype=F32))
    raises("scratch must have 4 elements", fb.fp8bq_check_scales, z(16, dtype=F32),
           z(3, dtype=torch.int64))
