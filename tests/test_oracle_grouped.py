"""Pins of the grouped (MoE) block-scaled GEMM oracle ("SGLang 源码完全拆解
(十九)", §MoE:专家权重多一个维度: expert weights [E, N, K] with a 128x128 FP32
scale grid per expert; the grouped GEMM takes tokens sorted by expert)."""
import numpy as np

import oracle
import synthetic_inputs as si


def _experts(E, N, K, seed=0):
    qs, ss = [], []
    for e in range(E):
        q, s = oracle.quant_weight_block(si.weights(N, K, base_seed=seed + 17 * e))
        qs.append(q)
        ss.append(s)
    return np.stack(qs), np.stack(ss)


def _numpy_grouped(qa, sa, qw, sw, row_expert):
    """Independent float64 form: per row, per 128-K block, the decoded dot of the
    row with its expert's weight rows times both block scales."""
    M, K = qa.shape
    E, N, _ = qw.shape
    KB = -(-K // 128)
    da = oracle.e4m3_decode(qa)
    y = np.full((M, N), np.nan)
    for i in range(M):
        e = row_expert[i]
        if e < 0:
            continue
        dw = oracle.e4m3_decode(qw[e])
        acc = np.zeros(N)
        for kb in range(KB):
            ks = slice(kb * 128, min(K, kb * 128 + 128))
            p = dw[:, ks] @ da[i, ks]
            acc += p * float(sa[i, kb]) * sw[e][np.arange(N) // 128, kb].astype(np.float64)
        y[i] = acc
    return y


def test_grouped_matches_numpy_blockwise_form():
    E, N, K = 3, 200, 300
    off = np.array([0, 5, 5, 12])          # expert 1 has no rows
    T = 14                                  # rows 12, 13 belong to no expert
    qa, sa = oracle.quant_group(si.activations(T, K))
    qw, sw = _experts(E, N, K)
    re = oracle.row_expert_contiguous(off, T)
    y = oracle.gemm_grouped(qa, sa, qw, sw, re)
    ref = _numpy_grouped(qa, sa, qw, sw, re)
    assert np.all(np.isnan(y[12:])) and np.all(np.isnan(ref[12:]))
    np.testing.assert_allclose(y[:12], ref[:12], rtol=1e-13, atol=1e-13)


def test_grouped_one_expert_is_the_block_gemm():
    N, K, T = 260, 384, 9
    qa, sa = oracle.quant_group(si.activations(T, K))
    qw, sw = _experts(1, N, K, seed=3)
    y = oracle.gemm_grouped(qa, sa, qw, sw, np.zeros(T, np.int32))
    np.testing.assert_array_equal(y, oracle.gemm_block(qa, sa, qw[0], sw[0]))


def test_grouped_expert_relabelling():
    """Swapping two experts' weights and their row labels leaves y unchanged."""
    E, N, K, T = 4, 128, 256, 20
    qa, sa = oracle.quant_group(si.activations(T, K))
    qw, sw = _experts(E, N, K, seed=5)
    re = (np.arange(T) % E).astype(np.int32)
    y = oracle.gemm_grouped(qa, sa, qw, sw, re)
    perm = np.array([2, 0, 3, 1])
    inv = np.argsort(perm)
    y2 = oracle.gemm_grouped(qa, sa, qw[perm], sw[perm], inv[re].astype(np.int32))
    np.testing.assert_array_equal(y, y2)


def test_masked_layout_rows_and_sampled():
    E, max_m, N, K = 3, 6, 128, 128
    masked = np.array([2, 6, 0])
    re = oracle.row_expert_masked(masked, max_m)
    assert list(re) == [0, 0, -1, -1, -1, -1] + [1] * 6 + [-1] * 6
    qa, sa = oracle.quant_group(si.activations(E * max_m, K))
    qw, sw = _experts(E, N, K, seed=9)
    y = oracle.gemm_grouped(qa, sa, qw, sw, re)
    rows = np.array([0, 1, 6, 11, 7], np.int64)
    cols = np.array([0, 127, 5, 64, 64], np.int64)
    np.testing.assert_array_equal(oracle.gemm_grouped_sampled(qa, sa, qw, sw, re, rows, cols),
                                  y[rows, cols])


def test_row_expert_helpers_clamp_out_of_range_bounds():
    """Segment bounds outside [0, T] and masked counts outside [0, max_m] are
    clamped, the reading the C interface documents for both layouts."""
    assert list(oracle.row_expert_contiguous([3, 5, 9], 7)) == [-1, -1, -1, 0, 0, 1, 1]
    assert list(oracle.row_expert_contiguous([-4, 2, 2], 4)) == [0, 0, -1, -1]
    assert list(oracle.row_expert_masked([-2, 9], 3)) == [-1, -1, -1, 1, 1, 1]
    assert list(oracle.row_expert_masked([0, 1], 2)) == [-1, -1, 1, -1]
