"""GPU parity of the grouped (MoE) block-scaled GEMM against the CPU oracle
("SGLang 源码完全拆解(十九)", §MoE:专家权重多一个维度: expert weights
[E, N, K] with one 128 x 128 FP32 scale grid per expert; rows sorted by
expert, contiguous, or the masked [E, max_m, K] layout).  Rows of no expert
must be left as they were (NaN here)."""
import numpy as np
import pytest
import torch

import block_wise_fp8_gb300 as fb
import oracle
import synthetic_inputs as si
from gpu_util import Guarded, assert_covers_every_block, check_close, dev, host, sample_indices

pytestmark = pytest.mark.gpu


def _experts(E, N, K, distinct=None, seed=0):
    """Expert codes [E, N, K] and scale grids [E, NB, KB].  With `distinct`,
    only that many weight sets are drawn and expert e reuses set e % distinct
    with its scale grid times 2^(e // distinct - 2): every expert still has its
    own exact values, so a mix-up of experts shows as a power-of-two error."""
    n = E if distinct is None else distinct
    sets = [oracle.quant_weight_block(si.weights(N, K, base_seed=seed + 31 * e)) for e in range(n)]
    qw = np.stack([sets[e % n][0] for e in range(E)])
    sw = np.stack([(sets[e % n][1] * np.float32(2.0 ** (e // n - 2))).astype(np.float32)
                   for e in range(E)])
    return qw, sw


def _acts(T, K, seed=0, layout=fb.SCALE_ROW_MAJOR):
    qa, sa = oracle.quant_group(si.activations(T, K, base_seed=seed))
    if layout == fb.SCALE_COL_MAJOR:
        KB = sa.shape[1]
        Mp = (T + 3) // 4 * 4
        sac = np.zeros((KB, Mp), np.float32)
        sac[:, :T] = sa.T
        return qa, sa, sac
    return qa, sa, sa


def _run_contiguous(qa, sa_dev_layout, qw, sw, offsets, layout=fb.SCALE_ROW_MAJOR):
    T, K = qa.shape
    E, N, _ = qw.shape
    y = Guarded((T, N), torch.bfloat16, fill=float("nan"))
    ws = Guarded((fb.fp8bq_workspace_bytes(fb.OP_GROUPED_GEMM, T, N, K),), torch.uint8)
    fb.fp8bq_workspace_init(ws.t)
    off = torch.tensor(np.asarray(offsets, np.int32), device="cuda")
    fb.fp8bq_grouped_gemm(dev(qa), dev(sa_dev_layout), dev(qw), dev(sw), off, y.t, ws.t,
                          s_layout=layout)
    assert fb.fp8bq_poll_status(ws.t) == 0
    y.check(f"grouped y {T}x{N}x{K}")
    ws.check(f"grouped workspace {T}x{N}x{K}")
    return host(y.t)


def _check_rows(y, ref, row_expert, what):
    on = row_expert >= 0
    assert np.all(np.isnan(y[~on])), f"{what}: rows of no expert were written"
    if on.any():
        check_close(y[on], ref[on], what)


@pytest.mark.parametrize("counts,T,N,K", [
    ([5, 0, 7], 14, 200, 304),          # an empty expert; two rows of no expert at the end
    ([300, 1, 0, 513], 814, 384, 512),  # segments straddling 256-row tiles, a 1-row segment
    ([40, 260], 300, 256, 6144),        # long K
    ([129, 127, 256, 33], 545, 136, 128),
])
def test_grouped_contiguous(counts, T, N, K):
    E = len(counts)
    off = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    qa, _, sa = _acts(T, K, seed=E)
    qw, sw = _experts(E, N, K, seed=K)
    re = oracle.row_expert_contiguous(off, T)
    y = _run_contiguous(qa, sa, qw, sw, off)
    _check_rows(y, oracle.gemm_grouped(qa, sa, qw, sw, re), re, f"grouped {counts} N={N} K={K}")


def test_grouped_leading_gap_and_col_major_scales():
    """Rows before offsets[0] belong to no expert; s_x column-major."""
    counts, T, N, K = [70, 200, 3], 300, 256, 384
    off = np.concatenate([[20], 20 + np.cumsum(counts)]).astype(np.int32)
    qa, sa, sac = _acts(T, K, seed=7, layout=fb.SCALE_COL_MAJOR)
    qw, sw = _experts(3, N, K, seed=11)
    re = oracle.row_expert_contiguous(off, T)
    y = _run_contiguous(qa, sac, qw, sw, off, layout=fb.SCALE_COL_MAJOR)
    _check_rows(y, oracle.gemm_grouped(qa, sa, qw, sw, re), re, "grouped gap col-major")


@pytest.mark.parametrize("layout", [fb.SCALE_ROW_MAJOR, fb.SCALE_COL_MAJOR])
def test_grouped_long_segments_pair_tiles(layout):
    """More than 512 rows per expert on average: 256-row pair tiles, with a
    3-row segment and segments ending inside both halves of a pair tile."""
    counts, N, K = [1100, 3, 900, 130], 384, 512
    T = sum(counts) + 5
    assert T > 512 * len(counts)
    off = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    qa, sa, sa_dev = _acts(T, K, seed=21, layout=layout)
    qw, sw = _experts(len(counts), N, K, seed=23)
    re = oracle.row_expert_contiguous(off, T)
    y = _run_contiguous(qa, sa_dev, qw, sw, off, layout=layout)
    _check_rows(y, oracle.gemm_grouped(qa, sa, qw, sw, re), re, f"grouped pair layout={layout}")


def test_grouped_many_experts():
    """70 experts: the tile scan runs over three 32-expert steps."""
    E, T, N, K = 70, 900, 128, 128
    counts = si.expert_counts(T, E, base_seed=3)
    off = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    qa, _, sa = _acts(T, K, seed=9)
    qw, sw = _experts(E, N, K, distinct=5, seed=2)
    re = oracle.row_expert_contiguous(off, T)
    y = _run_contiguous(qa, sa, qw, sw, off)
    _check_rows(y, oracle.gemm_grouped(qa, sa, qw, sw, re), re, "grouped 70 experts")


def test_grouped_masked():
    """masked_m outside [0, max_m] is clamped; unused slot rows stay unwritten."""
    E, max_m, N, K = 5, 300, 256, 256
    masked = np.array([0, 17, 300, 129, 999], np.int32)
    T = E * max_m
    qa, _, sa = _acts(T, K, seed=4)
    qw, sw = _experts(E, N, K, seed=5)
    y = Guarded((E, max_m, N), torch.bfloat16, fill=float("nan"))
    ws = Guarded((fb.fp8bq_workspace_bytes(fb.OP_GROUPED_GEMM, T, N, K),), torch.uint8)
    fb.fp8bq_workspace_init(ws.t)
    fb.fp8bq_grouped_gemm_masked(dev(qa).view(E, max_m, K), dev(sa), dev(qw), dev(sw),
                                 torch.tensor(masked, device="cuda"), y.t, ws.t)
    assert fb.fp8bq_poll_status(ws.t) == 0
    y.check("grouped masked y")
    ws.check("grouped masked workspace")
    re = oracle.row_expert_masked(masked, max_m)
    _check_rows(host(y.t).reshape(T, N), oracle.gemm_grouped(qa, sa, qw, sw, re), re,
                "grouped masked")


def test_grouped_masked_negative_count():
    E, max_m, N, K = 2, 64, 128, 128
    masked = np.array([-5, 64], np.int32)
    qa, _, sa = _acts(E * max_m, K, seed=6)
    qw, sw = _experts(E, N, K, seed=8)
    y = torch.full((E * max_m, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    ws = fb.new_workspace(fb.OP_GROUPED_GEMM, E * max_m, N, K)
    fb.fp8bq_grouped_gemm_masked(dev(qa), dev(sa), dev(qw), dev(sw),
                                 torch.tensor(masked, device="cuda"), y, ws)
    assert fb.fp8bq_poll_status(ws) == 0
    re = oracle.row_expert_masked(np.maximum(masked, 0), max_m)
    _check_rows(host(y), oracle.gemm_grouped(qa, sa, qw, sw, re), re, "masked negative")


def test_grouped_all_empty():
    E, T, N, K = 3, 40, 128, 128
    qa, _, sa = _acts(T, K)
    qw, sw = _experts(E, N, K)
    y = _run_contiguous(qa, sa, qw, sw, np.zeros(E + 1, np.int32))
    assert np.all(np.isnan(y))


@pytest.mark.parametrize("which", ["w13", "w2"])
def test_grouped_moe_workload_sampled(which):
    """The MoE workload: 32 local experts, 4096 routed rows with skewed routing;
    w13 [E, 2I, H] or w2 [E, H, I], checked on sampled outputs."""
    mo = si.MOE
    E, T = mo["E"], mo["T"]
    N, K = (2 * mo["I"], mo["H"]) if which == "w13" else (mo["H"], mo["I"])
    counts = si.expert_counts(T, E, mo["skew"])
    off = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    qa, _, sa = _acts(T, K, seed=1)
    qw, sw = _experts(E, N, K, distinct=4, seed=13)
    y = _run_contiguous(qa, sa, qw, sw, off)
    assert np.all(np.isfinite(y))
    re = oracle.row_expert_contiguous(off, T)
    rows, cols = sample_indices(T, N)
    assert_covers_every_block(rows, cols, T, N)
    # also the first and last row of every expert
    rows = np.concatenate([rows, off[:-1][counts > 0], off[1:][counts > 0] - 1]).astype(np.int64)
    cols = np.concatenate([cols, np.arange(2 * int((counts > 0).sum())) * 97 % N]).astype(np.int64)
    check_close(y[rows, cols], oracle.gemm_grouped_sampled(qa, sa, qw, sw, re, rows, cols),
                f"grouped {which}")
