"""GPU test of fp8bq_check_scales against the classification it documents
("SGLang 源码完全拆解(十九)", §scale 的初始值不是零: a scale still holding the
sentinel torch.finfo(float32).min was never loaded): counts of the sentinel,
of NaN / inf entries and of other entries <= 0, and the first bad index,
computed here with numpy on the same array."""
import numpy as np
import pytest
import torch

import block_wise_fp8_gb300 as fb
import oracle
import synthetic_inputs as si

pytestmark = pytest.mark.gpu

SENTINEL = np.finfo(np.float32).min


def _expect(a):
    a = np.asarray(a, np.float32).ravel()
    sent = a == SENTINEL
    nonfin = ~np.isfinite(a)
    nonpos = ~sent & ~nonfin & ~(a > 0)
    bad = np.flatnonzero(sent | nonfin | nonpos)
    return {"sentinel": int(sent.sum()), "nonfinite": int(nonfin.sum()),
            "nonpositive": int(nonpos.sum()), "first_bad": int(bad[0]) if bad.size else -1}


def _check(a):
    got = fb.fp8bq_check_scales(torch.from_numpy(np.ascontiguousarray(a, np.float32)).cuda())
    assert got == _expect(a)
    return got


def test_quantiser_scales_are_all_usable():
    _, sw = oracle.quant_weight_block(si.weights(384, 640))
    _, sx = oracle.quant_group(si.activations(33, 640))
    assert _check(sw)["first_bad"] == -1
    assert _check(sx)["first_bad"] == -1


@pytest.mark.parametrize("n", [1, 31, 1000, 4 * 1024 * 1024 + 13])
def test_planted_values(n):
    rng = np.random.default_rng(n)
    a = rng.uniform(1e-4, 1e-2, n).astype(np.float32)
    specials = np.array([SENTINEL, np.nan, np.inf, -np.inf, 0.0, -0.0, -1e-3,
                         np.float32(1e-45), -SENTINEL], np.float32)
    idx = rng.choice(n, size=min(n, 40), replace=False)
    a[idx] = specials[rng.integers(0, specials.size, idx.size)]
    _check(a)


def test_unloaded_grid():
    """A 128x128 block grid left at the sentinel except for the blocks that a
    checkpoint entry overwrote."""
    sw = np.full((48, 48), SENTINEL, np.float32)
    sw[:, :47] = 0.001
    got = _check(sw)
    assert got["sentinel"] == 48 and got["first_bad"] == 47
