"""The hardware binary32 -> E4M3 conversion that every quantiser ends with,
against the oracle's encoder, over all 2^32 binary32 bit patterns.

The rule ("SGLang 源码完全拆解(十九)", §从浮点到 FP8 的基本公式): q = clamp(
round(x/s), -448, 448) with round-to-nearest-even.  The quantisers feed
arbitrary binary32 quotients into the conversion, so the BF16-input sweeps of
test_gpu_quant.py reach only some of its inputs; this sweep reaches all of
them.  NaN inputs have no code in the rule: the oracle gives 0x7F, the test
accepts either E4M3 NaN (0x7F, 0xFF) from the conversion."""
import numpy as np
import pytest
import torch

import block_wise_fp8_gb300 as fb
import oracle

pytestmark = pytest.mark.gpu

CHUNK = 1 << 28


def _is_nan(first, idx):
    """Whether bit patterns first + idx are binary32 NaNs."""
    bits = (np.uint64(first) + idx.astype(np.uint64)).astype(np.uint32)
    return ((bits & 0x7F800000) == 0x7F800000) & ((bits & 0x007FFFFF) != 0)


def test_conversion_of_every_binary32_pattern():
    codes = torch.empty(CHUNK, dtype=torch.uint8, device="cuda")
    for c in range((1 << 32) // CHUNK):
        first = c * CHUNK
        fb.fp8bq_e4m3_from_bits(first, codes)
        got = codes.cpu().numpy()
        ref = oracle.e4m3_encode_bits_range(first, CHUNK)
        idx = np.flatnonzero(got != ref)
        if idx.size:
            nan = _is_nan(first, idx)
            assert np.all((got[idx[nan]] & 0x7F) == 0x7F), "a NaN input gave a finite code"
            bad = idx[~nan]
            assert bad.size == 0, (f"{bad.size} codes differ in chunk {c}, first at bits "
                                   f"{first + int(bad[0]):#010x}: got {got[bad[0]]:#04x}, "
                                   f"oracle {ref[bad[0]]:#04x}")
        # NaN inputs that agree with the oracle's 0x7F need no check; the
        # others were accepted above only as E4M3 NaN codes


def test_ragged_range_and_end_of_range():
    """A count that is not a multiple of 8 and the last patterns below 2^32."""
    for first, n in ((0x43DF_FFF0, 37), ((1 << 32) - 13, 13), (0, 1)):
        codes = torch.full((n,), 0x55, dtype=torch.uint8, device="cuda")
        fb.fp8bq_e4m3_from_bits(first, codes)
        got = codes.cpu().numpy()
        ref = oracle.e4m3_encode_bits_range(first, n)
        nan = _is_nan(first, np.arange(n))
        assert np.array_equal(got[~nan], ref[~nan])
        assert np.all((got[nan] & 0x7F) == 0x7F)


def test_range_past_the_last_pattern_is_rejected():
    codes = torch.empty(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(fb.Fp8bqError) as e:
        fb.fp8bq_e4m3_from_bits((1 << 32) - 8, codes)
    assert e.value.name == "FP8BQ_ERR_SHAPE"
