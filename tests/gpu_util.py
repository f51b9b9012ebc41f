"""Helpers shared by the GPU parity tests: host <-> device transfer of the
oracle's numpy arrays and the GEMM tolerance check."""
import numpy as np
import torch

# GEMM tolerance against the oracle's binary64 result on the same quantised
# inputs: per element |y - ref| <= 1e-2 * max(1, |ref|), and relative
# Frobenius error <= 4e-3.  BF16 output rounding alone is <= 2^-9 relative.
ELEM_TOL = 1e-2
FROB_TOL = 4e-3


def dev(a, dtype=None, device="cuda"):
    """numpy -> device tensor; uint16 arrays become bfloat16 (bit patterns)."""
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).to(device).view(torch.bfloat16)
    t = torch.from_numpy(a).to(device)
    return t if dtype is None else t.view(dtype)


def host(t):
    t = t.detach().cpu()
    if t.dtype == torch.bfloat16:
        return t.float().numpy().astype(np.float64)
    if t.dtype == torch.float8_e4m3fn:
        return t.view(torch.uint8).numpy()
    return t.numpy()


def check_close(y, ref, what=""):
    y = np.asarray(y, np.float64)
    ref = np.asarray(ref, np.float64)
    assert y.shape == ref.shape
    err = np.abs(y - ref)
    bound = ELEM_TOL * np.maximum(1.0, np.abs(ref))
    bad = np.argwhere(err > bound)
    assert bad.size == 0, (f"{what}: {len(bad)} elements out of tolerance, first "
                           f"{bad[:5].tolist()} y={y[tuple(bad[0])]} ref={ref[tuple(bad[0])]}")
    nref = np.linalg.norm(ref)
    if nref > 0:
        rel = np.linalg.norm(y - ref) / nref
        assert rel <= FROB_TOL, f"{what}: relative Frobenius error {rel}"
    assert np.all(np.isfinite(y))


def sample_indices(M, N, n, seed=0):
    """n (row, col) pairs covering the first/last rows and columns and random ones."""
    rng = np.random.default_rng(seed)
    rows = np.concatenate([[0, M - 1, 0, M - 1], rng.integers(0, M, n - 4)])
    cols = np.concatenate([[0, 0, N - 1, N - 1], rng.integers(0, N, n - 4)])
    return rows.astype(np.int64), cols.astype(np.int64)
