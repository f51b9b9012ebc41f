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


def sample_indices(M, N, seed=0, per_block=4, block=128):
    """Output coordinates that cover every block x block tile of an M x N
    output: each tile's four corners (clipped to the matrix) and `per_block`
    random elements inside it.  Every 128 x 128 promotion block -- and so every
    tile of every kernel form, whose tiles are unions of such blocks -- has
    checked elements, including the ragged last row and column of tiles."""
    rng = np.random.default_rng(seed)
    rows, cols = [], []
    for r0 in range(0, M, block):
        r1 = min(M, r0 + block) - 1
        for c0 in range(0, N, block):
            c1 = min(N, c0 + block) - 1
            rows += [r0, r0, r1, r1]
            cols += [c0, c1, c0, c1]
            rows += list(rng.integers(r0, r1 + 1, per_block))
            cols += list(rng.integers(c0, c1 + 1, per_block))
    return np.asarray(rows, np.int64), np.asarray(cols, np.int64)


def assert_covers_every_block(rows, cols, M, N, block=128):
    """Every block x block tile of the output holds at least one sample."""
    hit = np.zeros((-(-M // block), -(-N // block)), bool)
    hit[rows // block, cols // block] = True
    assert hit.all(), f"{(~hit).sum()} output blocks without a checked element"


# ------------------------------------------------------------ guard bands
#
# compute-sanitizer is not available on the GPU pool, so writes past the end of
# an output are caught with canaries: the output is a view into the middle of a
# larger buffer whose bytes before and after it hold a known pattern, checked
# after the call.  The view starts on a 256-byte boundary, like an allocation.

GUARD_BYTES = 4096
CANARY = 0xA5


class Guarded:
    """An output tensor of `shape` and `dtype` with canary bands on both sides."""

    def __init__(self, shape, dtype, fill=None, device="cuda"):
        elem = torch.empty((), dtype=dtype).element_size()
        n = int(np.prod(shape)) if len(shape) else 1
        body = -(-n * elem // 256) * 256
        self.buf = torch.full((GUARD_BYTES + body + GUARD_BYTES,), CANARY, dtype=torch.uint8,
                              device=device)
        self.lo, self.hi = GUARD_BYTES, GUARD_BYTES + n * elem
        self.t = self.buf[self.lo:self.hi].view(dtype).view(shape)
        if fill is not None:
            self.t.fill_(fill)

    def check(self, what=""):
        b = self.buf.cpu().numpy()
        before, after = b[:self.lo], b[self.hi:]
        bad_b = np.flatnonzero(before != CANARY)
        bad_a = np.flatnonzero(after != CANARY)
        assert bad_b.size == 0, f"{what}: {bad_b.size} bytes written before the output"
        assert bad_a.size == 0, (f"{what}: {bad_a.size} bytes written past the end of the "
                                 f"output, first at +{bad_a[0]}")
