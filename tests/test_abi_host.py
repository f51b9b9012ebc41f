"""Host-side checks of the C ABI that need no GPU: the library loads, exports
every symbol include/fp8bq.h declares, and rejects bad arguments on the host
before any CUDA call (so these calls are safe on a machine without a GPU)."""
import ctypes
import os
import re

import pytest

import block_wise_fp8_gb300 as fb

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fp8bq.h")

# fake, suitably aligned device addresses: validation never dereferences them
A = 0x100000
P = ctypes.c_void_p


def declared_symbols():
    text = open(HEADER).read()
    return re.findall(r"FP8BQ_API\s+[\w\s\*]+?\b(fp8bq_\w+)\s*\(", text)


def test_library_exports_every_declared_symbol():
    names = declared_symbols()
    assert len(names) >= 17
    lib = ctypes.CDLL(fb.library_path())
    missing = [n for n in names if not hasattr(lib, n)]
    assert not missing, missing


def test_only_declared_symbols_are_exported():
    """The library's public surface is exactly the header (hidden visibility)."""
    import subprocess
    out = subprocess.run(["nm", "-D", "--defined-only", fb.library_path()],
                         capture_output=True, text=True, check=True).stdout
    exported = {l.split()[-1] for l in out.splitlines() if " T " in l}
    ours = {s for s in exported if s.startswith("fp8bq_")}
    assert ours == set(declared_symbols())


def test_version_and_status_strings():
    assert fb.fp8bq_version() == 10000
    for s in range(10):
        assert fb.fp8bq_status_string(s) != "unknown status"
    assert fb.fp8bq_status_string(99) == "unknown status"
    assert fb.fp8bq_last_cuda_error() == 0


def test_workspace_bytes():
    small = fb.fp8bq_workspace_bytes(fb.OP_GEMM, 4096, 6144, 6144)
    assert small % 256 == 0 and small >= 256
    # decode shapes reserve split-K partials; the fused linear also holds Q and scales
    dec = fb.fp8bq_workspace_bytes(fb.OP_GEMM, 64, 6144, 6144)
    lin = fb.fp8bq_workspace_bytes(fb.OP_LINEAR, 64, 6144, 6144)
    assert dec >= 8 * 64 * 6144 * 4
    assert lin >= dec + 64 * 6144 + 48 * 64 * 4
    assert fb.fp8bq_workspace_bytes(99, 1, 1, 1) == 256
    # block GEMM and linear above 64 rows: room for the split tail tiles'
    # partials (at most 4 K ranges of 256 KB per pair tile of 256 x 192 or
    # wider, 80 in all)
    big = fb.fp8bq_workspace_bytes(fb.OP_GEMM, 4096, 6144, 6144)
    assert big >= 80 * 256 * 1024
    assert fb.fp8bq_workspace_bytes(fb.OP_GEMM, 256, 512, 2048) >= 12 * 256 * 1024
    assert fb.fp8bq_workspace_bytes(fb.OP_GEMM, 256, 512, 2048) < 13 * 256 * 1024
    assert fb.fp8bq_workspace_bytes(fb.OP_GEMM, 300, 1000, 6016) >= 48 * 256 * 1024
    assert fb.fp8bq_workspace_bytes(fb.OP_LINEAR, 4096, 6144, 6144) >= big + 4096 * 6144
    # other GEMMs keep no such partials
    assert fb.fp8bq_workspace_bytes(fb.OP_CHANNEL_GEMM, 4096, 6144, 6144) < 1024 * 1024
    assert fb.fp8bq_workspace_bytes(fb.OP_GROUPED_GEMM, 4096, 6144, 6144) < 1024 * 1024


L = fb._lib


def test_quant_act_validation():
    ok = dict(x=P(A), M=16, K=256, ldx=256, q=P(A), s=P(A), lay=0, st=None)
    call = lambda d: L.fp8bq_quant_act(d["x"], d["M"], d["K"], d["ldx"], d["q"], d["s"],
                                       d["lay"], d["st"])
    assert call({**ok, "x": None}) == 1
    assert call({**ok, "q": None}) == 1
    assert call({**ok, "M": -1}) == 2
    assert call({**ok, "K": 0}) == 2
    assert call({**ok, "ldx": 128}) == 2
    assert call({**ok, "K": 200, "ldx": 200}) == 3      # K % 16
    assert call({**ok, "ldx": 260}) == 3                # pitch % 8
    assert call({**ok, "x": P(A + 8)}) == 3             # 16-byte alignment
    assert call({**ok, "lay": 2}) == 4
    assert call({**ok, "M": 0}) == 0                    # empty batch: no launch


def test_gemm_validation():
    def call(q=P(A), sx=P(A), lay=0, w=P(A), sw=P(A), bias=None, y=P(A), M=16, N=384,
             K=256, ws=P(A), wsb=1 << 20):
        return L.fp8bq_gemm(q, sx, lay, w, sw, bias, y, M, N, K, ws, wsb, None)
    assert call(w=None) == 1
    assert call(N=0) == 2
    assert call(K=100) == 3
    assert call(lay=5) == 4
    assert call(bias=P(A + 1)) == 3
    assert call(ws=None) == 6
    assert call(wsb=16) == 6
    assert call(ws=P(A + 16)) == 3
    assert call(M=0) == 0


def test_gemm_noalloc_validation():
    def call(q=P(A), lay=0, w=P(A), bias=None, M=16, N=384, K=256):
        return L.fp8bq_gemm_noalloc(q, P(A), lay, w, P(A), bias, P(A), M, N, K, None)
    assert call(q=None) == 1
    assert call(K=100) == 3
    assert call(lay=2) == 4
    assert call(bias=P(A + 1)) == 3
    assert call(M=64, N=24576, K=6144) == 6      # split-K partials exceed the scratch
    assert call(M=0) == 0


def test_mx_and_static_validation():
    assert L.fp8bq_mx_quant_act(P(A), 4, 48, 48, P(A), P(A), None) == 3    # K % 32
    assert L.fp8bq_mx_gemm(P(A), P(A), P(A), P(A), None, P(A), 4, 64, 80, P(A), 1 << 20,
                           None) == 3
    parts = (ctypes.c_int64 * 3)(100, 100, 56)
    call = lambda n, N=256, p=parts: L.fp8bq_static_gemm(P(A), P(A), P(A), P(A), p, n, None,
                                                         P(A), 4, N, 128, P(A), 1 << 20, None)
    assert call(3, N=300) == 2           # partitions must sum to N
    assert call(0) == 2
    assert call(65) == 2
    assert call(3, p=None) == 1
    bad = (ctypes.c_int64 * 3)(100, 0, 156)
    assert call(3, p=bad) == 2
    assert L.fp8bq_static_quant_act(P(A), 4, 128, 128, None, P(A), None) == 1


def test_poll_and_init_validation():
    assert L.fp8bq_poll_status(None, None) == 1
    assert L.fp8bq_workspace_init(P(A + 64), 256, None) == 3


def test_binding_fails_loudly_without_library(tmp_path, monkeypatch):
    """The package refuses to import when the CUDA library is missing."""
    import importlib
    import sys
    from block_wise_fp8_gb300 import _build
    monkeypatch.setattr(_build, "LIB", str(tmp_path / "missing.so"))
    saved = sys.modules.pop("block_wise_fp8_gb300")
    try:
        with pytest.raises(ImportError):
            importlib.import_module("block_wise_fp8_gb300")
    finally:
        sys.modules["block_wise_fp8_gb300"] = saved


def test_grouped_gemm_validation():
    """Both grouped forms reject bad arguments before any CUDA call."""
    ws_small = 256
    ok = dict(q=P(A), sx=P(A), lay=0, w=P(A), sw=P(A), off=P(A), E=4, y=P(A), M=512, N=256,
              K=256, ws=P(A), wsb=1 << 20, st=None)
    call = lambda d: L.fp8bq_grouped_gemm(d["q"], d["sx"], d["lay"], d["w"], d["sw"], d["off"],
                                          d["E"], d["y"], d["M"], d["N"], d["K"], d["ws"],
                                          d["wsb"], d["st"])
    assert call({**ok, "off": None}) == 1
    assert call({**ok, "w": None}) == 1
    assert call({**ok, "E": 0}) == 2
    assert call({**ok, "E": 1025}) == 2
    assert call({**ok, "E": 1 << 20, "N": 1 << 12}) == 2
    assert call({**ok, "K": 200}) == 3
    assert call({**ok, "off": P(A + 2)}) == 3
    assert call({**ok, "y": P(A + 8)}) == 3
    assert call({**ok, "lay": 5}) == 4
    assert call({**ok, "wsb": ws_small - 1}) == 6
    assert call({**ok, "ws": None}) == 6
    assert call({**ok, "M": 0}) == 0                     # nothing to compute
    assert fb.fp8bq_workspace_bytes(fb.OP_GROUPED_GEMM, 512, 256, 256) <= 1 << 20
    # no split-K partials at small row counts: the grouped form always uses pair tiles
    assert fb.fp8bq_workspace_bytes(fb.OP_GROUPED_GEMM, 8, 6144, 6144) < 8 * 6144 * 4

    okm = dict(q=P(A), sx=P(A), lay=0, w=P(A), sw=P(A), mm=P(A), E=4, max_m=128, y=P(A), N=256,
               K=256, ws=P(A), wsb=1 << 20, st=None)
    callm = lambda d: L.fp8bq_grouped_gemm_masked(d["q"], d["sx"], d["lay"], d["w"], d["sw"],
                                                  d["mm"], d["E"], d["max_m"], d["y"], d["N"],
                                                  d["K"], d["ws"], d["wsb"], d["st"])
    assert callm({**okm, "mm": None}) == 1
    assert callm({**okm, "max_m": -1}) == 2
    assert callm({**okm, "E": 2000}) == 2
    assert callm({**okm, "E": 2, "max_m": 1 << 31}) == 2   # E * max_m overflows 32 bits
    assert callm({**okm, "max_m": 0}) == 0


def test_check_scales_validation():
    import ctypes as C
    counts = (C.c_int64 * 3)(7, 7, 7)
    first = C.c_int64(7)
    cp, fp = C.c_void_p(C.addressof(counts)), C.c_void_p(C.addressof(first))
    f = L.fp8bq_check_scales
    assert f(P(A), 16, P(A), None, fp, None) == 1
    assert f(P(A), 16, P(A), cp, None, None) == 1
    assert f(None, 16, P(A), cp, fp, None) == 1
    assert f(P(A), 16, None, cp, fp, None) == 1
    assert f(P(A), -1, P(A), cp, fp, None) == 2
    assert f(P(A + 2), 16, P(A), cp, fp, None) == 3
    assert f(P(A), 16, P(A + 4), cp, fp, None) == 3
    # an empty array: nothing is bad, nothing is launched
    assert f(None, 0, None, cp, fp, None) == 0
    assert list(counts) == [0, 0, 0] and first.value == -1


def test_grouped_binding_rejects_host_bounds():
    """The segment bounds are read on the device: the binding refuses host tensors."""
    import torch
    q = torch.empty(0, dtype=torch.uint8)
    with pytest.raises(ValueError):
        fb.fp8bq_grouped_gemm(q.view(0, 16), None, torch.empty(2, 16, 16, dtype=torch.uint8), None,
                              torch.zeros(3, dtype=torch.int32), None, None)
    with pytest.raises(ValueError):
        fb.fp8bq_grouped_gemm_masked(q, None, torch.empty(2, 16, 16, dtype=torch.uint8), None,
                                     torch.zeros(2, dtype=torch.int32), None, None)
