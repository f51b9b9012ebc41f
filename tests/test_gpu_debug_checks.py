"""The debug build of the library: the GEMM epilogues check every global write
(Y rows and columns, the workspace's partial region) against its buffer, skip
a write outside and report FP8BQ_ERR_BOUNDS through the workspace status word
-- the device-side counterpart of the canary bands of the other tests.

A process loads one build, so the debug build runs in a child process
(FP8BQ_LIBRARY points the binding at it).  Every GEMM form runs on ragged
shapes: decode split-K tiles (16, 32 and 64 tokens), the one-launch decode
linear, 2-CTA prefill tiles with split tail tiles (one wave or several),
grouped segments that end
inside tiles, MXFP8, per-tensor and channelwise tiles.  No check may fire
and every output must match the oracle."""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r"""
import json, os
import numpy as np
import torch
import block_wise_fp8_gb300 as fb
import oracle
import synthetic_inputs as si
from gpu_util import check_close, dev, host

assert fb.library_path() == os.environ["FP8BQ_LIBRARY"]
res = {}

def block(M, N, K, linear=False):
    x = si.activations(M, K, base_seed=M)
    qa, sa = oracle.quant_group(x)
    qw, sw = oracle.quant_weight_block(si.weights(N, K, base_seed=N))
    y = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    if linear:
        ws = fb.new_workspace(fb.OP_LINEAR, M, N, K)
        fb.fp8bq_linear(dev(x), dev(qw), dev(sw), y, ws)
    else:
        ws = fb.new_workspace(fb.OP_GEMM, M, N, K)
        fb.fp8bq_gemm(dev(qa), dev(sa), dev(qw), dev(sw), y, ws)
    st = fb.fp8bq_poll_status(ws)
    check_close(host(y), oracle.gemm_block(qa, sa, qw, sw), f"block {M}x{N}x{K}")
    return st

for M in (1, 20, 64):
    res[f"decode_{M}"] = block(M, 1000, 2048)
res["linear_5"] = block(5, 1000, 1040, linear=True)
res["prefill_split_tail"] = block(300, 1000, 6016)
res["prefill_ragged"] = block(257, 300, 512)
res["prefill_waves"] = block(1200, 3400, 1040)

counts, N, K = [300, 1, 0, 513], 384, 512
T = sum(counts) + 2
off = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
qa, sa = oracle.quant_group(si.activations(T, K, base_seed=3))
sets = [oracle.quant_weight_block(si.weights(N, K, base_seed=e)) for e in range(4)]
qw = np.stack([q for q, _ in sets]); sw = np.stack([s for _, s in sets])
y = torch.full((T, N), float("nan"), dtype=torch.bfloat16, device="cuda")
ws = fb.new_workspace(fb.OP_GROUPED_GEMM, T, N, K)
fb.fp8bq_grouped_gemm(dev(qa), dev(sa), dev(qw), dev(sw), torch.tensor(off, device="cuda"), y, ws)
res["grouped"] = fb.fp8bq_poll_status(ws)
re = oracle.row_expert_contiguous(off, T)
on = re >= 0
check_close(host(y)[on], oracle.gemm_grouped(qa, sa, qw, sw, re)[on], "grouped")

M, N, K = 257, 300, 416
qa, ua = oracle.quant_mx(si.activations(M, K))
qw, uw = oracle.quant_mx(si.weights(N, K))
y = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
ws = fb.new_workspace(fb.OP_MX_GEMM, M, N, K)
fb.fp8bq_mx_gemm(dev(qa), dev(ua), dev(qw), dev(uw), y, ws)
res["mx"] = fb.fp8bq_poll_status(ws)
check_close(host(y), oracle.gemm_mx(qa, ua, qw, uw), "mx")

for M in (3, 150):
    N, K, parts = 200, 208, [72, 128]
    qw, sp = oracle.quant_weight_static(si.weights(N, K), parts)
    s_x = oracle.absmax_scale(si.calibration(32, K))
    qa = oracle.quant_static(si.activations(M, K), s_x)
    y = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    ws = fb.new_workspace(fb.OP_STATIC_GEMM, M, N, K)
    fb.fp8bq_static_gemm(dev(qa), torch.tensor([s_x], dtype=torch.float32, device="cuda"),
                         dev(qw), dev(sp), parts, y, ws)
    res[f"static_{M}"] = fb.fp8bq_poll_status(ws)
    check_close(host(y), oracle.gemm_static(qa, s_x, qw, sp, parts), f"static {M}")

for M in (5, 130):
    N, K = 300, 512
    qa, sa = oracle.quant_channel(si.activations(M, K))
    qw, sw = oracle.quant_channel(si.weights(N, K))
    y = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    ws = fb.new_workspace(fb.OP_CHANNEL_GEMM, M, N, K)
    fb.fp8bq_channel_gemm(dev(qa), dev(sa), dev(qw), dev(sw), y, ws)
    res[f"channel_{M}"] = fb.fp8bq_poll_status(ws)
    check_close(host(y), oracle.gemm_channel(qa, sa, qw, sw), f"channel {M}")
print("RESULT " + json.dumps(res))
"""


def test_debug_build_checks_every_epilogue_write():
    sys.path.insert(0, os.path.join(ROOT, "block_wise_fp8_gb300"))
    try:
        import _build
        lib = _build.build(debug=True)
    finally:
        sys.path.pop(0)
    env = dict(os.environ)
    env["FP8BQ_LIBRARY"] = lib
    env["PYTHONPATH"] = os.pathsep.join([ROOT, os.path.join(ROOT, "tests"),
                                         env.get("PYTHONPATH", "")])
    p = subprocess.run([sys.executable, "-c", CHILD], cwd=ROOT, env=env, capture_output=True,
                       text=True, timeout=900)
    assert p.returncode == 0, p.stdout[-2000:] + p.stderr[-4000:]
    res = json.loads([l for l in p.stdout.splitlines() if l.startswith("RESULT ")][-1][7:])
    assert res and all(v == 0 for v in res.values()), res
