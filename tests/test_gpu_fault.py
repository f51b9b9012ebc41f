"""Failure detection on the GPU without a GPU fault: every device-side wait of
the GEMM kernels is bounded, and a wait that runs out is reported through the
workspace status word while the kernel exits cleanly.

The failure is made on purpose in a child process: FP8BQ_FAULT_INJECT makes CTA
0 of the next few GEMM launches skip the copy of its first K block, so the MMA
issuer's wait on that stage (and every wait behind it) runs out after
FP8BQ_WAIT_LIMIT_MS = 50 ms.  Each kernel form is hit once -- split-K decode
tiles (16 and 64 tokens), the one-launch decode linear (its quantiser warps
wait on the stage too), 2-CTA prefill tiles (with split tail tiles),
per-tensor pair tiles, MXFP8 tiles, grouped single-CTA and pair tiles -- and
each must report FP8BQ_ERR_TIMEOUT.  After that the same process must still be able to
use the GPU: the next GEMMs, on freshly zeroed workspaces, match the oracle."""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r"""
import json, sys
import numpy as np
import torch
import block_wise_fp8_gb300 as fb
import oracle
import synthetic_inputs as si
from gpu_util import check_close, dev, host

torch.manual_seed(0)
codes = lambda r, c: torch.randint(0, 0x7E, (r, c), dtype=torch.uint8, device="cuda")
res = {}

def block(M, N, K):
    q, w = codes(M, K), codes(N, K)
    sx = torch.rand(M, K // 128, device="cuda") + 0.5
    sw = torch.rand(-(-N // 128), K // 128, device="cuda") + 0.5
    y = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    ws = fb.new_workspace(fb.OP_GEMM, M, N, K)
    fb.fp8bq_gemm(q, sx, w, sw, y, ws)
    return fb.fp8bq_poll_status(ws)

def static(M, N, K):
    q, w = codes(M, K), codes(N, K)
    sx = torch.ones(1, device="cuda")
    sp = torch.ones(2, device="cuda")
    y = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    ws = fb.new_workspace(fb.OP_STATIC_GEMM, M, N, K)
    fb.fp8bq_static_gemm(q, sx, w, sp, [N // 2, N - N // 2], y, ws)
    return fb.fp8bq_poll_status(ws)

def mx(M, N, K):
    q, w = codes(M, K), codes(N, K)
    ux = torch.full((M, K // 32), 127, dtype=torch.uint8, device="cuda")
    uw = torch.full((N, K // 32), 127, dtype=torch.uint8, device="cuda")
    y = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    ws = fb.new_workspace(fb.OP_MX_GEMM, M, N, K)
    fb.fp8bq_mx_gemm(q, ux, w, uw, y, ws)
    return fb.fp8bq_poll_status(ws)

def linear(M, N, K):
    x = torch.randn(M, K, device="cuda").to(torch.bfloat16)
    w = codes(N, K)
    sw = torch.rand(-(-N // 128), K // 128, device="cuda") + 0.5
    y = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    ws = fb.new_workspace(fb.OP_LINEAR, M, N, K)
    fb.fp8bq_linear(x, w, sw, y, ws)
    return fb.fp8bq_poll_status(ws)

def grouped(N, K, counts):
    E, T = len(counts), sum(counts)
    q, w = codes(T, K), codes(E * N, K).view(E, N, K)
    sx = torch.rand(T, K // 128, device="cuda") + 0.5
    sw = torch.rand(E, -(-N // 128), K // 128, device="cuda") + 0.5
    off = torch.tensor(np.concatenate([[0], np.cumsum(counts)]).astype(np.int32), device="cuda")
    y = torch.empty(T, N, dtype=torch.bfloat16, device="cuda")
    ws = fb.new_workspace(fb.OP_GROUPED_GEMM, T, N, K)
    fb.fp8bq_grouped_gemm(q, sx, w, sw, off, y, ws)
    return fb.fp8bq_poll_status(ws)

# eight injected launches, one per kernel form
res["decode_block"] = block(8, 1024, 2048)
res["decode_block_64"] = block(64, 1024, 2048)
res["decode_linear_fused"] = linear(4, 1024, 2048)
res["prefill_block_pair"] = block(512, 768, 2048)
res["static_pair"] = static(512, 1024, 1024)
res["mx"] = mx(256, 512, 1024)
res["grouped_normal"] = grouped(512, 1024, [100, 200, 12, 200])
res["grouped_pair"] = grouped(512, 1024, [1100, 1000])
torch.cuda.synchronize()

# the injection is spent: the context must still work and give correct results
for M, N, K in [(8, 1024, 2048), (300, 704, 1040)]:
    x = si.activations(M, K, base_seed=11)
    qa, sa = oracle.quant_group(x)
    qw, sw = oracle.quant_weight_block(si.weights(N, K, base_seed=11))
    y = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    ws = fb.new_workspace(fb.OP_GEMM, M, N, K)
    fb.fp8bq_gemm(dev(qa), dev(sa), dev(qw), dev(sw), y, ws)
    res[f"after_{M}x{N}x{K}"] = fb.fp8bq_poll_status(ws)
    check_close(host(y), oracle.gemm_block(qa, sa, qw, sw), f"after timeout {M}x{N}x{K}")
print("RESULT " + json.dumps(res))
"""


def test_bounded_waits_report_timeout_and_leave_the_context_usable():
    env = dict(os.environ)
    env["FP8BQ_FAULT_INJECT"] = "skip_first_load:8"
    env["FP8BQ_WAIT_LIMIT_MS"] = "50"
    env["PYTHONPATH"] = os.pathsep.join([ROOT, os.path.join(ROOT, "tests"),
                                         env.get("PYTHONPATH", "")])
    p = subprocess.run([sys.executable, "-c", CHILD], cwd=ROOT, env=env, capture_output=True,
                       text=True, timeout=300)
    assert p.returncode == 0, p.stdout[-2000:] + p.stderr[-4000:]
    line = [l for l in p.stdout.splitlines() if l.startswith("RESULT ")][-1]
    res = json.loads(line[len("RESULT "):])
    timeout = 8  # FP8BQ_ERR_TIMEOUT
    for k in ("decode_block", "decode_block_64", "decode_linear_fused", "prefill_block_pair",
              "static_pair", "mx", "grouped_normal", "grouped_pair"):
        assert res[k] == timeout, res
    assert res["after_8x1024x2048"] == 0 and res["after_300x704x1040"] == 0, res
