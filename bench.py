"""Benchmark of the block-wise FP8 linear on GB300 (one JSON line on stdout).

Workload (the prefill shape the headline metric is quoted on): BF16
activations X [4096, 6144] (N(0,1), 1% of channels x50) through the block-FP8
linear for both projection widths N = 6144 and N = 24576 (E4M3 weights with
FP32 128x128 scales, N(0, 0.02) before quantisation).  One step = activation
quantisation (group 128) + block-scaled GEMM for each width, i.e. the whole
forward of the two layers.  `value` is whole-job TFLOPS (2*M*K*N summed over
both widths and all ranks, divided by the slowest rank's summed step time).

Also reported, measured in the same run:
  roofline     the block GEMM kernel against the FP8 dense peak (2x the measured
               BF16 burst peak), with the ncu DRAM traffic of that kernel;
  e2e          the same metric through fp8bq_linear with host buffers, the
               pinned-host -> device copy of X and the device -> host copy of Y
               of every step inside the timed region (copies on two further
               streams, overlapping the kernels of neighbouring steps);
  extra        decode (M in {1,8,32,64}), quantiser and fused residual-add +
               RMSNorm + quantisation GB/s against HBM, MXFP8, static
               per-tensor, channelwise and block-with-UE8M0 TFLOPS, the
               grouped (MoE) GEMM against its HBM / FP8 roofline, and as
               context the vendor's plain per-tensor FP8 GEMM (cuBLASLt via
               torch._scaled_mm), which has no block scales to promote;
  cpu_baseline the CPU oracle on a bounded sample of the same workload.
`--profile-case <case>` runs only a few launches of one kernel (MXFP8, UE8M0,
channelwise, static and decode GEMMs, group-128 quantisation, norm +
quantisation, grouped w13 / w2) for ncu captures.

L2 is flushed (256 MiB write) between timed steps; every step is timed with
CUDA events on the launching stream, synchronised on both sides.

`--impl reference` times the CPU oracle itself on the host cores.
Multi-GPU: `torchrun --nproc-per-node N bench.py --gpus N`: every rank runs the
same per-GPU workload on its own GPU (independent token batches, no
collective on the data path: weak scaling); rank 0 prints the line.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synthetic_inputs as si  # noqa: E402

METRIC = ("block-FP8 linear TFLOPS & % FP8 peak (prefill); "
          "GB/s & % HBM (quant, decode)")
PREFILL_M, PREFILL_K = si.PREFILL["M"], si.PREFILL["K"]
PREFILL_NS = si.PREFILL["N_list"]
FLUSH_BYTES = 256 << 20
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
FP8_PER_BF16 = 2.0   # nominal dense FP8 / BF16 tensor rate
ORACLE_ROWS = 8      # token rows of a large output that the CPU baseline recomputes

# DRAM traffic (dram__bytes_read.sum + dram__bytes_write.sum) of one prefill
# block-GEMM launch from an ncu capture, valid only for the kernel sources whose
# digest is recorded; anything else reports null.
NCU_TRAFFIC = {
    # profiles/block_gemm_prefill_4096x24576x6144.md (N = 24576 launch)
    "source_sha256": "4e3efad97d785c9e2e1e7e0d8b08b272b386ea2ce87892662fa9ba02e8abb606",
    "bytes_per_launch": 185408256 + 183538944,
}


def kernel_source_digest() -> str:
    """SHA-256 of the GEMM kernel sources with // comments and blank lines
    removed: any change to the code invalidates the recorded traffic, a change
    to the comments alone does not."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "block_wise_fp8_gb300", "csrc")
    for f in sorted(os.listdir(csrc)):
        if f.startswith("gemm") or f in ("ptx.cuh", "common.cuh"):
            with open(os.path.join(csrc, f), encoding="utf-8") as fh:
                code = [l.split("//", 1)[0].rstrip() for l in fh]
            h.update(f.encode() + "\n".join(l for l in code if l).encode())
    return h.hexdigest()


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return FALLBACK_PEAKS, "fallback"


# ---------------------------------------------------------------------------
# distributed plumbing (weak scaling, no data-path collective)
# ---------------------------------------------------------------------------

def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def aggregate(values, world_size, rank, reduce_max, device=None):
    """Max (time) or sum (units) of per-rank floats over all ranks."""
    if world_size == 1:
        return list(values)
    import torch
    import torch.distributed as dist
    t = torch.tensor(values, dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX if reduce_max else dist.ReduceOp.SUM)
    return t.tolist()


def barrier(world_size):
    if world_size > 1:
        import torch.distributed as dist
        dist.barrier()


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,utilization.gpu,"
              "clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.out = ""
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()

    def summary(self):
        rows = []
        for line in (self.out or "").strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 10:
                continue
            try:
                rows.append(dict(sm=float(parts[1]), smax=float(parts[2]),
                                 util=float(parts[4]), reasons=parts[6:10]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        load = [r for r in rows if r["util"] >= 50] or rows
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in load for i, v in enumerate(r["reasons"])
                          if v.lower() in ("active", "1", "yes")})
        return {"sm_mhz": statistics.median(r["sm"] for r in load),
                "sm_max_mhz": max(r["smax"] for r in load),
                "samples_under_load": len(load), "reasons": reasons}


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------

def pcts(v):
    """10th, 50th and 90th percentile of a list of times (ms)."""
    return [round(float(x), 4) for x in np.percentile(np.asarray(v, np.float64), [10, 50, 90])]


def run_ours(args):
    import torch
    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    import block_wise_fp8_gb300 as fb

    stream = torch.cuda.current_stream(dev)
    peaks, peak_src = load_peaks()
    hbm_peak = peaks["hbm_gbs"]
    # FP8 dense peak: the larger of 2 x the measured BF16 burst rate (the
    # nominal FP8 / BF16 ratio) and the vendor's plain FP8 GEMM measured here at
    # 8192^3 -- the larger denominator keeps every fraction conservative
    nominal = peaks["bf16_tflops"] * FP8_PER_BF16
    vendor = vendor_fp8_reference(torch, dev, stream)
    v8192 = vendor.get("square_8192", {}).get("tflops")
    fp8_peak = max(nominal, v8192 or 0.0)
    fp8_src = (f"same-run cuBLASLt FP8 GEMM 8192^3 ({v8192} TFLOP/s)" if v8192 and v8192 > nominal
               else f"{peak_src}: 2 x bf16 burst {peaks['bf16_tflops']} TFLOP/s")
    for k in ("prefill_4096x24576x6144", "square_8192"):
        if k in vendor:
            vendor[k]["frac_fp8"] = round(vendor[k]["tflops"] / fp8_peak, 4)

    def to_dev(bits):
        return torch.from_numpy(bits.view(np.int16)).to(dev).view(torch.bfloat16)

    # ---- inputs (seeded, synthetic), weights quantised on the device by the
    # library's own 128x128 block quantiser
    M, K = PREFILL_M, PREFILL_K
    x = to_dev(si.activations(M, K))
    layers = []
    for N in PREFILL_NS:
        wb = to_dev(si.weights(N, K))
        qw = torch.empty(N, K, dtype=torch.uint8, device=dev)
        sw = torch.empty(-(-N // 128), -(-K // 128), dtype=torch.float32, device=dev)
        fb.fp8bq_quant_weight_block(wb, qw, sw)
        del wb
        y = torch.empty(M, N, dtype=torch.bfloat16, device=dev)
        ws = fb.new_workspace(fb.OP_GEMM, M, N, K, device=dev)
        layers.append(dict(N=N, qw=qw, sw=sw, y=y, ws=ws))
    q = torch.empty(M, K, dtype=torch.uint8, device=dev)
    sx = torch.empty(M, -(-K // 128), dtype=torch.float32, device=dev)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    flops_step = sum(2.0 * M * K * L["N"] for L in layers)

    nv = torch.cuda.nvtx

    def step(ev=None):
        # A1: group-128 activation quantisation (row-major scales)
        nv.range_push("quant_act 4096x6144")
        fb.fp8bq_quant_act(x, q, sx, fb.SCALE_ROW_MAJOR)
        nv.range_pop()
        for i, L in enumerate(layers):
            if ev is not None:
                ev[i][0].record(stream)
            # A2: block-scaled GEMM
            nv.range_push(f"block GEMM {M}x{L['N']}x{K}")
            fb.fp8bq_gemm(q, sx, L["qw"], L["sw"], L["y"], L["ws"],
                          s_layout=fb.SCALE_ROW_MAJOR)
            nv.range_pop()
            if ev is not None:
                ev[i][1].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    for L in layers:
        if fb.fp8bq_poll_status(L["ws"]) != 0:
            raise RuntimeError("device wait timed out during warm-up")

    # ---- timed region: exactly K steps, L2 flushed between them
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    gev = [[[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in layers]
           for _ in range(args.steps)]
    with ClockSampler(local) as clk:
        # keep the GPU busy ~1 s before the timed steps so clock samples see load
        t_end = time.time() + 1.0
        while time.time() < t_end:
            step()
            torch.cuda.synchronize()
        barrier(world)
        torch.cuda.synchronize()
        for i in range(args.steps):
            flush.zero_()
            starts[i].record(stream)
            step(gev[i])
            ends[i].record(stream)
        torch.cuda.synchronize()
        barrier(world)
    step_list = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    ms = sum(step_list)
    gemm_lists = [[gev[i][j][0].elapsed_time(gev[i][j][1]) for i in range(args.steps)]
                  for j in range(len(layers))]
    gemm_ms = [sum(g) / args.steps for g in gemm_lists]
    for L in layers:
        if fb.fp8bq_poll_status(L["ws"]) != 0:
            raise RuntimeError("device wait timed out in the timed region")
    ms_max, = aggregate([ms], world, rank, True, dev)
    value = flops_step * args.steps * world / (ms_max * 1e-3) / 1e12

    # ---- roofline of the dominant kernel: the block GEMM, N = 24576
    j = int(np.argmax([L["N"] for L in layers]))
    achieved = 2.0 * M * K * layers[j]["N"] / (gemm_ms[j] * 1e-3) / 1e12
    traffic = None
    if NCU_TRAFFIC["source_sha256"] == kernel_source_digest():
        traffic = NCU_TRAFFIC["bytes_per_launch"]
    roofline = {"bound": "tensor", "achieved": round(achieved, 1), "peak": round(fp8_peak, 1),
                "unit": "TFLOP/s", "frac": round(achieved / fp8_peak, 4), "traffic": traffic,
                "kernel": f"block-scaled GEMM {M}x{layers[j]['N']}x{K}",
                "peak_source": fp8_src,
                "peak_candidates": {"2x_bf16_burst": round(nominal, 1),
                                    "vendor_fp8_8192_cubed": v8192},
                "frac_of_2x_bf16_burst": round(achieved / nominal, 4),
                "gemm_ms": {str(L["N"]): round(t, 4) for L, t in zip(layers, gemm_ms)},
                "gemm_ms_p10_p50_p90": {str(L["N"]): pcts(g) for L, g in zip(layers, gemm_lists)}}

    # ---- e2e through fp8bq_linear with host buffers
    e2e = run_e2e(fb, torch, dev, stream, layers, x, args, world, rank)

    keep = {"prefill": {L["N"]: L["y"][:ORACLE_ROWS].cpu() for L in layers}}
    extra = run_extra(fb, torch, dev, stream, hbm_peak, fp8_peak, keep) if (
        rank == 0 and not args.no_extra) else {}
    extra["vendor_fp8_gemm"] = vendor
    cpu = cpu_baseline(args, keep) if (rank == 0 and not args.no_cpu) else None
    records = build_records(M, K, layers, gemm_lists, step_list, flops_step, extra, cpu,
                            hbm_peak, fp8_peak, achieved) if rank == 0 else []

    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "TFLOPS", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_max / args.steps, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "e4m3",
        "data": "synthetic (seeded splitmix64/Box-Muller; X ~ N(0,1) with 1% channels x50, "
                "W ~ N(0,0.02) quantised to E4M3 with 128x128 FP32 scales)",
        "config": {"workload": f"prefill block-FP8 linear: X[{M},{K}] BF16 -> N in "
                               f"{list(PREFILL_NS)}, BF16 out",
                   "step": "group-128 quant (row-major scales) + block-scaled GEMM per N",
                   "global_batch": M * world, "per_gpu_tokens": M,
                   "parallelism": f"replicas x{world} (independent token batches)",
                   "l2": "flushed between timed steps (256 MiB write)"},
        "roofline": roofline,
        "e2e": e2e,
        "step_ms_p10_p50_p90": pcts(step_list),
        "gpu_launches": 3 * args.steps,
        "clocks": clk.summary(),
        "records": records,
        "extra": extra,
        "cpu_baseline": cpu,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def run_e2e(fb, torch, dev, stream, layers, x, args, world, rank):
    """fp8bq_linear per width through the public API, with every step's input
    copied in from pinned host memory and every step's outputs copied back to
    pinned host memory inside the timed region.  Copies run on two further
    streams, one per direction (separate copy engines), and overlap the
    neighbouring steps' kernels, as a serving loop would: X and Y are
    double-buffered on the device and ordered by events (a copy starts when
    the kernel that writes its source has finished, and a buffer is rewritten
    only after the copy that reads it)."""
    M, K = x.shape
    copy_in = torch.cuda.Stream(dev)   # host -> device and device -> host run
    copy = torch.cuda.Stream(dev)      # on separate copy engines
    x_host = torch.empty(M, K, dtype=torch.bfloat16, pin_memory=True)
    x_host.copy_(x.cpu())
    x_dev = [torch.empty_like(x) for _ in range(2)]
    y_dev = [[torch.empty(M, L["N"], dtype=torch.bfloat16, device=dev) for L in layers]
             for _ in range(2)]
    y_host = [torch.empty(M, L["N"], dtype=torch.bfloat16, pin_memory=True) for L in layers]
    ws = [fb.new_workspace(fb.OP_LINEAR, M, L["N"], K, device=dev) for L in layers]
    ev = lambda: torch.cuda.Event()
    x_in = [ev() for _ in range(2)]                   # X copied in
    x_free = [ev() for _ in range(2)]                 # last kernel reading X done
    y_done = [[ev() for _ in layers] for _ in range(2)]  # Y written
    y_free = [[ev() for _ in layers] for _ in range(2)]  # Y copied out

    def step(i):
        p = i % 2
        copy_in.wait_event(x_free[p])
        with torch.cuda.stream(copy_in):
            x_dev[p].copy_(x_host, non_blocking=True)
        x_in[p].record(copy_in)
        stream.wait_event(x_in[p])
        for j, L in enumerate(layers):
            stream.wait_event(y_free[p][j])
            fb.fp8bq_linear(x_dev[p], L["qw"], L["sw"], y_dev[p][j], ws[j], stream=stream)
            y_done[p][j].record(stream)
            copy.wait_event(y_done[p][j])
            with torch.cuda.stream(copy):
                y_host[j].copy_(y_dev[p][j], non_blocking=True)
            y_free[p][j].record(copy)
        x_free[p].record(stream)

    for i in range(max(2, args.warmup)):
        step(i)
    torch.cuda.synchronize()
    steps = max(1, args.steps)
    s = torch.cuda.Event(enable_timing=True)
    e = torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    s.record(stream)
    for i in range(steps):
        step(i)
    stream.wait_stream(copy)     # the last step's copies are inside the timed region
    stream.wait_stream(copy_in)
    e.record(stream)
    torch.cuda.synchronize()
    ms = s.elapsed_time(e)
    ms_max, = aggregate([ms], world, rank, True, dev)
    flops = sum(2.0 * M * K * L["N"] for L in layers) * steps * world
    h2d = M * K * 2
    d2h = sum(M * L["N"] * 2 for L in layers)
    return {"value": round(flops / (ms_max * 1e-3) / 1e12, 2), "unit": "TFLOPS",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "ms_per_step": round(ms_max / steps, 4),
            "overlap": "host copies on two further streams (one per direction), overlapping "
                       "the neighbouring steps' kernels"}


class Timing(float):
    """Mean ms per launch (the float value) with the 10th / 50th / 90th
    percentiles of the per-launch times beside it."""

    def __new__(cls, mean_ms, samples_ms):
        t = super().__new__(cls, mean_ms)
        t.pct = pcts(samples_ms) if len(samples_ms) else [mean_ms] * 3
        return t

    def us_pct(self):
        return [round(v * 1e3, 2) for v in self.pct]


def _time_back_to_back(torch, stream, fns, reps):
    """Mean ms per launch of `reps` launches issued back to back, cycling through
    `fns` (one per independent copy of the inputs, so that together they exceed
    L2 and every launch streams its operands from HBM).  A second pass with an
    event pair around every launch gives the per-launch percentiles (events
    between launches stop dependent launches from overlapping, so the mean
    comes from the first pass)."""
    for f in fns:
        f()
    for _ in range(3):
        fns[0]()
    torch.cuda.synchronize()
    s = torch.cuda.Event(enable_timing=True)
    e = torch.cuda.Event(enable_timing=True)
    s.record(stream)
    for i in range(reps):
        fns[i % len(fns)]()
    e.record(stream)
    e.synchronize()
    mean = s.elapsed_time(e) / reps
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(reps + 1)]
    ev[0].record(stream)
    for i in range(reps):
        fns[i % len(fns)]()
        ev[i + 1].record(stream)
    ev[-1].synchronize()
    return Timing(mean, [ev[i].elapsed_time(ev[i + 1]) for i in range(reps)])


def _time_graph(torch, fns, per_graph, reps=20):
    """Mean ms per launch of `per_graph` launches (cycling through `fns`) captured
    back to back in one CUDA graph and replayed `reps` times: launches follow
    each other with no host in between, as in a captured decode step.  The
    percentiles are over the replays (each replay's time / per_graph)."""
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        for f in fns:
            f()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for i in range(per_graph):
            fns[i % len(fns)]()
    g.replay()
    torch.cuda.synchronize()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(reps + 1)]
    ev[0].record()
    for i in range(reps):
        g.replay()
        ev[i + 1].record()
    ev[-1].synchronize()
    per = [ev[i].elapsed_time(ev[i + 1]) / per_graph for i in range(reps)]
    return Timing(ev[0].elapsed_time(ev[-1]) / (reps * per_graph), per)


def _copies(t, n):
    return [t] + [t.clone() for _ in range(n - 1)]


def vendor_fp8_reference(torch, dev, stream):
    res = {"what": "torch._scaled_mm (cuBLASLt), E4M3 x E4M3, per-tensor FP32 scales, BF16 out"}
    try:
        for name, (M, N, K) in (("prefill_4096x24576x6144", (PREFILL_M, PREFILL_NS[1], PREFILL_K)),
                                ("square_8192", (8192, 8192, 8192))):
            a = torch.randint(0, 0x7E, (M, K), dtype=torch.uint8, device=dev).view(torch.float8_e4m3fn)
            b = torch.randint(0, 0x7E, (N, K), dtype=torch.uint8, device=dev).view(torch.float8_e4m3fn)
            one = torch.ones((), dtype=torch.float32, device=dev)
            f = lambda: torch._scaled_mm(a, b.t(), scale_a=one, scale_b=one, out_dtype=torch.bfloat16)
            t = _time_back_to_back(torch, stream, [f], 20)
            tf = 2.0 * M * N * K / (t * 1e-3) / 1e12
            res[name] = {"us": round(t * 1e3, 2), "tflops": round(tf, 1)}
            del a, b
    except Exception as e:  # noqa: BLE001 - context figure only
        res["unavailable"] = f"{type(e).__name__}: {str(e)[:160]}"
    return res


def run_extra(fb, torch, dev, stream, hbm_peak, fp8_peak, keep):
    """Decode, quantiser and fused residual-add + RMSNorm + quantisation GB/s,
    MXFP8 and static TFLOPS (informational).  Each
    figure is the mean over back-to-back launches rotating through enough input
    copies to exceed 1.5x the L2 size.  Launches shorter than the host's own
    cost per call (about 11 us through the Python binding) are timed inside a
    CUDA graph (`*_us`, used for the fractions); the eager figures
    (`*_eager_us`) are reported beside them.  `keep` receives host copies of
    the outputs of the workload configurations, for the oracle's check in the
    CPU baseline leg."""
    out = {}
    nv = torch.cuda.nvtx
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size

    def to_dev(bits):
        return torch.from_numpy(bits.view(np.int16)).to(dev).view(torch.bfloat16)

    def n_sets(bytes_per_set):
        return max(2, int(np.ceil(1.5 * l2 / bytes_per_set)))

    # decode GEMM and linear: weights streamed from HBM each launch
    K = N = si.DECODE["K"]
    wb = to_dev(si.weights(N, K))
    qw = torch.empty(N, K, dtype=torch.uint8, device=dev)
    sw = torch.empty(N // 128, K // 128, dtype=torch.float32, device=dev)
    fb.fp8bq_quant_weight_block(wb, qw, sw)
    del wb
    ns = n_sets(N * K)
    qws, sws = _copies(qw, ns), _copies(sw, ns)
    dec = {}
    keep["decode"] = {}
    nv.range_push("decode GEMM and linear 6144x6144")
    for M in si.DECODE["M_list"]:
        x = to_dev(si.activations(M, K))
        q = torch.empty(M, K, dtype=torch.uint8, device=dev)
        sx = torch.empty(M, K // 128, dtype=torch.float32, device=dev)
        fb.fp8bq_quant_act(x, q, sx)
        y = torch.empty(M, N, dtype=torch.bfloat16, device=dev)
        ws = fb.new_workspace(fb.OP_LINEAR, M, N, K, device=dev)
        g = [lambda i=i: fb.fp8bq_gemm(q, sx, qws[i], sws[i], y, ws) for i in range(ns)]
        l = [lambda i=i: fb.fp8bq_linear(x, qws[i], sws[i], y, ws) for i in range(ns)]
        te = _time_back_to_back(torch, stream, g, 60)
        tle = _time_back_to_back(torch, stream, l, 60)
        t = _time_graph(torch, g, 2 * ns)
        tl = _time_graph(torch, l, 2 * ns)
        g[0]()
        keep["decode"][M] = y.cpu()
        gemm_bytes = N * K + sw.numel() * 4 + M * (K + K // 128 * 4) + 2 * M * N
        lin_bytes = N * K + sw.numel() * 4 + 2 * M * K + 2 * M * N
        dec[str(M)] = {"gemm_us": round(t * 1e3, 2), "gemm_us_p10_p50_p90": t.us_pct(),
                       "linear_us_p10_p50_p90": tl.us_pct(),
                       "gemm_gbs": round(gemm_bytes / (t * 1e-3) / 1e9, 1),
                       "gemm_frac_hbm": round(gemm_bytes / (t * 1e-3) / 1e9 / hbm_peak, 4),
                       "gemm_eager_us": round(te * 1e3, 2),
                       "linear_us": round(tl * 1e3, 2),
                       "linear_gbs": round(lin_bytes / (tl * 1e-3) / 1e9, 1),
                       "linear_frac_hbm": round(lin_bytes / (tl * 1e-3) / 1e9 / hbm_peak, 4),
                       "linear_eager_us": round(tle * 1e3, 2)}
    out["decode_N6144_K6144"] = dec
    nv.range_pop()
    del qw, sw, qws, sws

    # quantisers at the workload shapes
    quant = {}
    nv.range_push("quantisers")
    M, K = 4096, 6144
    b = M * K * 2 + M * K + M * (K // 128) * 4
    ns = n_sets(b)
    xs = _copies(to_dev(si.activations(M, K)), ns)
    qs = [torch.empty(M, K, dtype=torch.uint8, device=dev) for _ in range(ns)]
    ss = [torch.empty(M, K // 128, dtype=torch.float32, device=dev) for _ in range(ns)]
    t = _time_graph(torch, [lambda i=i: fb.fp8bq_quant_act(xs[i], qs[i], ss[i])
                            for i in range(ns)], 2 * ns)
    quant["group128_4096x6144"] = {"us": round(t * 1e3, 2), "us_p10_p50_p90": t.us_pct(),
                                   "gbs": round(b / (t * 1e-3) / 1e9, 1),
                                   "frac_hbm": round(b / (t * 1e-3) / 1e9 / hbm_peak, 4)}
    keep["quant_group"] = (qs[0].cpu(), ss[0].cpu())
    del xs, qs, ss
    M, K = si.MXFP8["M"], si.MXFP8["K"]
    b = M * K * 3 + M * K // 32
    ns = n_sets(b)
    xm = to_dev(si.activations(M, K))
    xms = _copies(xm, ns)
    qms = [torch.empty(M, K, dtype=torch.uint8, device=dev) for _ in range(ns)]
    ums = [torch.empty(M, K // 32, dtype=torch.uint8, device=dev) for _ in range(ns)]
    t = _time_graph(torch, [lambda i=i: fb.fp8bq_mx_quant_act(xms[i], qms[i], ums[i])
                            for i in range(ns)], 2 * ns)
    quant["mx_2048x7168"] = {"us": round(t * 1e3, 2), "us_p10_p50_p90": t.us_pct(),
                             "gbs": round(b / (t * 1e-3) / 1e9, 1),
                             "frac_hbm": round(b / (t * 1e-3) / 1e9 / hbm_peak, 4)}
    keep["quant_mx"] = (qms[0].cpu(), ums[0].cpu())
    out["quant"] = quant
    nv.range_pop()
    qm, um = qms[0], ums[0]
    del xms

    # MXFP8 GEMM 2048 x 4096 x 7168
    N = si.MXFP8["N"]
    wb = to_dev(si.weights(N, K))
    qwm = torch.empty(N, K, dtype=torch.uint8, device=dev)
    uwm = torch.empty(N, K // 32, dtype=torch.uint8, device=dev)
    fb.fp8bq_mx_quant_act(wb, qwm, uwm)
    del wb
    ym = torch.empty(M, N, dtype=torch.bfloat16, device=dev)
    wsm = fb.new_workspace(fb.OP_MX_GEMM, M, N, K, device=dev)
    nv.range_push("MXFP8 GEMM 2048x4096x7168")
    t = _time_back_to_back(torch, stream, [lambda: fb.fp8bq_mx_gemm(qm, um, qwm, uwm, ym, wsm)], 30)
    nv.range_pop()
    keep["mx_gemm"] = ym[:ORACLE_ROWS].cpu()
    tf = 2.0 * M * N * K / (t * 1e-3) / 1e12
    out["mx_gemm_2048x4096x7168"] = {"us": round(t * 1e3, 2), "us_p10_p50_p90": t.us_pct(),
                                     "tflops": round(tf, 1), "frac_fp8": round(tf / fp8_peak, 4)}
    del qwm, uwm

    # static per-tensor GEMM, N = 14336 (4096/4096/6144), K = 4096
    K, N, parts = si.STATIC["K"], si.STATIC["N"], si.STATIC["parts"]
    wb = to_dev(si.weights(N, K))
    qws = torch.empty(N, K, dtype=torch.uint8, device=dev)
    sp = torch.empty(len(parts), dtype=torch.float32, device=dev)
    r0 = 0
    for p, n in enumerate(parts):
        fb.fp8bq_absmax_scale(wb[r0:r0 + n], sp[p:p + 1])
        fb.fp8bq_static_quant_act(wb[r0:r0 + n], sp[p:p + 1], qws[r0:r0 + n])
        r0 += n
    del wb
    ns = n_sets(N * K)
    qwss = _copies(qws, ns)
    s_x = torch.empty(1, dtype=torch.float32, device=dev)
    fb.fp8bq_absmax_scale(to_dev(si.calibration(si.STATIC["calib_rows"], K)), s_x)
    st = {}
    keep["static"] = {}
    nv.range_push("static per-tensor GEMM N=14336")
    for M in si.STATIC["M_list"]:
        xs = to_dev(si.activations(M, K, outliers=False))
        qs = torch.empty(M, K, dtype=torch.uint8, device=dev)
        fb.fp8bq_static_quant_act(xs, s_x, qs)
        ys = torch.empty(M, N, dtype=torch.bfloat16, device=dev)
        wss = fb.new_workspace(fb.OP_STATIC_GEMM, M, N, K, device=dev)
        t = _time_graph(
            torch, [lambda i=i: fb.fp8bq_static_gemm(qs, s_x, qwss[i], sp, parts, ys, wss)
                    for i in range(ns)], 2 * ns)
        keep["static"][M] = ys[:ORACLE_ROWS].cpu()
        tf = 2.0 * M * N * K / (t * 1e-3) / 1e12
        b = N * K + M * K + 2 * M * N
        st[str(M)] = {"us": round(t * 1e3, 2), "us_p10_p50_p90": t.us_pct(), "tflops": round(tf, 2),
                      "frac_fp8": round(tf / fp8_peak, 4),
                      "gbs": round(b / (t * 1e-3) / 1e9, 1),
                      "frac_hbm": round(b / (t * 1e-3) / 1e9 / hbm_peak, 4)}
    out["static_N14336_K4096"] = st
    nv.range_pop()
    del qwss, qws

    # channelwise W8A8: per-token quantiser, GEMM at the prefill and decode shapes
    ch = {}
    nv.range_push("channelwise W8A8")
    M, K = si.PREFILL["M"], si.PREFILL["K"]
    b = M * K * 3 + M * 4
    ns = n_sets(b)
    xs = _copies(to_dev(si.activations(M, K)), ns)
    qs = [torch.empty(M, K, dtype=torch.uint8, device=dev) for _ in range(ns)]
    ss = [torch.empty(M, dtype=torch.float32, device=dev) for _ in range(ns)]
    t = _time_graph(torch, [lambda i=i: fb.fp8bq_channel_quant_act(xs[i], qs[i], ss[i])
                            for i in range(ns)], 2 * ns)
    ch["quant_4096x6144"] = {"us": round(t * 1e3, 2), "us_p10_p50_p90": t.us_pct(),
                             "gbs": round(b / (t * 1e-3) / 1e9, 1),
                             "frac_hbm": round(b / (t * 1e-3) / 1e9 / hbm_peak, 4)}
    qa, sa = qs[0], ss[0]
    del xs
    for N in si.PREFILL["N_list"]:
        wb = to_dev(si.weights(N, K))
        qw = torch.empty(N, K, dtype=torch.uint8, device=dev)
        sw = torch.empty(N, dtype=torch.float32, device=dev)
        fb.fp8bq_channel_quant_act(wb, qw, sw)
        del wb
        y = torch.empty(M, N, dtype=torch.bfloat16, device=dev)
        ws = fb.new_workspace(fb.OP_CHANNEL_GEMM, M, N, K, device=dev)
        t = _time_back_to_back(torch, stream, [lambda: fb.fp8bq_channel_gemm(qa, sa, qw, sw, y, ws)], 20)
        tf = 2.0 * M * N * K / (t * 1e-3) / 1e12
        ch[f"gemm_{M}x{N}x{K}"] = {"us": round(t * 1e3, 2), "us_p10_p50_p90": t.us_pct(),
                                   "tflops": round(tf, 1), "frac_fp8": round(tf / fp8_peak, 4)}
        del qw, sw, y
    K = N = si.DECODE["K"]
    wb = to_dev(si.weights(N, K))
    qw = torch.empty(N, K, dtype=torch.uint8, device=dev)
    sw = torch.empty(N, dtype=torch.float32, device=dev)
    fb.fp8bq_channel_quant_act(wb, qw, sw)
    del wb
    ns = n_sets(N * K)
    qws, sws = _copies(qw, ns), _copies(sw, ns)
    for M in si.DECODE["M_list"]:
        qd = torch.empty(M, K, dtype=torch.uint8, device=dev)
        sd = torch.empty(M, dtype=torch.float32, device=dev)
        fb.fp8bq_channel_quant_act(to_dev(si.activations(M, K)), qd, sd)
        y = torch.empty(M, N, dtype=torch.bfloat16, device=dev)
        ws = fb.new_workspace(fb.OP_CHANNEL_GEMM, M, N, K, device=dev)
        t = _time_graph(torch, [lambda i=i: fb.fp8bq_channel_gemm(qd, sd, qws[i], sws[i], y, ws)
                                for i in range(ns)], 2 * ns)
        bb = N * K + N * 4 + M * (K + 4) + 2 * M * N
        ch[f"gemm_decode_{M}x{N}x{K}"] = {"us": round(t * 1e3, 2), "us_p10_p50_p90": t.us_pct(),
                                          "gbs": round(bb / (t * 1e-3) / 1e9, 1),
                                          "frac_hbm": round(bb / (t * 1e-3) / 1e9 / hbm_peak, 4)}
    out["channel_w8a8"] = ch
    nv.range_pop()
    del qw, sw, qws, sws

    # block FP8 with UE8M0 scales on the block-scaled MMA, at the prefill shapes
    ue = {}
    nv.range_push("block FP8 with UE8M0 scales")
    M, K = si.PREFILL["M"], si.PREFILL["K"]
    KB = K // 128
    b = M * K * 3 + M * KB
    ns = n_sets(b)
    xs = _copies(to_dev(si.activations(M, K)), ns)
    qs = [torch.empty(M, K, dtype=torch.uint8, device=dev) for _ in range(ns)]
    us = [torch.empty(M, KB, dtype=torch.uint8, device=dev) for _ in range(ns)]
    t = _time_graph(torch, [lambda i=i: fb.fp8bq_quant_act_ue8m0(xs[i], qs[i], us[i])
                            for i in range(ns)], 2 * ns)
    ue["quant_4096x6144"] = {"us": round(t * 1e3, 2), "us_p10_p50_p90": t.us_pct(),
                             "gbs": round(b / (t * 1e-3) / 1e9, 1),
                             "frac_hbm": round(b / (t * 1e-3) / 1e9 / hbm_peak, 4)}
    qa, ua = qs[0], us[0]
    del xs
    for N in si.PREFILL["N_list"]:
        wb = to_dev(si.weights(N, K))
        qw = torch.empty(N, K, dtype=torch.uint8, device=dev)
        sw = torch.empty(N // 128, KB, dtype=torch.float32, device=dev)
        fb.fp8bq_quant_weight_block(wb, qw, sw)
        uw = torch.empty(N // 128, KB, dtype=torch.uint8, device=dev)
        fb.fp8bq_requant_weight_ue8m0(qw, sw, qw, uw)
        del wb
        y = torch.empty(M, N, dtype=torch.bfloat16, device=dev)
        ws = fb.new_workspace(fb.OP_UE8M0_GEMM, M, N, K, device=dev)
        t = _time_back_to_back(torch, stream, [lambda: fb.fp8bq_ue8m0_gemm(qa, ua, qw, uw, y, ws)], 20)
        tf = 2.0 * M * N * K / (t * 1e-3) / 1e12
        ue[f"gemm_{M}x{N}x{K}"] = {"us": round(t * 1e3, 2), "us_p10_p50_p90": t.us_pct(),
                                   "tflops": round(tf, 1), "frac_fp8": round(tf / fp8_peak, 4)}
        del qw, sw, uw, y
    out["block_ue8m0"] = ue
    nv.range_pop()
    del qs, us

    # grouped (MoE) block GEMM: 32 local experts, 4096 routed rows with skewed
    # routing, the w13 and w2 shapes.  Four weight sets are drawn and copied to
    # fill the experts (distinct memory, so every expert's weight streams from
    # HBM; together they exceed L2 several times over).
    mo = si.MOE
    E, T = mo["E"], mo["T"]
    counts = si.expert_counts(T, E, mo["skew"])
    off = torch.tensor(np.concatenate([[0], np.cumsum(counts)]).astype(np.int32), device=dev)
    live = int((counts > 0).sum())
    gr = {"experts": E, "rows": T, "max_rows": int(counts.max()), "min_rows": int(counts.min()),
          "m_tiles_256": int(np.sum((counts + 255) // 256))}
    nv.range_push("grouped (MoE) GEMM")
    for which, N, K in (("w13", 2 * mo["I"], mo["H"]), ("w2", mo["H"], mo["I"])):
        KB, NB = K // 128, N // 128
        qw = torch.empty(E, N, K, dtype=torch.uint8, device=dev)
        sw = torch.empty(E, NB, KB, dtype=torch.float32, device=dev)
        for e in range(4):
            wb = to_dev(si.weights(N, K, base_seed=e))
            fb.fp8bq_quant_weight_block(wb, qw[e], sw[e])
            del wb
        for e in range(4, E):
            qw[e].copy_(qw[e % 4])
            sw[e].copy_(sw[e % 4])
        qa = torch.empty(T, K, dtype=torch.uint8, device=dev)
        sa = torch.empty(T, KB, dtype=torch.float32, device=dev)
        fb.fp8bq_quant_act(to_dev(si.activations(T, K)), qa, sa)
        y = torch.empty(T, N, dtype=torch.bfloat16, device=dev)
        ws = fb.new_workspace(fb.OP_GROUPED_GEMM, T, N, K, device=dev)
        t = _time_back_to_back(torch, stream,
                               [lambda: fb.fp8bq_grouped_gemm(qa, sa, qw, sw, off, y, ws)], 20)
        flops = 2.0 * T * N * K
        bb = live * (N * K + NB * KB * 4) + T * (K + KB * 4) + 2 * T * N
        tf = flops / (t * 1e-3) / 1e12
        gbs = bb / (t * 1e-3) / 1e9
        # the bound: the larger of the HBM time and the FP8 tensor time
        t_min = max(bb / (hbm_peak * 1e9), flops / (fp8_peak * 1e12))
        gr[f"{which}_N{N}_K{K}"] = {"us": round(t * 1e3, 2), "us_p10_p50_p90": t.us_pct(),
                                    "tflops": round(tf, 1),
                                    "gbs": round(gbs, 1), "frac_fp8": round(tf / fp8_peak, 4),
                                    "frac_hbm": round(gbs / hbm_peak, 4),
                                    "frac_roofline": round(t_min / (t * 1e-3), 4)}
        del qa, sa, y
        if which == "w13":
            # decode-time MoE in the masked layout: 256 routed rows over the 32
            # experts, slots of 64 rows; the launch streams every expert's
            # weights once for a few rows each
            Td, max_m = 256, 64
            cd = np.minimum(si.expert_counts(Td, E, mo["skew"], base_seed=1), max_m)
            mm = torch.tensor(cd.astype(np.int32), device=dev)
            qd = torch.randint(0, 0x7E, (E * max_m, K), dtype=torch.uint8, device=dev)
            sd = torch.rand(E * max_m, KB, device=dev) + 0.5
            yd = torch.empty(E * max_m, N, dtype=torch.bfloat16, device=dev)
            wsd = fb.new_workspace(fb.OP_GROUPED_GEMM, E * max_m, N, K, device=dev)
            t = _time_back_to_back(torch, stream,
                                   [lambda: fb.fp8bq_grouped_gemm_masked(qd, sd, qw, sw, mm, yd, wsd)],
                                   20)
            live_d = int((cd > 0).sum())
            bd = live_d * (N * K + NB * KB * 4) + int(cd.sum()) * (K + KB * 4 + 2 * N)
            gr[f"masked_decode_{which}_rows{int(cd.sum())}_slots{max_m}"] = {
                "us": round(t * 1e3, 2), "us_p10_p50_p90": t.us_pct(),
                "gbs": round(bd / (t * 1e-3) / 1e9, 1),
                "frac_hbm": round(bd / (t * 1e-3) / 1e9 / hbm_peak, 4)}
            del qd, sd, yd
        del qw, sw
    out["grouped_moe"] = gr
    nv.range_pop()

    # context only (not a denominator): the vendor's plain FP8 GEMM with
    # per-tensor scales (cuBLASLt through torch._scaled_mm) at the prefill shape
    # and at 8192^3; it has no per-block promotion to do

    # residual add + RMSNorm + quantisation (the step before the linear):
    # x, residual in; updated residual, E4M3 codes (and group scales) out
    norm = {}
    nv.range_push("residual add + RMSNorm + quantisation")
    eps = si.NORM["eps"]
    cases = [("group", 4096, 6144), ("group", 64, 6144), ("group", 1, 6144),
             ("static", 4096, 4096), ("static", 512, 4096), ("static", 1, 4096)]
    for mode, M, K in cases:
        b = M * K * 2 * 3 + M * K + 2 * K + (M * (K // 128) * 4 if mode == "group" else 0)
        ns = n_sets(b)
        xs = _copies(to_dev(si.activations(M, K)), ns)
        rs = _copies(to_dev(si.residual_stream(M, K)), ns)
        gn = to_dev(si.norm_gain(K))
        if mode == "static":  # the scale of the normalised rows, from one run
            y0 = torch.empty(M, K, dtype=torch.bfloat16, device=dev)
            fb.fp8bq_add_rmsnorm_quant_act(xs[0], gn, eps, residual=rs[0], y=y0)
            s_n = torch.empty(1, dtype=torch.float32, device=dev)
            fb.fp8bq_absmax_scale(y0, s_n)
            del y0
        ros = [torch.empty(M, K, dtype=torch.bfloat16, device=dev) for _ in range(ns)]
        qs = [torch.empty(M, K, dtype=torch.uint8, device=dev) for _ in range(ns)]
        if mode == "group":
            ss = [torch.empty(M, K // 128, dtype=torch.float32, device=dev) for _ in range(ns)]
            fns = [lambda i=i: fb.fp8bq_add_rmsnorm_quant_act(
                xs[i], gn, eps, residual=rs[i], residual_out=ros[i], q=qs[i], s=ss[i])
                for i in range(ns)]
        else:
            fns = [lambda i=i: fb.fp8bq_add_rmsnorm_static_quant_act(
                xs[i], gn, eps, s_n, qs[i], residual=rs[i], residual_out=ros[i])
                for i in range(ns)]
        t = _time_graph(torch, fns, 2 * ns)
        norm[f"{mode}_{M}x{K}"] = {"us": round(t * 1e3, 2), "us_p10_p50_p90": t.us_pct(),
                                   "gbs": round(b / (t * 1e-3) / 1e9, 1),
                                   "frac_hbm": round(b / (t * 1e-3) / 1e9 / hbm_peak, 4)}
        del xs, rs, ros, qs
    out["add_rmsnorm_quant"] = norm
    nv.range_pop()

    # the tiny linear (16 x 384 x 256): launch-bound, timed in a graph
    nv.range_push("tiny linear 16x384x256")
    M, K, N = si.TINY["M"], si.TINY["K"], si.TINY["N"]
    xt = to_dev(si.activations(M, K, outliers=False))
    wb = to_dev(si.weights(N, K))
    qwt = torch.empty(N, K, dtype=torch.uint8, device=dev)
    swt = torch.empty(-(-N // 128), -(-K // 128), dtype=torch.float32, device=dev)
    fb.fp8bq_quant_weight_block(wb, qwt, swt)
    yt = torch.empty(M, N, dtype=torch.bfloat16, device=dev)
    wst = fb.new_workspace(fb.OP_LINEAR, M, N, K, device=dev)
    t = _time_graph(torch, [lambda: fb.fp8bq_linear(xt, qwt, swt, yt, wst)], 20)
    keep["tiny"] = yt.cpu()
    out["tiny_linear_16x384x256"] = {"us": round(t * 1e3, 2), "us_p10_p50_p90": t.us_pct()}
    nv.range_pop()
    return out


# ---------------------------------------------------------------------------
# CPU oracle (baseline leg and the reference arm)
# ---------------------------------------------------------------------------

def oracle_sample(rows: int):
    """Prepared inputs for the oracle on the first `rows` tokens of the workload."""
    import oracle
    K = PREFILL_K
    x = si.activations(rows, K)
    ws = []
    for N in PREFILL_NS:
        qw, sw = oracle.quant_weight_block(si.weights(N, K))
        ws.append((qw, sw))
    return x, ws


def oracle_step(x, ws, threads):
    import oracle
    qa, sa = oracle.quant_group(x)
    for qw, sw in ws:
        oracle.gemm_block(qa, sa, qw, sw, threads=threads)


def _bf16_host(t):
    """A host BF16 tensor (GPU output) as float64 numpy."""
    return t.float().numpy().astype(np.float64)


def _close(y, ref):
    """The parity tests' GEMM tolerance: per element |y - ref| <= 1e-2 max(1, |ref|),
    relative Frobenius error <= 4e-3."""
    y = np.asarray(y, np.float64)
    ref = np.asarray(ref, np.float64)
    err = np.abs(y - ref)
    ok = bool(np.all(err <= 1e-2 * np.maximum(1.0, np.abs(ref))) and np.all(np.isfinite(y)))
    nref = np.linalg.norm(ref)
    rel = float(np.linalg.norm(y - ref) / nref) if nref > 0 else 0.0
    return {"ok": ok and rel <= 4e-3, "max_abs_err": float(err.max()) if err.size else 0.0,
            "rel_frob": round(rel, 7)}


def _exact(got, ref):
    got, ref = np.asarray(got), np.asarray(ref)
    bad = int(np.count_nonzero(got != ref)) if got.shape == ref.shape else -1
    return {"ok": bad == 0, "mismatches": bad}


def cpu_baseline(args, keep=None):
    """The oracle on the host cores: one bounded sample of every workload
    configuration, timed (its quantisers single-threaded C, its binary64 GEMMs
    on all cores).  Where `keep` holds the GPU's outputs for the same seeded
    inputs, each sample also checks them: codes and scales bit for bit, GEMM
    outputs within the parity tests' tolerance.  The headline figure (value,
    unit) is the prefill linear's; `configs` has one entry per configuration."""
    import oracle
    keep = keep or {}
    threads = os.cpu_count() or 1
    cfg = {}
    perf = time.perf_counter

    # tiny linear 16 x 384 x 256: all of it
    M, K, N = si.TINY["M"], si.TINY["K"], si.TINY["N"]
    qw, sw = oracle.quant_weight_block(si.weights(N, K))
    x = si.activations(M, K, outliers=False)
    t0 = perf()
    qa, sa = oracle.quant_group(x)
    y = oracle.gemm_block(qa, sa, qw, sw, threads=threads)
    dt = perf() - t0
    cfg["tiny_linear_16x384x256"] = {
        "s": round(dt, 4), "tflops": 2.0 * M * N * K / dt / 1e12, "cores": threads,
        "sample": "the whole linear",
        "parity": _close(_bf16_host(keep["tiny"]), y) if "tiny" in keep else None}

    # decode GEMMs K = N = 6144, M in {1, 8, 32, 64}: every output
    K = N = si.DECODE["K"]
    qw, sw = oracle.quant_weight_block(si.weights(N, K))
    dec = {}
    for M in si.DECODE["M_list"]:
        x = si.activations(M, K)
        t0 = perf()
        qa, sa = oracle.quant_group(x)
        y = oracle.gemm_block(qa, sa, qw, sw, threads=threads)
        dt = perf() - t0
        b = N * K + sw.size * 4 + M * (K + K // 128 * 4) + 2 * M * N
        got = keep.get("decode", {}).get(M)
        dec[str(M)] = {"s": round(dt, 4), "gbs": round(b / dt / 1e9, 4),
                       "parity": _close(_bf16_host(got), y) if got is not None else None}
    cfg["decode_6144x6144"] = {"cores": threads, "sample": "quant + GEMM, every output",
                               "per_M": dec}

    # prefill: the first rows of the 4096-token batch through quant + both GEMMs
    rows = args.cpu_rows
    K = PREFILL_K
    x = si.activations(rows, K)
    wts = {N: oracle.quant_weight_block(si.weights(N, K)) for N in PREFILL_NS}
    t0 = perf()
    qa, sa = oracle.quant_group(x)
    t1 = perf()
    ys = {N: oracle.gemm_block(qa, sa, qw, sw, threads=threads) for N, (qw, sw) in wts.items()}
    t2 = perf()
    dt = t2 - t0
    flops = sum(2.0 * rows * K * N for N in PREFILL_NS)
    par = {str(N): _close(_bf16_host(keep["prefill"][N][:rows]), ys[N])
           for N in PREFILL_NS if N in keep.get("prefill", {})}
    prefill_tf = flops / dt / 1e12
    cfg["prefill_4096x6144"] = {
        "s": round(dt, 3), "tflops": prefill_tf, "cores": threads,
        "sample": f"first {rows} tokens through quant + FP64 block GEMM for N in "
                  f"{list(PREFILL_NS)}",
        "quant_s": round(t1 - t0, 4), "gemm_s": round(t2 - t1, 3), "parity": par or None}
    del wts, ys

    # MXFP8 2048 x 4096 x 7168: the first rows
    M, K, N = si.MXFP8["M"], si.MXFP8["K"], si.MXFP8["N"]
    r = min(ORACLE_ROWS, M)
    qw, uw = oracle.quant_mx(si.weights(N, K))
    x = si.activations(r, K)
    t0 = perf()
    qa, ua = oracle.quant_mx(x)
    y = oracle.gemm_mx(qa, ua, qw, uw, threads=threads)
    dt = perf() - t0
    cfg["mxfp8_2048x4096x7168"] = {
        "s": round(dt, 4), "tflops": 2.0 * r * N * K / dt / 1e12, "cores": threads,
        "sample": f"first {r} tokens through MX quant + FP64 MX GEMM",
        "parity": _close(_bf16_host(keep["mx_gemm"][:r]), y) if "mx_gemm" in keep else None}

    # static per-tensor N = 14336 (4096 / 4096 / 6144), K = 4096
    K, N, parts = si.STATIC["K"], si.STATIC["N"], list(si.STATIC["parts"])
    s_x = oracle.absmax_scale(si.calibration(si.STATIC["calib_rows"], K))
    qw, sp = oracle.quant_weight_static(si.weights(N, K), parts)
    st = {}
    for M in si.STATIC["M_list"]:
        r = min(ORACLE_ROWS, M)
        x = si.activations(r, K, outliers=False)
        t0 = perf()
        qa = oracle.quant_static(x, s_x)
        y = oracle.gemm_static(qa, s_x, qw, sp, parts, threads=threads)
        dt = perf() - t0
        got = keep.get("static", {}).get(M)
        st[str(M)] = {"s": round(dt, 4), "tflops": 2.0 * r * N * K / dt / 1e12,
                      "rows": r, "parity": _close(_bf16_host(got[:r]), y)
                      if got is not None else None}
    cfg["static_14336x4096"] = {"cores": threads, "per_M": st,
                                "sample": f"first min(M, {ORACLE_ROWS}) tokens per M"}
    del qw

    # quantisers (single-threaded C), whole workload inputs
    M, K = 4096, 6144
    x = si.activations(M, K)
    t0 = perf()
    q, s = oracle.quant_group(x)
    dt = perf() - t0
    par = None
    if "quant_group" in keep:
        gq, gs = keep["quant_group"]
        a, b = _exact(gq.numpy(), q), _exact(gs.numpy().view(np.uint32), s.view(np.uint32))
        par = {"ok": a["ok"] and b["ok"], "code_mismatches": a["mismatches"],
               "scale_mismatches": b["mismatches"]}
    cfg["quant_group128_4096x6144"] = {
        "s": round(dt, 4), "gbs": round(M * (3 * K + 4 * (K // 128)) / dt / 1e9, 4),
        "cores": 1, "sample": "the whole 4096 x 6144 input", "parity": par}
    M, K = si.MXFP8["M"], si.MXFP8["K"]
    x = si.activations(M, K)
    t0 = perf()
    q, u = oracle.quant_mx(x)
    dt = perf() - t0
    par = None
    if "quant_mx" in keep:
        gq, gu = keep["quant_mx"]
        a, b = _exact(gq.numpy(), q), _exact(gu.numpy(), u)
        par = {"ok": a["ok"] and b["ok"], "code_mismatches": a["mismatches"],
               "scale_mismatches": b["mismatches"]}
    cfg["quant_mx_2048x7168"] = {
        "s": round(dt, 4), "gbs": round(M * (3 * K + K // 32) / dt / 1e9, 4), "cores": 1,
        "sample": "the whole 2048 x 7168 input", "parity": par}

    return {"value": prefill_tf, "unit": "TFLOPS", "cores": threads, "kind": "oracle",
            "sample": cfg["prefill_4096x6144"]["sample"] + f" ({cfg['prefill_4096x6144']['s']} s)",
            "configs": cfg}


def build_records(M, K, layers, gemm_lists, step_list, flops_step, extra, cpu, hbm_peak,
                  fp8_peak, achieved):
    """One record per (workload configuration, op): time percentiles, the
    roofline fraction, the oracle's parity check and its time with its cores."""
    recs = []
    cc = (cpu or {}).get("configs", {})

    def rec(config, op, shape, us_pct, bound, value, unit, frac, parity=None, oracle=None):
        recs.append({"config": config, "op": op, "shape": shape, "us_p10_p50_p90": us_pct,
                     "bound": bound, "achieved": value, "unit": unit, "frac": frac,
                     "parity": parity, "oracle": oracle})

    def orc(entry, keys=("s", "cores", "sample")):
        return None if entry is None else {k: entry.get(k) for k in keys if k in entry}

    pre = cc.get("prefill_4096x6144")
    for L, g in zip(layers, gemm_lists):
        us = [round(v * 1e3, 2) for v in pcts(g)]
        tf = 2.0 * M * K * L["N"] / (np.median(g) * 1e-3) / 1e12
        rec("prefill", "block GEMM", f"{M}x{L['N']}x{K}", us, "tensor", round(tf, 1), "TFLOP/s",
            round(tf / fp8_peak, 4), (pre or {}).get("parity", {}).get(str(L["N"])) if pre
            else None, orc(pre))
    st_us = [round(v * 1e3, 2) for v in pcts(step_list)]
    rec("prefill", "quant + 2 GEMMs (bench step)", f"X[{M},{K}]", st_us, "tensor",
        round(flops_step / (np.median(step_list) * 1e-3) / 1e12, 1), "TFLOP/s", None,
        None, orc(pre))
    if not extra:
        return recs
    tiny = extra.get("tiny_linear_16x384x256")
    if tiny:
        rec("tiny", "linear", "16x384x256", tiny["us_p10_p50_p90"], "launch", None, None, None,
            (cc.get("tiny_linear_16x384x256") or {}).get("parity"),
            orc(cc.get("tiny_linear_16x384x256")))
    dec_o = (cc.get("decode_6144x6144") or {}).get("per_M", {})
    for Ms, d in extra.get("decode_N6144_K6144", {}).items():
        o = dec_o.get(Ms)
        rec("decode", "block GEMM", f"{Ms}x6144x6144", d.get("gemm_us_p10_p50_p90"), "hbm",
            d["gemm_gbs"], "GB/s", d["gemm_frac_hbm"], (o or {}).get("parity"),
            None if o is None else {"s": o["s"], "cores": cc["decode_6144x6144"]["cores"],
                                    "sample": "every output"})
        rec("decode", "linear", f"{Ms}x6144x6144", d.get("linear_us_p10_p50_p90"), "hbm",
            d["linear_gbs"], "GB/s", d["linear_frac_hbm"], None, None)
    qd = extra.get("quant", {})
    if "group128_4096x6144" in qd:
        d, o = qd["group128_4096x6144"], cc.get("quant_group128_4096x6144")
        rec("prefill", "group-128 quant", "4096x6144", d.get("us_p10_p50_p90"), "hbm", d["gbs"],
            "GB/s", d["frac_hbm"], (o or {}).get("parity"), orc(o))
    if "mx_2048x7168" in qd:
        d, o = qd["mx_2048x7168"], cc.get("quant_mx_2048x7168")
        rec("mxfp8", "MX quant", "2048x7168", d.get("us_p10_p50_p90"), "hbm", d["gbs"], "GB/s",
            d["frac_hbm"], (o or {}).get("parity"), orc(o))
    d = extra.get("mx_gemm_2048x4096x7168")
    if d:
        o = cc.get("mxfp8_2048x4096x7168")
        rec("mxfp8", "MX GEMM", "2048x4096x7168", d.get("us_p10_p50_p90"), "tensor", d["tflops"],
            "TFLOP/s", d["frac_fp8"], (o or {}).get("parity"), orc(o))
    st_o = (cc.get("static_14336x4096") or {}).get("per_M", {})
    for Ms, d in extra.get("static_N14336_K4096", {}).items():
        o = st_o.get(Ms)
        hbm = Ms == "1"
        rec("static", "per-tensor GEMM", f"{Ms}x14336x4096", d.get("us_p10_p50_p90"),
            "hbm" if hbm else "tensor", d["gbs"] if hbm else d["tflops"],
            "GB/s" if hbm else "TFLOP/s", d["frac_hbm"] if hbm else d["frac_fp8"],
            (o or {}).get("parity"),
            None if o is None else {"s": o["s"], "rows": o["rows"],
                                    "cores": cc["static_14336x4096"]["cores"]})
    # rows past the five configurations: parity is in the -m gpu tests
    gpu_tests = "tests -m gpu (not rechecked here)"
    for k, d in extra.get("channel_w8a8", {}).items():
        hbm = "gbs" in d and "tflops" not in d
        rec("channelwise", k, k.split("_")[-1], d.get("us_p10_p50_p90"), "hbm" if hbm else "tensor",
            d["gbs"] if hbm else d["tflops"], "GB/s" if hbm else "TFLOP/s",
            d["frac_hbm"] if hbm else d["frac_fp8"], gpu_tests, None)
    for k, d in extra.get("block_ue8m0", {}).items():
        hbm = "tflops" not in d
        rec("block UE8M0", k, k.split("_")[-1], d.get("us_p10_p50_p90"), "hbm" if hbm else "tensor",
            d["gbs"] if hbm else d["tflops"], "GB/s" if hbm else "TFLOP/s",
            d["frac_hbm"] if hbm else d["frac_fp8"], gpu_tests, None)
    for k, d in extra.get("grouped_moe", {}).items():
        if isinstance(d, dict):
            rec("grouped MoE", k, k, d.get("us_p10_p50_p90"), "hbm", d["gbs"], "GB/s",
                d["frac_hbm"], gpu_tests, None)
    for k, d in extra.get("add_rmsnorm_quant", {}).items():
        rec("add + RMSNorm + quant", k, k.split("_")[-1], d.get("us_p10_p50_p90"), "hbm", d["gbs"],
            "GB/s", d["frac_hbm"], gpu_tests, None)
    return recs


def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return
    threads = os.cpu_count() or 1
    rows = args.ref_rows
    x, ws = oracle_sample(rows)
    for _ in range(args.warmup):
        oracle_step(x, ws, threads)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle_step(x, ws, threads)
    dt = time.perf_counter() - t0
    flops = sum(2.0 * rows * PREFILL_K * N for N in PREFILL_NS) * args.steps
    value = flops / dt / 1e12
    sample = (f"each step: first {rows} tokens of the prefill batch through the oracle's "
              f"quant + FP64 block GEMM for N in {list(PREFILL_NS)}")
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOPS",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": dt * 1e3 / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": f"prefill block-FP8 linear: X[{PREFILL_M},{PREFILL_K}] BF16 -> "
                               f"N in {list(PREFILL_NS)}, BF16 out (CPU sample)"},
        "cpu_baseline": {"value": value, "unit": "TFLOPS", "cores": threads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "TFLOPS", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }), flush=True)


PROFILE_CASES = ("mx", "norm_group", "norm_static", "grouped_w13", "grouped_w2", "channel",
                 "ue8m0", "quant_group", "decode_m1", "decode_m64", "static_4096", "static_512",
                 "decode_linear_m1", "decode_linear_m16")


def run_profile_case(case: str, launches: int = 3):
    """A few launches of one kernel at its workload shape and nothing else, for
    an ncu capture (no timing, no JSON line).  Operand values are random codes
    and scales drawn on the device: counters do not depend on them."""
    import torch
    sys.path.insert(0, ROOT)
    import block_wise_fp8_gb300 as fb
    dev = torch.device("cuda")
    torch.manual_seed(0)
    codes = lambda *shape: torch.randint(0, 0x7E, shape, dtype=torch.uint8, device=dev)
    if case in ("mx", "ue8m0"):
        M, K, N = (si.MXFP8["M"], si.MXFP8["K"], si.MXFP8["N"]) if case == "mx" else \
                  (PREFILL_M, PREFILL_K, PREFILL_NS[1])
        G = K // 32 if case == "mx" else K // 128
        q, w = codes(M, K), codes(N, K)
        u = torch.randint(120, 130, (M, G), dtype=torch.uint8, device=dev)
        uw = torch.randint(120, 130, (N if case == "mx" else N // 128, G), dtype=torch.uint8,
                           device=dev)
        y = torch.empty(M, N, dtype=torch.bfloat16, device=dev)
        op = fb.OP_MX_GEMM if case == "mx" else fb.OP_UE8M0_GEMM
        ws = fb.new_workspace(op, M, N, K, device=dev)
        fn = (lambda: fb.fp8bq_mx_gemm(q, u, w, uw, y, ws)) if case == "mx" else \
             (lambda: fb.fp8bq_ue8m0_gemm(q, u, w, uw, y, ws))
    elif case == "channel":
        M, K, N = PREFILL_M, PREFILL_K, PREFILL_NS[1]
        q, w = codes(M, K), codes(N, K)
        sx = torch.rand(M, device=dev) + 0.5
        sw = torch.rand(N, device=dev) * 1e-3
        y = torch.empty(M, N, dtype=torch.bfloat16, device=dev)
        ws = fb.new_workspace(fb.OP_CHANNEL_GEMM, M, N, K, device=dev)
        fn = lambda: fb.fp8bq_channel_gemm(q, sx, w, sw, y, ws)
    elif case.startswith("norm"):
        static = case == "norm_static"
        M, K = (4096, 4096) if static else (4096, 6144)
        to_dev = lambda b: torch.from_numpy(b.view(np.int16)).to(dev).view(torch.bfloat16)
        x, r = to_dev(si.activations(M, K)), to_dev(si.residual_stream(M, K))
        g = to_dev(si.norm_gain(K))
        ro = torch.empty(M, K, dtype=torch.bfloat16, device=dev)
        q = torch.empty(M, K, dtype=torch.uint8, device=dev)
        eps = si.NORM["eps"]
        if static:
            s_n = torch.full((1,), 0.05, dtype=torch.float32, device=dev)
            fn = lambda: fb.fp8bq_add_rmsnorm_static_quant_act(x, g, eps, s_n, q, residual=r,
                                                               residual_out=ro)
        else:
            s = torch.empty(M, K // 128, dtype=torch.float32, device=dev)
            fn = lambda: fb.fp8bq_add_rmsnorm_quant_act(x, g, eps, residual=r, residual_out=ro,
                                                        q=q, s=s)
    elif case == "quant_group":
        M, K = PREFILL_M, PREFILL_K
        x = torch.randn(M, K, device=dev).to(torch.bfloat16)
        q = torch.empty(M, K, dtype=torch.uint8, device=dev)
        sx = torch.empty(M, K // 128, dtype=torch.float32, device=dev)
        fn = lambda: fb.fp8bq_quant_act(x, q, sx)
    elif case.startswith("decode_linear"):
        # the one-launch decode linear: BF16 activations quantised inside the GEMM
        M, K, N = int(case[len("decode_linear_m"):]), si.DECODE["K"], si.DECODE["N"]
        x = torch.randn(M, K, device=dev).to(torch.bfloat16)
        w = codes(N, K)
        sw = torch.rand(N // 128, K // 128, device=dev) * 1e-3
        y = torch.empty(M, N, dtype=torch.bfloat16, device=dev)
        ws = fb.new_workspace(fb.OP_LINEAR, M, N, K, device=dev)
        fn = lambda: fb.fp8bq_linear(x, w, sw, y, ws)
    elif case.startswith("decode"):
        M, K, N = int(case[len("decode_m"):]), si.DECODE["K"], si.DECODE["N"]
        q, w = codes(M, K), codes(N, K)
        sx = torch.rand(M, K // 128, device=dev) + 0.5
        sw = torch.rand(N // 128, K // 128, device=dev) * 1e-3
        y = torch.empty(M, N, dtype=torch.bfloat16, device=dev)
        ws = fb.new_workspace(fb.OP_GEMM, M, N, K, device=dev)
        fn = lambda: fb.fp8bq_gemm(q, sx, w, sw, y, ws)
    elif case in ("static_4096", "static_512"):
        M, K, N = int(case.split("_")[1]), si.STATIC["K"], si.STATIC["N"]
        q, w = codes(M, K), codes(N, K)
        sxs = torch.full((1,), 0.01, dtype=torch.float32, device=dev)
        sp = torch.rand(len(si.STATIC["parts"]), device=dev) * 1e-3
        y = torch.empty(M, N, dtype=torch.bfloat16, device=dev)
        ws = fb.new_workspace(fb.OP_STATIC_GEMM, M, N, K, device=dev)
        fn = lambda: fb.fp8bq_static_gemm(q, sxs, w, sp, list(si.STATIC["parts"]), y, ws)
    elif case.startswith("grouped"):
        mo = si.MOE
        E, T = mo["E"], mo["T"]
        N, K = (2 * mo["I"], mo["H"]) if case == "grouped_w13" else (mo["H"], mo["I"])
        counts = si.expert_counts(T, E, mo["skew"])
        off = torch.tensor(np.concatenate([[0], np.cumsum(counts)]).astype(np.int32), device=dev)
        qw, qa = codes(E, N, K), codes(T, K)
        sw = torch.rand(E, N // 128, K // 128, device=dev) * 1e-3
        sa = torch.rand(T, K // 128, device=dev) + 0.5
        y = torch.empty(T, N, dtype=torch.bfloat16, device=dev)
        ws = fb.new_workspace(fb.OP_GROUPED_GEMM, T, N, K, device=dev)
        fn = lambda: fb.fp8bq_grouped_gemm(qa, sa, qw, sw, off, y, ws)
    else:
        raise SystemExit(f"unknown profile case {case}")
    for _ in range(launches):
        fn()
    torch.cuda.synchronize()
    print(f"profile case {case}: {launches} launches", file=sys.stderr)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cpu-rows", type=int, default=8)
    ap.add_argument("--ref-rows", type=int, default=2)
    ap.add_argument("--no-extra", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--profile-case", choices=PROFILE_CASES,
                    help="only run a few launches of one kernel (for ncu captures)")
    args = ap.parse_args(argv)
    if args.profile_case:
        run_profile_case(args.profile_case)
        return
    if args.warmup < 3 and args.impl == "ours":
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
