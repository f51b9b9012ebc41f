"""The multi-rank path of bench.py on CPU (no GPU): world size 2 over gloo.

bench.py runs one independent replica per GPU (the quantiser and the GEMM
shard over tokens with no exchange), so its only cross-rank steps are the
barrier around the timed region, the max over ranks of the time and the sum
of the work.  Those are checked here with two gloo processes; the reference
arm is run under torchrun with two ranks, where rank 0 alone prints."""
import json
import os
import socket
import subprocess
import sys

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench.barrier(world)
        t_max = bench.aggregate([1.5 + rank, 10.0 * rank], world, rank, True)
        w_sum = bench.aggregate([100.0 + rank], world, rank, False)
        bench.barrier(world)
        out.put((rank, t_max, w_sum))
    finally:
        dist.destroy_process_group()


def test_aggregate_and_barrier_gloo_world2():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    for rank, t_max, w_sum in res:
        assert t_max == [2.5, 10.0]     # max over ranks, element by element
        assert w_sum == [201.0]         # sum over ranks


def test_reference_arm_under_torchrun_world2():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "0", "--ref-rows", "1"]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1                      # rank 0 alone prints
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle"
