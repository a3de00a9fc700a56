"""The multi-rank path of bench.py on CPU (gloo, world size 2).

The operation has no exchange step, so N GPUs run N independent replicas;
what crosses ranks is only the timing: a barrier on both sides of the timed
steps and the maximum step time over ranks.  These tests run those helpers
in two gloo ranks, and the reference arm launched the way the driver
launches N > 1 (torch.distributed.run), where rank 0 alone prints the line.
"""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, port, q):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE="2", LOCAL_RANK=str(rank))
    import bench
    ws, r, local = bench.dist_env()
    dist.init_process_group("gloo", init_method="env://")
    try:
        bench.barrier(ws)
        m = bench.reduce_max(1.5 + r, ws)       # each rank's "step time"
        bench.barrier(ws)
        q.put((r, ws, local, m))
    finally:
        dist.destroy_process_group()


def test_barrier_and_max_over_two_ranks():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    got = sorted(q.get(timeout=5) for _ in range(2))
    assert got == [(0, 2, 0, 2.5), (1, 2, 1, 2.5)]


def test_single_rank_helpers_need_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.reduce_max(3.25, 1) == 3.25
    bench.barrier(1)


def test_reference_arm_under_torchrun_two_ranks():
    """Rank 0 prints exactly one JSON line for the reference arm; rank 1 does
    no work and exits 0."""
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="", OMP_NUM_THREADS="2")
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()), "bench.py",
           "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "3",
           "--workload", "tiny_1x256_h4kv1"]
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-3000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "TFLOP/s" and d["value"] > 0
    assert d["config"]["workload"] == "tiny_1x256_h4kv1"
    assert d["cpu_baseline"]["kind"] == "oracle"
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["value"] == d["value"]
