"""The multi-process path of bench.py, on CPU with the gloo backend.

The layer shards across (sequence, head) with no exchange, so N GPUs run N
replicas; the only cross-rank steps are the barriers around the timed region
and the max / sum reductions of the timings and token counts.  These tests run
them with world_size 2 on CPU, and check that under torchrun only rank 0 of
the reference arm prints its JSON line.
"""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    r, w, _ = bench.dist_setup()
    bench.barrier(w)
    mx = bench.max_over_ranks(1.5 + r, w)        # e.g. per-rank ms per step
    sm = bench.sum_over_ranks(100.0 * (r + 1), w)  # e.g. per-rank tokens
    bench.barrier(w)
    out.put((r, w, mx, sm))
    import torch.distributed as dist
    dist.destroy_process_group()


def test_rank_reductions_world_size_2():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r for r, *_ in res] == [0, 1]
    for _, w, mx, sm in res:
        assert w == 2 and mx == 2.5 and sm == 300.0


def test_reference_arm_under_torchrun_prints_once():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr", "127.0.0.1", "--master-port", str(port),
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
           "--steps", "1", "--warmup", "1"]
    env = dict(os.environ, OMP_NUM_THREADS="1")
    res = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600, env=env)
    assert res.returncode == 0, res.stderr[-2000:]
    lines = [l for l in res.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, res.stdout
    rec = json.loads(lines[0])
    assert rec["impl"] == "reference" and rec["n_gpus"] == 2 and rec["steps"] == 1
    assert rec["cpu_baseline"]["kind"] == "oracle" and rec["value"] > 0
