"""Multi-process paths of bench.py on the CPU, world size 2 over gloo.

Heads are independent, so several GPUs run replicas: no data-path
collective, only the timing barrier and the max over ranks.  These tests run
that host logic with two CPU ranks (127.0.0.1 rendezvous), and the reference
arm as ``torch.distributed.run`` launches it, where rank 0 alone works and
prints.
"""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.multiprocessing as mp

# on a GPU machine bench.py's ranks take NCCL and one GPU each: CPU only here
pytestmark = pytest.mark.skipif(torch.cuda.is_available(), reason="CPU (gloo) test")

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, port, out):
    os.environ.update({"RANK": str(rank), "LOCAL_RANK": str(rank), "WORLD_SIZE": "2",
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    sys.path.insert(0, ROOT)
    import bench

    r, world, local, dist = bench.dist_setup(2)
    bench.barrier(dist)
    # each rank times something different; the job's time is the slowest rank's
    m = bench.max_over_ranks(1.5 + 3.0 * rank, dist)
    bench.barrier(dist)
    out.put((r, world, local, dist.get_backend(), m))
    dist.destroy_process_group()


def test_replica_timing_helpers_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted(out.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [g[0] for g in got] == [0, 1]
    for r, world, local, backend, m in got:
        assert world == 2 and local == r and backend == "gloo"
        assert m == 4.5  # the max over ranks, seen by both


def test_reference_arm_prints_once_from_rank_zero():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port),
           "bench.py", "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "0",
           "--workload", "tiny"]
    env = dict(os.environ, OMP_NUM_THREADS="1")
    res = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert res.returncode == 0, res.stderr[-2000:]
    lines = [ln for ln in res.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, res.stdout
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"
