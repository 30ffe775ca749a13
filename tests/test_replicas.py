"""The N > 1 path of bench.py (independent replicas, one process per GPU) on CPU: the slowest
rank's timing is what every rank reports, whole-job throughput counts every replica's bytes,
and under torchrun only rank 0 prints the result line.  Two gloo ranks on 127.0.0.1."""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    # rank r's timings: r + 1 ms and 10 - r ms; every rank must see the per-column maximum
    got = bench.max_over_ranks([rank + 1.0, 10.0 - rank], "cpu", world)
    out.put((rank, got))
    dist.barrier()
    dist.destroy_process_group()


def test_max_over_ranks_with_two_gloo_ranks():
    import multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert res[0] == res[1] == [2.0, 10.0]


def test_replica_throughput_counts_every_rank():
    import bench
    # 2 replicas, 1 GB per step each, 10 steps in 5 ms (slowest rank): 4000 GB/s whole-job
    assert bench.replica_gbs(1e9, 10, 2, 5.0) == pytest.approx(4000.0)
    assert bench.replica_gbs(1e9, 10, 1, 5.0) == pytest.approx(2000.0)


def test_reference_arm_under_torchrun_prints_one_line():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes", "1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--config", "1", "--gpus", "2", "--steps", "1", "--warmup", "1"]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    rec = json.loads(lines[0])
    assert rec["impl"] == "reference" and rec["n_gpus"] == 2 and rec["value"] > 0
