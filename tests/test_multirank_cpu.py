"""Multi-rank logic of bench.py on the CPU (gloo, world size 2).

The block shards over sequences with no exchange step, so bench.py runs one replica
per rank and only reduces its timing: the slowest rank's time, all ranks' tokens.
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
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench
    r, w, _ = bench.dist_setup()
    t = bench.reduce_max(10.0 * (rank + 1), w)
    bench.barrier(w)
    q.put((r, w, t, dist.get_backend()))
    dist.destroy_process_group()


def test_two_ranks_reduce_the_slowest_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [o[0] for o in out] == [0, 1]
    assert all(o[1] == 2 and o[2] == 20.0 and o[3] == "gloo" for o in out)


def _ref_env(rank):
    return dict(os.environ, RANK=str(rank), WORLD_SIZE="2", LOCAL_RANK=str(rank))


def test_reference_arm_runs_on_rank0_only():
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--config", "tiny",
           "--steps", "2", "--warmup", "1", "--gpus", "2"]
    r1 = subprocess.run(cmd, env=_ref_env(1), capture_output=True, text=True, timeout=300)
    assert r1.returncode == 0 and r1.stdout.strip() == ""
    r0 = subprocess.run(cmd, env=_ref_env(0), capture_output=True, text=True, timeout=300)
    assert r0.returncode == 0, r0.stderr
    line = json.loads(r0.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["d2h_bytes_per_step"] == 0
