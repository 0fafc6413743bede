"""Multi-rank path on the CPU: world_size 2 over gloo (no GPU).

Each rank draws its own batch values, runs one step of the layer (here the CPU
oracle stands in for the GPU step), and the ranks agree on the maximum time;
bench.py's reference arm under torchrun prints exactly one line (rank 0).
"""
import json
import os
import socket
import subprocess
import sys

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world),
                      RANK=str(rank), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import time

    import oracle
    from ragged_blocked_kv_raggedbatch_gb300 import replicas
    from ragged_blocked_kv_raggedbatch_gb300 import workloads as W
    grp = replicas.Group("gloo")
    wl = W.make_workload("tiny_gqa_d64", 0)
    qkv, pool = W.make_values(wl, "cpu", seed=replicas.rank_seed(0, grp.rank))
    grp.barrier()
    t0 = time.perf_counter()
    out = oracle.layer(wl, qkv, pool, n_threads=1)["out"]
    mine = time.perf_counter() - t0
    mx = grp.max(mine)
    q.put((grp.rank, mine, mx, float(np.abs(out).sum())))
    grp.close()


def test_two_ranks_over_gloo():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = [q.get(timeout=300) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    res.sort()
    times = [r[1] for r in res]
    assert all(abs(r[2] - max(times)) < 1e-12 for r in res)  # every rank sees the max
    assert res[0][3] != res[1][3]  # each rank ran its own batch values


def test_reference_arm_under_torchrun_prints_one_line():
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()),
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2", "--steps", "3",
           "--warmup", "3", "--workload", "tiny_gqa_d64"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle"
