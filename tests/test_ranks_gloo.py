"""The bench's multi-rank host logic on CPU: two gloo ranks, independent
replicas, a barrier and the max over ranks of a timing (world_size 2)."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update({"RANK": str(rank), "LOCAL_RANK": str(rank), "WORLD_SIZE": str(world),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port), "DDP_BENCH_BACKEND": "gloo"})
    import bench
    r = bench.Ranks()
    try:
        r.barrier()
        got = r.max(10.0 + rank * 2.5)
        q.put((rank, r.world, got))
    finally:
        r.close()


def test_two_gloo_ranks_take_the_max():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for pr in procs:
        pr.start()
    res = [q.get(timeout=120) for _ in range(world)]
    for pr in procs:
        pr.join(timeout=60)
        assert pr.exitcode == 0
    assert sorted(x[0] for x in res) == [0, 1]
    assert all(x[1] == 2 and x[2] == 12.5 for x in res)


def test_single_process_needs_no_group(monkeypatch):
    monkeypatch.delenv("WORLD_SIZE", raising=False)
    import bench
    r = bench.Ranks()
    assert r.world == 1 and r.max(3.0) == 3.0
    r.barrier()
    r.close()


def test_reference_arm_under_torchrun_prints_one_line_from_rank_0():
    """`bench.py --impl reference` launched by torchrun with two ranks: rank 0
    alone times the oracle and prints the JSON line; the other rank exits 0
    without work."""
    import json
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = dict(os.environ, DDP_BENCH_BACKEND="gloo", OMP_NUM_THREADS="1")
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()),
           "bench.py", "--impl", "reference", "--gpus", "2", "--steps", "2", "--warmup", "1", "--config", "tiny"]
    r = subprocess.run(cmd, cwd=root, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.strip().startswith("{")]
    assert len(lines) == 1, r.stdout[-2000:]
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
