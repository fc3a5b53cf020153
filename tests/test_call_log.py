"""The per-call JSON-lines log (DDP_RING_LOG): one record per collective call
with the entry point, algo, p, n, dtype, algorithmic bytes, the bytes each
simulated rank sends in the method's schedule, the status and the device
time. The variable is read once per process, so each case runs in a child
process."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(code, log_path, timeout=240):
    env = dict(os.environ, DDP_RING_LOG=str(log_path), PYTHONPATH=ROOT)
    r = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True, timeout=timeout)
    assert r.returncode == 0, r.stderr[-2000:]
    with open(log_path) as f:
        return [json.loads(line) for line in f if line.strip()]


def test_log_records_status_and_bytes_without_a_gpu(tmp_path):
    """Zero-size calls and argument errors need no device: the records carry
    the status, the byte counts and no time."""
    code = """
import ring_all_reduce_ddp_gb300 as D
D.ddp_allreduce([0, 0, 0, 0], 0, D.DDP_FLOAT32, 4.0, stream=0)
try:
    D.ddp_allreduce([0, 0, 0, 0], 0, D.DDP_FLOAT32, 0.0, stream=0)
except D.DDPError:
    pass
D.ddp_broadcast([0, 0, 0], 0, 1, stream=0)
"""
    recs = _run(code, tmp_path / "log.jsonl")
    assert [r["op"] for r in recs] == ["ddp_allreduce", "ddp_allreduce", "ddp_broadcast"]
    assert recs[0]["status"] == "DDP_OK" and recs[0]["p"] == 4 and recs[0]["n"] == 0
    # no device: no time; with one, the no-op is timed like any call
    assert recs[0]["bytes_algorithmic"] == 0 and (recs[0]["elapsed_us"] is None or recs[0]["elapsed_us"] >= 0)
    assert recs[1]["status"] == "DDP_ERR_ARG"
    assert recs[2]["status"] == "DDP_OK" and recs[2]["p"] == 3


def test_no_log_without_the_variable(tmp_path):
    env = dict(os.environ, PYTHONPATH=ROOT)
    env.pop("DDP_RING_LOG", None)
    code = "import ring_all_reduce_ddp_gb300 as D; D.ddp_allreduce([0, 0], 0, D.DDP_FLOAT32, 2.0, stream=0)"
    r = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True, timeout=120, cwd=tmp_path)
    assert r.returncode == 0, r.stderr
    assert os.listdir(tmp_path) == []


@pytest.mark.gpu
def test_log_times_real_calls(tmp_path):
    code = """
import torch
import ring_all_reduce_ddp_gb300 as D
import synth
from ring_all_reduce_ddp_gb300.reducer import Reducer
from synth import workloads as W
p, n = 8, 1000003
bufs = [torch.empty(n, device="cuda") for _ in range(p)]
for r, b in enumerate(bufs):
    synth.fill_(b, "uniform", 3, r)
D.ddp_allreduce(bufs, n, D.DDP_FLOAT32, 8.0, D.DDP_ALGO_FUSED)
D.ddp_allreduce(bufs, n, D.DDP_FLOAT32, 8.0, D.DDP_ALGO_RECURSIVE_DOUBLING)
outs = [torch.empty(n // p + 1, device="cuda") for _ in range(p)]
D.ddp_reduce_scatter(bufs, outs, n, D.DDP_FLOAT32, 1.0, D.DDP_OWN_RING, D.DDP_ALGO_RING_STEPS)
cfg = W.CONFIGS["tiny"]
grads, _ = W.make_grads(cfg)
red = Reducer(grads, cfg["first_cap"], cfg["cap"])
red.sync_gradients(W.divisor(cfg))
g = torch.cuda.CUDAGraph()
with torch.cuda.graph(g):
    red.sync_gradients(W.divisor(cfg))
torch.cuda.synchronize()
bn = [[torch.zeros(10, device="cuda"), torch.zeros(3, dtype=torch.int64, device="cuda")] for _ in range(len(grads))]
red.set_buffers(bn, root=1)
red.step(W.divisor(cfg))
torch.cuda.synchronize()
"""
    recs = _run(code, tmp_path / "log.jsonl")
    ops = [r["op"] for r in recs]
    assert ops == ["ddp_allreduce", "ddp_allreduce", "ddp_reduce_scatter", "ddp_reducer_sync", "ddp_reducer_sync",
                   "ddp_reducer_step"]
    p, n, cs = 8, 1000003, -(-1000003 // 8)
    ar, rd, rs, sync, captured, step = recs
    assert ar["bytes_algorithmic"] == 2 * p * n * 4 and ar["bytes_per_rank"] == 2 * (p - 1) * cs * 4
    assert rd["bytes_per_rank"] == 3 * n * 4  # log2 8 whole-buffer exchanges
    assert rs["bytes_algorithmic"] == (p + 1) * n * 4 and rs["bytes_per_rank"] == (p - 1) * cs * 4
    for r in (ar, rd, rs, sync):
        assert r["status"] == "DDP_OK" and r["elapsed_us"] > 0
    assert sync["p"] == 4 and sync["n"] == 277421
    assert captured["elapsed_us"] is None  # inside a stream capture nothing is timed
    # the step adds the broadcast of B = 10*4 + 3*8 bytes: p*B algorithmic,
    # log2(p) copies of B per rank (the doubling tree's depth)
    B = 10 * 4 + 3 * 8
    assert step["status"] == "DDP_OK" and step["elapsed_us"] > 0 and step["n"] == sync["n"]
    assert step["bytes_algorithmic"] == sync["bytes_algorithmic"] + 4 * B
    assert step["bytes_per_rank"] == sync["bytes_per_rank"] + 2 * B
