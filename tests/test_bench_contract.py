"""The JSON line bench.py prints: one line, the keys and types the driver
reads. The reference arm (the oracle on the host) runs anywhere; the GPU arm
needs a GB300."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
BASE_KEYS = {"metric": str, "value": (int, float), "unit": str, "n_gpus": int, "steps": int, "warmup": int,
             "ms_per_step": (int, float), "higher_is_better": bool, "scaling": str, "dtype": str, "data": str,
             "config": dict}


def _run(args, timeout=600):
    r = subprocess.run([sys.executable, "bench.py", *args], cwd=ROOT, capture_output=True, text=True,
                       timeout=timeout)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1, r.stdout[-2000:]
    return json.loads(lines[0])


def _base(d):
    for k, t in BASE_KEYS.items():
        assert isinstance(d[k], t), (k, d.get(k))
    assert d["vs_baseline"] is None and "workload" in d["config"]


def test_reference_arm_line():
    d = _run(["--impl", "reference", "--steps", "2", "--warmup", "1", "--config", "tiny"])
    _base(d)
    assert d["impl"] == "reference" and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
    assert d["config"]["same_config"] is True  # a few tiny steps: the whole step every time


def test_reference_arm_times_the_gpu_arms_step_bytes():
    """The oracle's step is credited with the bytes the GPU arm's in-place step
    is credited with: 2pM for the sync and pB for the buffers' broadcast."""
    import bench
    from synth import workloads as W
    from synth import shapes as S
    cfg = W.CONFIGS["resnet50"]
    M = sum(W.numels(cfg)) * 4
    B = sum(4 * S.numel(shp) if dt == "f32" else 8 * S.numel(shp) for _, shp, dt in S.resnet50_buffers())
    assert bench.oracle_step_bytes(cfg) == 2 * 8 * M + 8 * B
    tiny = W.CONFIGS["tiny"]
    assert bench.oracle_step_bytes(tiny) == 2 * 4 * sum(W.numels(tiny)) * 4


@pytest.mark.gpu
def test_gpu_arm_line():
    d = _run(["--steps", "20", "--warmup", "3", "--no-cpu-baseline"])
    _base(d)
    assert d["metric"] and d["value"] > 0 and d["dtype"] == "f32"
    r = d["roofline"]
    assert r["bound"] == "hbm" and r["unit"] == "GB/s" and 0 < r["frac"] < 1.2 and r["peak"] > 0
    assert abs(r["frac"] - r["achieved"] / r["peak"]) < 1e-3
    assert r["event_timed_launches"] >= 32
    assert r["kernel"].startswith("k_bucket_table_staged")  # fp32 at p = 8 takes the staged form
    assert r["traffic"] is None or 0.9 < r["traffic"] / r["algorithmic_bytes_per_launch"] < 1.05
    e = d["e2e"]
    assert e["value"] > 0 and e["h2d_bytes_per_step"] > 0 and e["d2h_bytes_per_step"] > 0
    assert d["gpu_launches"] == 20  # the buffer broadcast and the sync: one launch every step
    assert set(d["clocks"]) >= {"sm_mhz", "sm_max_mhz", "reasons"}
    pts = d["sweep"]["points"]
    assert {(x["p"], x["bytes"] >> 20) for x in pts} == {(p, m) for p in (2, 8, 64) for m in (1, 25, 256)}
    assert all(x["gbs"] > 0 and abs(x["frac"] - x["gbs"] / r["peak"]) < 1e-3 for x in pts)
    assert set(d["configs"]) == {"gpt2_small", "llama_1b"}
    assert all(c["us"] > 0 and c["buckets_per_s"] > 0 for c in d["configs"].values())


@pytest.mark.gpu
def test_gpu_arm_under_torchrun_two_ranks():
    """The N > 1 launch the contract uses (torchrun, one process per GPU),
    here two gloo ranks sharing this machine's GPUs: one JSON line from rank
    0, the whole-job value over both ranks, max-over-ranks timing."""
    import socket
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    env = dict(os.environ, DDP_BENCH_BACKEND="gloo", OMP_NUM_THREADS="1")
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port),
           "bench.py", "--gpus", "2", "--steps", "5", "--warmup", "3", "--no-cpu-baseline"]
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.strip().startswith("{")]
    assert len(lines) == 1, r.stdout[-2000:]
    d = json.loads(lines[0])
    _base(d)
    assert d["n_gpus"] == 2 and d["value"] > 0 and d["gpu_launches"] == 5
    assert "sweep" not in d and d["cpu_baseline"] is None
