#!/usr/bin/env python3
"""Benchmark of one DDP gradient-synchronisation step over p simulated replicas
held in one GPU's memory.

A step is one pass of the whole hot path on the workload's synthetic
gradients: bucket assignment (host), the per-forward coalesced broadcast of the
model's buffers from replica 0, then the gradient sync of every bucket. By
default (--mode in_place) the sync is one launch that, for every bucket,
flattens, ring-all-reduces and unflattens in a single pass over the
gradients; --mode flatten runs the three separate kernels per bucket.

Default workload: the ResNet-50-shaped gradient set (161 fp32 tensors, 25.6M
parameters) on p = 8 replicas, 1 MiB first bucket / 25 MiB buckets, averaged
by 1/8, plus the broadcast of its 159 BatchNorm buffers.

Prints ONE JSON line (rank 0). value = algorithmic bytes of all the step's ops
(all-reduce 2pM; in flatten mode also flatten 2pM and unflatten 2pM; broadcast
p * buffer bytes) over the device-timed step, in GB/s, summed over ranks. --impl reference times the
CPU oracle instead (on a bounded sample of the same workload).
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "simulated ring-allreduce HBM GB/s (frac of GB300 peak) vs bucket size, rank count"
UNIT = "GB/s"
FALLBACK_HBM_GBS = 6800.0

WORKLOAD_TEXT = {
    "resnet50": ("ResNet-50-shaped gradient set: 161 fp32 tensors (25,557,032 params), p=8 simulated "
                 "replicas, reversed-registration buckets with 1 MiB first / 25 MiB cap, average by 1/8; "
                 "plus per-forward coalesced broadcast of the 159 BatchNorm buffers from replica 0"),
    "gpt2_small": ("GPT-2-small-shaped gradient set: 148 fp32 tensors (124,439,808 params), p=8, 25 MiB "
                   "buckets, divide once by the global token count"),
    "llama_1b": ("Llama-style 1B gradient set: 147 bf16 tensors (1,204,881,408 params), p=8, 25 MiB "
                 "buckets, fp32 accumulate, average by 1/8; plus per-forward broadcast of 64 fp32 buffers"),
    "tiny": "ten odd-sized fp32 tensors (277,421 elements), p=4, 16 KiB / 256 KiB buckets, average by 1/4",
}

# DRAM traffic of the dominant kernel (the in-place bucket all-reduce) from an
# ncu capture, as bytes per algorithmic byte; valid only while the kernel
# source it was taken on is unchanged (checked by hash).
EVENT_EVERY = 16  # timed steps per event-timed launch of the dominant kernel
NCU_TRAFFIC = {"kernel_sha256": "bcda9671e69737c3c345e46175295989edaac7c9ca0e1b38bafa06760dca6851",
               "config": "resnet50",  # the workload the capture ran; other workloads report null
               "dram_bytes_per_algorithmic_byte": (818.002432 + 758.240256) / 1635.650048}  # ncu: read + write MB per launch


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=4000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", default="resnet50", choices=sorted(WORKLOAD_TEXT))
    ap.add_argument("--algo", default="fused", choices=["fused", "ldst", "tma", "ring_steps"])
    ap.add_argument("--mode", default="in_place", choices=["in_place", "flatten"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget-s", type=float, default=12.0)
    ap.add_argument("--sweep", action="store_true", help="message-size / rank-count sweep, one line per point")
    ap.add_argument("--overlap", action="store_true", help="exposed communication vs bucket cap, one line per cap")
    return ap.parse_args()


# --------------------------------------------------------------- ranks
class Ranks:
    """One process per GPU (torchrun); independent replicas, no data-path collective.
    The process group serves the barrier and the max over ranks of the timings."""

    def __init__(self):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local = int(os.environ.get("LOCAL_RANK", "0"))
        self.dist = None
        if self.world > 1:
            import torch
            import torch.distributed as dist
            backend = os.environ.get("DDP_BENCH_BACKEND") or ("nccl" if torch.cuda.is_available() else "gloo")
            dist.init_process_group(backend)
            self.backend = backend
            self.dist = dist

    def barrier(self):
        if self.dist is not None:
            import torch
            if self.backend == "nccl":
                self.dist.barrier(device_ids=[self.local])
            else:
                self.dist.barrier()

    def max(self, x: float) -> float:
        if self.dist is None:
            return x
        import torch
        dev = f"cuda:{self.local}" if self.backend == "nccl" else "cpu"
        t = torch.tensor([x], dtype=torch.float64, device=dev)
        self.dist.all_reduce(t, op=self.dist.ReduceOp.MAX)
        return float(t.item())

    def close(self):
        if self.dist is not None:
            self.dist.destroy_process_group()


# --------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during the timed region."""
    FIELDS = ["timestamp", "clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.active",
              "clocks_event_reasons.hw_slowdown", "clocks_event_reasons.hw_thermal_slowdown",
              "clocks_event_reasons.sw_thermal_slowdown", "clocks_event_reasons.sw_power_cap"]

    def __init__(self, device_index: int):
        self.idx = device_index
        self.proc = None
        self.lines: list[str] = []

    def start(self):
        try:
            import torch
            ident = "GPU-" + str(torch.cuda.get_device_properties(self.idx).uuid)
        except Exception:
            ident = str(self.idx)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "--query-gpu=" + ",".join(self.FIELDS), "--format=csv,noheader,nounits",
                 "-i", ident, "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self._t = threading.Thread(target=self._read, daemon=True)
            self._t.start()
        except FileNotFoundError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self, window=None) -> dict | None:
        """Median SM clock and active throttle reasons over the samples taken
        inside window = (start, end) host wall-clock seconds (all samples if None)."""
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self._t.join(timeout=2)
        rows = self._parse(window)
        in_window = window is not None and bool(rows)
        if not rows:  # clock skew between nvidia-smi and the host: report every sample
            rows = self._parse(None)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        sm = [r[0] for r in rows]
        reasons = sorted(set().union(*[r[2] for r in rows]))
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(r[1] for r in rows), "reasons": reasons,
                "samples": len(rows), "in_timed_window": in_window}

    def _parse(self, window):
        import datetime
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        rows = []
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) != len(self.FIELDS):
                continue
            try:
                when = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                clk, clk_max = float(parts[1]), float(parts[2])
            except ValueError:
                continue
            if window is not None and not (window[0] - 0.05 <= when <= window[1] + 0.05):
                continue
            active = {nm for nm, v in zip(names, parts[5:]) if v.lower().startswith("active")}
            rows.append((clk, clk_max, active))
        return rows


# --------------------------------------------------------------- helpers
def peak_hbm() -> tuple[float, str]:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def cores_used() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def cpu_model() -> str:
    """The host CPU's model name, from lscpu (Arm hosts) or /proc/cpuinfo."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except Exception:
        pass
    return "unknown"


def algo_code(name):
    import ring_all_reduce_ddp_gb300 as D
    return {"fused": D.DDP_ALGO_FUSED, "ldst": D.DDP_ALGO_FUSED_LDST, "tma": D.DDP_ALGO_FUSED_TMA,
            "ring_steps": D.DDP_ALGO_RING_STEPS}[name]


def l2_note(grad_bytes: int, dev: int) -> str:
    """What the timed steps find in L2: the gradients of every replica are
    read and written once per step, so above twice the L2 size no step can
    find the previous step's data there."""
    import torch
    l2 = getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 0) or (126 << 20)
    if grad_bytes > 2 * l2:
        return "inputs larger than L2: %.2f GB of gradients per step, L2 %.0f MB" % (grad_bytes / 1e9, l2 / 1e6)
    return ("inputs fit in L2: %.1f MB of gradients per step, L2 %.0f MB; steps run L2-warm, so this "
            "workload measures latency, not HBM bandwidth" % (grad_bytes / 1e6, l2 / 1e6))


def kernel_sha() -> str:
    import hashlib
    h = hashlib.sha256()
    for f in ("k_bucket.cu",):
        with open(os.path.join(ROOT, "ring_all_reduce_ddp_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


# --------------------------------------------------------------- CPU oracle
def oracle_sync_sample(cfg, budget_s: float, max_buckets=None):
    """Time the oracle's gradient sync (flatten, literal ring all-reduce,
    unflatten) bucket by bucket until the budget is used. Returns
    (algorithmic bytes, seconds, description). Inputs are generated untimed."""
    import numpy as np

    from oracle import buckets as ob
    from oracle import ring as orc
    from synth import workloads as W
    numel = W.numels(cfg)
    starts = W.tensor_starts(cfg)
    es = W.esize(cfg)
    p = cfg["p"]
    plan = ob.assign_buckets(numel, es, cfg["first_cap"], cfg["cap"])
    _, offset, bnumel = ob.bucket_layout(numel, plan)
    Dv = W.divisor(cfg)
    total_bytes, total_t, done = 0, 0.0, []
    for b, members in enumerate(plan):
        if max_buckets is not None and len(done) >= max_buckets:
            break
        grads = [{t: W.host_values(cfg, r, np.arange(starts[t], starts[t] + numel[t])) for t in members}
                 for r in range(p)]
        t0 = time.perf_counter()
        flats = []
        for r in range(p):
            flats.append(ob.flatten([grads[r].get(t, np.zeros(0, np.float32 if es == 4 else np.uint16))
                                     for t in range(len(numel))], members, offset, bnumel[b]))
        outs, _ = orc.allreduce(flats, bnumel[b], Dv, cfg["dtype"])
        for r in range(p):
            ob.unflatten(outs[r], members, offset, numel)
        total_t += time.perf_counter() - t0
        total_bytes += 3 * 2 * p * bnumel[b] * es
        done.append(b)
        if total_t >= budget_s:
            break
    desc = (f"oracle flatten + literal ring all-reduce + unflatten of buckets {done} "
            f"({sum(bnumel[b] for b in done)} of {sum(bnumel)} elements per replica, p={p}), single thread")
    return total_bytes, total_t, desc


# --------------------------------------------------------------- our arm
def run_ours(args, ranks: Ranks):
    import torch

    import ring_all_reduce_ddp_gb300 as D
    from ring_all_reduce_ddp_gb300 import build as B
    from ring_all_reduce_ddp_gb300.reducer import BufferSync, Reducer
    from synth import workloads as W

    B.build_library()
    dev = ranks.local if torch.cuda.device_count() > 1 else 0
    torch.cuda.set_device(dev)
    cfg = W.CONFIGS[args.config]
    p = cfg["p"]
    algo = algo_code(args.algo)
    mode = D.DDP_SYNC_IN_PLACE if args.mode == "in_place" else D.DDP_SYNC_FLATTEN
    if args.algo == "ring_steps":
        mode = D.DDP_SYNC_FLATTEN
    grads, arenas = W.make_grads(cfg, f"cuda:{dev}")
    bufs = W.buffer_set(cfg, f"cuda:{dev}") if cfg.get("buffers") else None
    red = Reducer(grads, cfg["first_cap"], cfg["cap"])
    bsync = BufferSync(bufs, 0) if bufs else None
    divisor = W.divisor(cfg)
    stream = torch.cuda.current_stream()
    bc_algo = D.DDP_ALGO_RING_STEPS if args.algo == "ring_steps" else D.DDP_ALGO_FUSED
    buf_bytes = sum(bsync.nbytes) if bsync else 0
    esz = W.esize(cfg)

    def step(events=None, m=mode):
        if not red.assign():  # a1: bucket assignment (host)
            raise RuntimeError("bucket assignment changed")
        if bsync:             # a9: the forward's buffer broadcast
            bsync(bc_algo, stream)
        if events is not None:
            e0 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
        red.sync_gradients(divisor, algo, m, 1.0, stream)  # a2-a8
        if events is not None:
            e1 = torch.cuda.Event(enable_timing=True)
            e1.record(stream)
            events.append((e0, e1))

    ab = red.algorithmic_bytes(mode)
    step_bytes = ab["total"] + p * buf_bytes
    for _ in range(max(args.warmup, 0)):
        step()
    torch.cuda.synchronize()
    ranks.barrier()

    sampler = ClockSampler(dev)
    sampler.start()
    time.sleep(0.3)
    launches0 = D.ddp_kernel_launches()
    sync_events: list = []
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    ranks.barrier()
    w0 = time.time()
    e0.record(stream)
    for i in range(args.steps):
        # the dominant kernel is timed by events around it on every 16th step:
        # an event pair on every step would add its own cost to the step time
        step(sync_events if i % EVENT_EVERY == 0 else None)
    e1.record(stream)
    torch.cuda.synchronize()
    w1 = time.time()
    ranks.barrier()
    launches = D.ddp_kernel_launches() - launches0
    clocks = sampler.stop((w0, w1))
    ms = e0.elapsed_time(e1)
    ms_max = ranks.max(ms)
    ms_per_step = ms_max / args.steps
    value = step_bytes * args.steps * ranks.world / (ms_max / 1e3) / 1e9

    # Dominant kernel: the in-place bucket all-reduce, one launch per step over
    # every bucket. Its duration comes from events recorded around that launch
    # on its stream (every EVENT_EVERY-th step of the timed region), so any
    # launch latency the events catch counts against it.
    sync_ms = [a.elapsed_time(b) for a, b in sync_events]
    nb = len(red.buckets)
    launches_per_sync = 1 if mode == D.DDP_SYNC_IN_PLACE else None
    achieved = ab["allreduce"] * len(sync_ms) / (sum(sync_ms) / 1e3) / 1e9
    peak, peak_kind = peak_hbm()
    traffic = None
    if (NCU_TRAFFIC["kernel_sha256"] == kernel_sha() and NCU_TRAFFIC["config"] == args.config
            and mode == D.DDP_SYNC_IN_PLACE and NCU_TRAFFIC["dram_bytes_per_algorithmic_byte"]):
        traffic = int(NCU_TRAFFIC["dram_bytes_per_algorithmic_byte"] * ab["allreduce"])
    bucket_mb = [round(n * esz / 2 ** 20, 2) for n in red.bucket_numel]
    kernel_name = ("k_bucket_allreduce_table: every bucket's flatten + ring-order all-reduce + unflatten "
                   "in one launch" if mode == D.DDP_SYNC_IN_PLACE
                   else "flatten, fused all-reduce, unflatten per bucket (whole sync timed)")

    # End to end through the public API: every step copies every replica's
    # gradients in from pinned host memory, synchronises them and copies the
    # result out. Three device copies of the workload rotate, so step i+1's
    # copy-in (H2D stream) never waits for step i's sync: it only needs the
    # copy-out of step i-2, long done. Both link directions stay busy; the
    # sync runs on the compute stream between them.
    NSETS = 3
    sets = [(arenas, red)]
    for _ in range(NSETS - 1):
        g_x, a_x = W.make_grads(cfg, f"cuda:{dev}")
        sets.append((a_x, Reducer(g_x, cfg["first_cap"], cfg["cap"])))
    host_in = [a.detach().to("cpu").pin_memory() for a in arenas]
    host_out = [torch.empty_like(h).pin_memory() for h in host_in]
    h2d_s, d2h_s = torch.cuda.Stream(), torch.cuda.Stream()
    ev = lambda: torch.cuda.Event()
    h2d_done, comp_done, d2h_done = [ev() for _ in range(NSETS)], [ev() for _ in range(NSETS)], [None] * NSETS

    def e2e_step(i):
        k = i % NSETS
        ar_k, red_k = sets[k]
        with torch.cuda.stream(h2d_s):
            if d2h_done[k] is not None:
                h2d_s.wait_event(d2h_done[k])  # this set's previous result has been read out
            for a, h in zip(ar_k, host_in):
                a.copy_(h, non_blocking=True)
            h2d_done[k].record(h2d_s)
        stream.wait_event(h2d_done[k])
        if not red_k.assign():
            raise RuntimeError("bucket assignment changed")
        if bsync:
            bsync(bc_algo, stream)
        red_k.sync_gradients(divisor, algo, mode, 1.0, stream)
        comp_done[k].record(stream)
        with torch.cuda.stream(d2h_s):
            d2h_s.wait_event(comp_done[k])
            for a, h in zip(ar_k, host_out):
                h.copy_(a, non_blocking=True)
            d2h_done[k] = torch.cuda.Event()
            d2h_done[k].record(d2h_s)

    for i in range(max(4, min(args.warmup, 8))):
        e2e_step(i)
    torch.cuda.synchronize()
    ranks.barrier()
    f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    k_e2e = min(args.steps, 300)
    f0.record(h2d_s)
    stream.wait_stream(h2d_s)
    for i in range(k_e2e):
        e2e_step(i)
    stream.wait_stream(d2h_s)
    f1.record(stream)
    torch.cuda.synchronize()
    ranks.barrier()
    e2e_ms = ranks.max(f0.elapsed_time(f1))
    io = sum(a.numel() * a.element_size() for a in arenas)
    e2e = {"value": round(step_bytes * k_e2e * ranks.world / (e2e_ms / 1e3) / 1e9, 2), "unit": UNIT,
           "h2d_bytes_per_step": io, "d2h_bytes_per_step": io, "ms_per_step": round(e2e_ms / k_e2e, 4),
           "steps": k_e2e,
           "pipeline": "step i's copy-out overlaps step i+1's copy-in (three device copies, three streams)"}
    del sets

    # the same step body (buffer broadcast + sync) captured once as a CUDA graph
    # and replayed: what host launch overhead costs the eager step
    graph = None
    if mode == D.DDP_SYNC_IN_PLACE and ranks.world == 1:
        cg = torch.cuda.CUDAGraph()
        with torch.cuda.graph(cg):
            if bsync:
                bsync(bc_algo, None)
            red.sync_gradients(divisor, algo, mode, 1.0, None)
        for _ in range(3):
            cg.replay()
        torch.cuda.synchronize()
        k_g = min(args.steps, 2000)
        g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        g0.record(stream)
        for _ in range(k_g):
            cg.replay()
        g1.record(stream)
        torch.cuda.synchronize()
        graph = {"ms_per_step": round(g0.elapsed_time(g1) / k_g, 5), "steps": k_g,
                 "note": "buffer broadcast + in-place sync replayed from one CUDA graph (bucket assignment stays on the host)"}
        del cg

    # the three-kernel form of the same step, for comparison (not the headline)
    other = None
    if mode == D.DDP_SYNC_IN_PLACE:
        k2 = max(10, args.steps // 5)
        for _ in range(3):
            step(None, D.DDP_SYNC_FLATTEN)
        torch.cuda.synchronize()
        g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        g0.record(stream)
        for _ in range(k2):
            step(None, D.DDP_SYNC_FLATTEN)
        g1.record(stream)
        torch.cuda.synchronize()
        fl = red.algorithmic_bytes(D.DDP_SYNC_FLATTEN)["total"] + p * buf_bytes
        ms2 = g0.elapsed_time(g1) / k2
        other = {"mode": "flatten + all-reduce + unflatten", "ms_per_step": round(ms2, 5),
                 "gbs": round(fl / (ms2 / 1e3) / 1e9, 1), "steps": k2}

    cpu = None
    if ranks.rank == 0 and ranks.world == 1 and not args.no_cpu_baseline:
        nbytes, secs, desc = oracle_sync_sample(cfg, args.cpu_budget_s)
        cpu = {"value": round(nbytes / secs / 1e9, 4), "unit": UNIT, "cores": 1, "kind": "oracle", "sample": desc,
               "host_cores_available": cores_used(), "cpu_model": cpu_model()}

    line = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": ranks.world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": cfg["dtype"], "data": "synthetic",
        "config": {"workload": WORKLOAD_TEXT[args.config], "p": p, "buckets": nb, "bucket_mb": bucket_mb,
                   "algo": args.algo, "sync": "in_place" if mode == D.DDP_SYNC_IN_PLACE else "flatten",
                   "divisor": divisor,
                   "l2": l2_note(sum(a.numel() * a.element_size() for a in arenas), dev),
                   "parallelism": f"replicas only: {ranks.world} independent GPU(s)"},
        "roofline": {"bound": "hbm", "kernel": kernel_name, "achieved": round(achieved, 1),
                     "peak": peak, "peak_kind": peak_kind, "unit": "GB/s", "frac": round(achieved / peak, 4),
                     "traffic": traffic,
                     "algorithmic_bytes_per_launch": int(ab["allreduce"]) if launches_per_sync else None,
                     "avg_launch_us": round(1e3 * statistics.mean(sync_ms), 2) if launches_per_sync else None,
                     "avg_sync_us": round(1e3 * statistics.mean(sync_ms), 2),
                     "event_timed_launches": len(sync_ms), "event_every_steps": EVENT_EVERY},
        "allreduce_gbs": round(achieved, 1),
        "buckets_per_s": round(nb * args.steps * ranks.world / (ms_max / 1e3), 1),
        "busbw_gbs": round(sum(n * esz for n in red.bucket_numel) / (statistics.mean(sync_ms) / 1e3) / 1e9
                           * 2 * (p - 1) / p, 1),
        "flatten_form": other,
        "cuda_graph": graph,
        "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": launches, "clocks": clocks,
    }
    if ranks.rank == 0:
        print(json.dumps(line), flush=True)


# --------------------------------------------------------------- reference arm
def run_reference(args, ranks: Ranks):
    """The CPU oracle as it stands, on rank 0 only. Each step runs the oracle's
    literal ring all-reduce on all p replicas of a leading slice of the
    workload's first bucket, the slice sized so the whole run takes under a
    minute (the whole bucket when steps are few). Inputs are generated once,
    outside the timed region."""
    if ranks.rank != 0:
        return
    import numpy as np

    from oracle import buckets as ob
    from oracle import ring as orc
    from synth import workloads as W
    cfg = W.CONFIGS[args.config]
    p, es = cfg["p"], W.esize(cfg)
    numel = W.numels(cfg)
    starts = W.tensor_starts(cfg)
    plan = ob.assign_buckets(numel, es, cfg["first_cap"], cfg["cap"])
    _, offset, bnumel = ob.bucket_layout(numel, plan)
    n = bnumel[0]
    members = plan[0]
    flat = []
    for r in range(p):
        hv = {t: W.host_values(cfg, r, np.arange(starts[t], starts[t] + numel[t])) for t in members}
        zero = np.zeros(0, np.float32 if es == 4 else np.uint16)
        flat.append(ob.flatten([hv.get(t, zero) for t in range(len(numel))], members, offset, n))
    Dv = W.divisor(cfg)
    t0 = time.perf_counter()
    orc.allreduce(flat, n, Dv, cfg["dtype"])
    t_full = time.perf_counter() - t0
    budget = 45.0
    frac = min(1.0, budget / max(1e-9, (args.steps + args.warmup) * t_full))
    m = max(64 * p, int(n * frac))
    sample = [f[:m].copy() for f in flat]  # the first m elements of the bucket, reduced as one buffer
    for _ in range(max(args.warmup, 0)):
        orc.allreduce(sample, m, Dv, cfg["dtype"])
    t_tot = 0.0
    for _ in range(args.steps):
        t0 = time.perf_counter()
        orc.allreduce(sample, m, Dv, cfg["dtype"])
        t_tot += time.perf_counter() - t0
    nbytes = 2 * p * m * es * args.steps
    value = nbytes / t_tot / 1e9
    desc = (f"oracle literal ring all-reduce, per step, of the first {m} of the {n} elements of bucket 0 "
            f"(p={p}), single thread")
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": UNIT, "n_gpus": ranks.world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1e3 * t_tot / max(args.steps, 1), 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": cfg["dtype"],
        "data": "synthetic",
        "config": {"workload": WORKLOAD_TEXT[args.config], "p": p, "algo": "oracle literal ring"},
        "cpu_baseline": {"value": round(value, 4), "unit": UNIT, "kind": "oracle", "cores": 1, "sample": desc,
                         "host_cores_available": cores_used(), "cpu_model": cpu_model()},
        "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)

# --------------------------------------------------------------- sweep
def literal_traffic_bytes(op: str, algo: str, p: int, M: int):
    """HBM bytes one literal (launch-per-step) fp32 schedule moves, counted from
    its kernels, for the sweep's actual-traffic rate; None for the fused forms
    and the tree-shaped schedules. M is the sweep size in bytes.
    - all-reduce: p-1 reduce-scatter steps that read the local and the received
      chunk and write the sum (3 x 4 bytes per element, n elements per step
      over all ranks), then p-1 all-gather steps that copy one chunk per rank
      (2 x 4 bytes per element): 5(p-1) M;
    - reduce-scatter: p-1 steps of 3 x 4 bytes per element (inputs and fp32
      partials in, partials or the output out): 3(p-1) M;
    - all-gather of M / p bytes per rank into M: the placement copy and p-1
      steps, each copying M / p bytes on every rank: 2 p M;
    - broadcast by the doubling tree: p-1 copies of M: 2(p-1) M."""
    if algo != "ring_steps" or p < 2:
        return None
    if op == "allreduce":
        return 5 * (p - 1) * M
    if op.startswith("reduce_scatter"):
        return 3 * (p - 1) * M
    if op == "allgather":
        return 2 * p * M
    if op == "broadcast":
        return 2 * (p - 1) * M
    return None


def run_sweep(args, ranks: Ranks):
    """Message-size / rank-count sweep: one fp32 buffer of M = 1 KiB * 4^k bytes
    on each of p replicas (p * M <= 64 GiB), values uniform on [-1, 1);
    all-reduce, reduce-scatter (both ownerships), all-gather and broadcast in
    the fused and the literal form, and the tree-shaped all-reduces. One JSON
    line per point.

    Timing. Each point runs batches of `reps` launches back to back, each
    launch on its own copy of the inputs when the working set is under 2x L2
    (copies rotate through at most 4 GiB), so no launch finds its inputs in L2
    and every write-back a launch leaves is paid by a later launch of the same
    batch. Before each batch L2 is flushed: a 512 MiB write, then a 512 MiB
    read of another buffer, so the batch starts with clean lines that belong
    to neither. `us` = median over batches of (batch time / reps), the batch
    captured once in a CUDA graph and replayed (host launch cost excluded);
    `us_eager` = the same batch launched from the host. The persistent ring is
    timed eagerly only."""
    import torch

    import ring_all_reduce_ddp_gb300 as D
    from ring_all_reduce_ddp_gb300 import build as B
    import synth
    B.build_library()
    if ranks.rank != 0:
        return
    torch.cuda.set_device(0)
    peak, peak_kind = peak_hbm()
    ps = [int(x) for x in os.environ.get("SWEEP_P", "2,4,8,16,64").split(",")]
    min_k = int(os.environ.get("SWEEP_MIN_K", "0"))
    max_k = int(os.environ.get("SWEEP_MAX_K", "10"))
    ops = os.environ.get("SWEEP_OPS", "allreduce,reduce_scatter_rank,reduce_scatter_ring,allgather,broadcast")
    algos = os.environ.get("SWEEP_ALGOS", "fused,ring_steps,persistent,rd,rab,tree").split(",")
    tree_codes = {"rd": D.DDP_ALGO_RECURSIVE_DOUBLING, "rab": D.DDP_ALGO_RABENSEIFNER, "tree": D.DDP_ALGO_TREE}
    reps = int(os.environ.get("SWEEP_REPS", "20"))
    batches = int(os.environ.get("SWEEP_BATCHES", "5"))
    wflush = torch.empty(512 << 20, dtype=torch.uint8, device="cuda")
    rflush = torch.ones(128 << 20, dtype=torch.float32, device="cuda")
    l2 = torch.cuda.get_device_properties(0).L2_cache_size
    rotate_budget = 4 << 30

    def flush():
        wflush.fill_(1)
        rflush.sum()

    for p in ps:
        for k in range(min_k, max_k + 1):
            M = 1024 * 4 ** k
            if p * M > 64 << 30:
                continue
            n = M // 4
            m = n // p
            with_outs = ops != "allreduce"
            out_elems = max(n, p * m)
            set_bytes = p * M + (p * out_elems * 4 if with_outs else 0)
            nsets = 1
            if set_bytes < 2 * l2:
                nsets = max(1, min(reps, rotate_budget // set_bytes))
            sets = []
            for _ in range(nsets):
                bufs = []
                for r in range(p):
                    t = torch.empty(n, dtype=torch.float32, device="cuda")
                    synth.fill_(t, "uniform", 1005, r)
                    bufs.append(t)
                outs = [torch.empty(out_elems, dtype=torch.float32, device="cuda") for _ in range(p)] \
                    if with_outs else []
                sets.append((bufs, outs))
            for op in ops.split(","):
                for an in algos:
                    if an in ("persistent", "rd", "rab", "tree") and op != "allreduce":
                        continue
                    al = tree_codes[an] if an in tree_codes else (algo_code(an) if an != "persistent" else None)

                    def call(i, op=op, an=an, al=al):
                        bufs, outs = sets[i % nsets]
                        if op == "allreduce" and an == "persistent":
                            D.ddp_allreduce_persistent(bufs, n, D.DDP_FLOAT32, float(p))
                        elif op == "allreduce":
                            D.ddp_allreduce(bufs, n, D.DDP_FLOAT32, float(p), al)
                        elif op.startswith("reduce_scatter"):
                            own = D.DDP_OWN_RANK if op.endswith("rank") else D.DDP_OWN_RING
                            D.ddp_reduce_scatter(bufs, outs, n, D.DDP_FLOAT32, 1.0, own, al)
                        elif op == "allgather":
                            D.ddp_allgather(bufs, outs, m, D.DDP_FLOAT32, D.DDP_OWN_RANK, al)
                        else:
                            D.ddp_broadcast(bufs, M, 0, al)

                    nbytes = {"allreduce": 2 * p * M, "allgather": M + p * M, "broadcast": p * M}.get(
                        op, p * M + M)

                    # warm-up (first-use lookups, workspace pools), then one timed
                    # launch to size the batch: up to `reps` launches, fewer when
                    # one launch is long (a batch of about 5 ms is enough there)
                    for i in range(min(nsets, 3) + 1):
                        call(i)
                    flush()
                    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    a.record()
                    call(0)
                    b.record()
                    b.synchronize()
                    t1 = a.elapsed_time(b) / 1e3
                    nrep = max(3, min(reps, int(math.ceil(5e-3 / max(t1, 1e-9)))))
                    nbat = batches if t1 < 1e-3 else 3

                    def batch(nrep=nrep):
                        for i in range(nrep):
                            call(i)

                    def timed(run, nrep=nrep, nbat=nbat):
                        out = []
                        for _ in range(nbat):
                            flush()
                            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                            a.record()
                            run()
                            b.record()
                            b.synchronize()
                            out.append(a.elapsed_time(b) / 1e3 / nrep)
                        return statistics.median(out)

                    t_eager = timed(batch)
                    t_graph = None
                    if an != "persistent":
                        g = torch.cuda.CUDAGraph()
                        with torch.cuda.graph(g):
                            batch()
                        g.replay()
                        torch.cuda.synchronize()
                        t_graph = timed(g.replay)
                        del g
                    t = t_graph if t_graph is not None else t_eager
                    gbs = nbytes / t / 1e9
                    moved = literal_traffic_bytes(op, an, p, M)
                    line = {"sweep": op, "algo": an, "p": p, "bytes": M, "us": round(t * 1e6, 2),
                            "us_eager": round(t_eager * 1e6, 2), "timing": "graph" if t_graph else "eager",
                            "gbs": round(gbs, 1), "frac": round(gbs / peak, 4), "peak_kind": peak_kind,
                            "busbw_gbs": round(M / t / 1e9 * 2 * (p - 1) / p, 1) if op == "allreduce" else None,
                            "traffic_gbs": round(moved / t / 1e9, 1) if moved else None,
                            "traffic_frac": round(moved / t / 1e9 / peak, 4) if moved else None,
                            "input_copies": nsets, "reps": nrep, "batches": nbat}
                    print(json.dumps(line), flush=True)
            del sets
            torch.cuda.empty_cache()


# --------------------------------------------------------------- overlap
def run_overlap(args, ranks: Ranks):
    """Exposed communication against bucket cap, with readiness-driven firing.

    A synthetic backward walks the parameters last-registered first on the
    compute stream; each weight gradient costs two bf16 GEMMs with
    4 * numel * n_tok FLOPs in all (backward is about 4N FLOPs per token);
    after each gradient an event is recorded and the Reducer is told the
    gradient is ready, which launches every newly complete bucket's in-place
    all-reduce on a communication stream. For each cap: the backward alone,
    backward + overlapped sync, and backward followed by the sync. One JSON
    line per cap."""
    import torch

    import ring_all_reduce_ddp_gb300 as D
    from ring_all_reduce_ddp_gb300 import build as B
    from ring_all_reduce_ddp_gb300.reducer import Reducer
    from synth import workloads as W
    B.build_library()
    if ranks.rank != 0:
        return
    torch.cuda.set_device(0)
    cfg = W.CONFIGS[args.config]
    grads, _ = W.make_grads(cfg, "cuda:0")
    numel = W.numels(cfg)
    k = len(numel)
    divisor = W.divisor(cfg)
    n_tok = int(os.environ.get("OVERLAP_TOKENS", "65536"))
    kdim = 1024
    x = torch.randn(n_tok, kdim, device="cuda", dtype=torch.bfloat16)
    wmax = max((n + kdim - 1) // kdim for n in numel)
    w = torch.randn(kdim, wmax, device="cuda", dtype=torch.bfloat16)
    y = torch.empty(n_tok, wmax, device="cuda", dtype=torch.bfloat16)
    compute = torch.cuda.current_stream()
    # the communication stream at normal priority, or at the device's highest
    # (the block scheduler then starts pending all-reduce blocks ahead of the
    # backward's GEMM blocks)
    lo_prio, hi_prio = torch.cuda.Stream.priority_range()
    comm_streams = {"normal": torch.cuda.Stream(priority=lo_prio), "high": torch.cuda.Stream(priority=hi_prio)}
    comm = comm_streams["normal"]

    ready_events = [torch.cuda.Event() for _ in range(k)]

    def backward(red=None):
        for t in range(k - 1, -1, -1):
            cols = (numel[t] + kdim - 1) // kdim
            if numel[t] >= 4096:  # 2 GEMMs: 2 * (2 * n_tok * kdim * cols) ~ 4 * numel * n_tok FLOPs
                torch.mm(x, w[:, :cols], out=y[:, :cols])
                torch.mm(x, w[:, :cols], out=y[:, :cols])
            if red is not None:
                ready_events[t].record(compute)
                red.mark_ready(t, divisor, ready_events[t], comm)

    def timed(fn, reps):
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(compute)
        for _ in range(reps):
            fn()
        for cs in comm_streams.values():
            compute.wait_stream(cs)
        b.record(compute)
        torch.cuda.synchronize()
        return a.elapsed_time(b) / reps

    reps = max(5, min(args.steps, 50))
    t_bwd = timed(lambda: backward(None), reps)
    flops = 4.0 * sum(n for n in numel if n >= 4096) * n_tok
    caps = [int(float(c) * (1 << 20)) for c in os.environ.get("OVERLAP_CAPS_MB", "0.25,1,5,25,100,100000").split(",")]
    prios = os.environ.get("OVERLAP_PRIORITIES", "normal,high").split(",")
    for cap, prio in [(c, q) for c in caps for q in prios]:
        comm = comm_streams[prio]
        red = Reducer(grads, min(cfg["first_cap"], cap), cap)

        def overlapped():
            red.prepare()
            backward(red)

        def serial():
            backward(None)
            red.sync_gradients(divisor, D.DDP_ALGO_FUSED, D.DDP_SYNC_IN_PLACE, 1.0, compute)

        t_ov = timed(overlapped, reps)
        t_se = timed(serial, reps)
        t_comm = timed(lambda: red.sync_gradients(divisor, D.DDP_ALGO_FUSED, D.DDP_SYNC_IN_PLACE, 1.0, compute), reps)
        print(json.dumps({"overlap": args.config, "p": cfg["p"], "bucket_cap_mb": cap / (1 << 20),
                          "comm_stream_priority": prio,
                          "buckets": len(red.buckets), "n_tok": n_tok,
                          "backward_ms": round(t_bwd, 4), "backward_tflops": round(flops / (t_bwd / 1e3) / 1e12, 1),
                          "sync_alone_ms": round(t_comm, 4), "overlapped_ms": round(t_ov, 4),
                          "serial_ms": round(t_se, 4), "exposed_ms": round(t_ov - t_bwd, 4),
                          "hidden_frac": (round(1 - (t_ov - t_bwd) / (t_se - t_bwd), 3)
                                          if t_se - t_bwd > 0.05 * t_comm else None)}), flush=True)
        red.destroy()


def main():
    args = parse_args()
    ranks = Ranks()
    try:
        if args.sweep:
            run_sweep(args, ranks)
        elif args.overlap:
            run_overlap(args, ranks)
        elif args.impl == "reference":
            run_reference(args, ranks)
        else:
            run_ours(args, ranks)
    finally:
        ranks.close()


if __name__ == "__main__":
    main()
