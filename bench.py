#!/usr/bin/env python3
"""Benchmark of one DDP gradient-synchronisation step over p simulated replicas
held in one GPU's memory.

A step is one pass of the whole hot path on the workload's synthetic
gradients: bucket assignment (host), the per-forward coalesced broadcast of the
model's buffers from replica 0, and the gradient sync of every bucket. By
default (--mode in_place) the broadcast and the sync are ONE launch: every
bucket is flattened, ring-all-reduced and unflattened in a single pass over
the gradients, and the buffers are copied in the same grid. --mode flatten
runs the broadcast, then the three separate kernels per bucket.

Default workload: the ResNet-50-shaped gradient set (161 fp32 tensors, 25.6M
parameters) on p = 8 replicas, 1 MiB first bucket / 25 MiB buckets, averaged
by 1/8, plus the broadcast of its 159 BatchNorm buffers.

Prints ONE JSON line (rank 0). value = algorithmic bytes of all the step's ops
(all-reduce 2pM; in flatten mode also flatten 2pM and unflatten 2pM; broadcast
p * buffer bytes) over the device-timed step, in GB/s, summed over ranks. The
same line carries the dominant kernel's roofline over a separate pass of 64
back-to-back launches, the message-size / rank-count points of the fused
all-reduce (`sweep`) and the GPT-2 and Llama-1B gradient sets (`configs`).
--impl reference times the CPU oracle instead, on the same step.
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
# sources it was taken on (k_bucket.cu, common.cuh) are unchanged (checked by
# hash).
ROOFLINE_LAUNCHES = 64  # back-to-back launches of the dominant kernel timed for the roofline
NCU_TRAFFIC = {"kernel_sha256": "9bc41f2b30cbca65a7928e7c18642316fb3c61d2373a651de84977a612302484",
               "config": "resnet50",  # the workload the capture ran; other workloads report null
               "dram_bytes_per_algorithmic_byte": (818.093568 + 759.851264) / 1637.353280}  # ncu: read + write MB per launch


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
    ap.add_argument("--cpu-budget-s", type=float, default=8.0)
    ap.add_argument("--no-extras", action="store_true", help="leave out the sweep and configs fields")
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
    """Hash of the dominant kernel's sources: its file and the header that
    fixes its tile size and argument layout."""
    import hashlib
    h = hashlib.sha256()
    for f in ("k_bucket.cu", "common.cuh"):
        with open(os.path.join(ROOT, "ring_all_reduce_ddp_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


# --------------------------------------------------------------- CPU oracle
def oracle_inputs(cfg):
    """Host copies of the workload's inputs, from the seeded generator (not
    read from any device): per replica its gradients in registration order,
    and the per-forward buffers' bytes (None if the workload has none)."""
    import numpy as np

    from synth import workloads as W
    numel = W.numels(cfg)
    starts = W.tensor_starts(cfg)
    grads = [[W.host_values(cfg, r, np.arange(starts[t], starts[t] + numel[t])) for t in range(len(numel))]
             for r in range(cfg["p"])]
    bufs = W.buffer_set_host(cfg) if cfg.get("buffers") else None
    return grads, bufs


def oracle_step_bytes(cfg, frac: float = 1.0) -> int:
    """Algorithmic bytes of one step, counted as the GPU arm counts them: the
    sync reads and writes every replica's gradients once (2pM), the broadcast
    reads the root's buffers once and writes the p - 1 others (p B). With
    frac < 1, the leading frac of every bucket (see oracle_step)."""
    from oracle import buckets as ob
    from synth import workloads as W
    numel = W.numels(cfg)
    es, p = W.esize(cfg), cfg["p"]
    plan = ob.assign_buckets(numel, es, cfg["first_cap"], cfg["cap"])
    _, _, bnumel = ob.bucket_layout(numel, plan)
    n = sum(bnumel) if frac >= 1 else sum(max(p, int(x * frac)) for x in bnumel)
    buf = sum(x.size for x in W.buffer_set_host(cfg, p=1)[0]) if cfg.get("buffers") and p > 1 else 0
    return 2 * p * n * es + p * buf


def oracle_step(cfg, grads, bufs, frac: float = 1.0):
    """One step of the path in the oracle, as it stands: bucket assignment,
    the coalesced broadcast of the buffers from replica 0, and for every bucket
    flatten, literal ring all-reduce and unflatten. With frac < 1 (a timing
    sample when the whole step would take too long) each bucket's all-reduce
    runs on its leading frac of elements and nothing is unflattened."""
    from oracle import buckets as ob
    from oracle import ring as orc
    from synth import workloads as W
    numel = W.numels(cfg)
    p = cfg["p"]
    plan = ob.assign_buckets(numel, W.esize(cfg), cfg["first_cap"], cfg["cap"])
    _, offset, bnumel = ob.bucket_layout(numel, plan)
    if bufs is not None:
        orc.broadcast_coalesced(bufs, 0)
    Dv = W.divisor(cfg)
    for b, members in enumerate(plan):
        flats = [ob.flatten(grads[r], members, offset, bnumel[b]) for r in range(p)]
        if frac >= 1:
            outs, _ = orc.allreduce(flats, bnumel[b], Dv, cfg["dtype"])
            for r in range(p):
                ob.unflatten(outs[r], members, offset, numel)
        else:
            m = max(p, int(bnumel[b] * frac))
            orc.allreduce([f[:m] for f in flats], m, Dv, cfg["dtype"])


def oracle_baseline(cfg, budget_s: float):
    """The oracle's whole step on the host, single thread, timed step by step
    until the budget is used (at least one step). Inputs are made untimed."""
    grads, bufs = oracle_inputs(cfg)
    times = []
    while not times or sum(times) < budget_s:
        t0 = time.perf_counter()
        oracle_step(cfg, grads, bufs)
        times.append(time.perf_counter() - t0)
    nbytes = oracle_step_bytes(cfg)
    return {"value": round(nbytes * len(times) / sum(times) / 1e9, 4), "unit": UNIT, "cores": 1, "kind": "oracle",
            "ms_per_step": round(1e3 * statistics.mean(times), 1), "steps": len(times),
            "sample": (f"the whole step in the oracle, {len(times)} time(s): bucket assignment, coalesced "
                       f"broadcast of the buffers, flatten + literal ring all-reduce + unflatten of every bucket "
                       f"(all {cfg['p']} replicas, every element); single thread; bytes counted as the GPU "
                       f"arm counts them (2pM + pB)"),
            "host_cores_available": cores_used(), "cpu_model": cpu_model()}


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
    one_launch = mode == D.DDP_SYNC_IN_PLACE
    grads, arenas = W.make_grads(cfg, f"cuda:{dev}")
    bufs = W.buffer_set(cfg, f"cuda:{dev}") if cfg.get("buffers") else None
    red = Reducer(grads, cfg["first_cap"], cfg["cap"])
    bsync = BufferSync(bufs, 0) if bufs else None
    if bufs and one_launch:
        red.set_buffers(bufs, 0)
    divisor = W.divisor(cfg)
    stream = torch.cuda.current_stream()
    bc_algo = D.DDP_ALGO_RING_STEPS if args.algo == "ring_steps" else D.DDP_ALGO_FUSED
    buf_bytes = sum(bsync.nbytes) if bsync else 0
    esz = W.esize(cfg)

    def step(r=red):
        if not r.assign():  # a1: bucket assignment (host)
            raise RuntimeError("bucket assignment changed")
        if one_launch:      # a9 + a2-a8: buffer broadcast and in-place sync, one launch
            r.step(divisor, stream)
        else:
            if bsync:
                bsync(bc_algo, stream)
            r.sync_gradients(divisor, algo, mode, 1.0, stream)

    ab = red.algorithmic_bytes(mode)
    bc_bytes = p * buf_bytes if p > 1 else 0
    step_bytes = ab["total"] + bc_bytes
    for _ in range(max(args.warmup, 0)):
        step()
    torch.cuda.synchronize()
    ranks.barrier()

    sampler = ClockSampler(dev)
    sampler.start()
    time.sleep(0.3)
    launches0 = D.ddp_kernel_launches()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    ranks.barrier()
    w0 = time.time()
    e0.record(stream)
    for _ in range(args.steps):
        step()
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

    # Dominant kernel: the one-launch step (the piece-table kernel, in the form
    # ddp_reducer_staged names, over the gradient pieces and the buffers' copy
    # pieces). Its average duration is
    # taken over ROOFLINE_LAUNCHES launches back to back on its stream, events
    # around the whole run: each launch reads the gradients the one before it
    # wrote, 0.8 GB at the default workload, more than L2 holds.
    peak, peak_kind = peak_hbm()
    roof_launches = ROOFLINE_LAUNCHES
    kernel_bytes = ab["allreduce"] + (bc_bytes if one_launch else 0)

    def launch():
        if one_launch:
            red.step(divisor, stream)
        else:
            red.sync_gradients(divisor, algo, mode, 1.0, stream)

    for _ in range(3):
        launch()
    torch.cuda.synchronize()
    r0, r1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    r0.record(stream)
    for _ in range(roof_launches):
        launch()
    r1.record(stream)
    torch.cuda.synchronize()
    avg_us = 1e3 * r0.elapsed_time(r1) / roof_launches
    achieved = kernel_bytes / (avg_us / 1e6) / 1e9
    traffic = None
    if (NCU_TRAFFIC["kernel_sha256"] == kernel_sha() and NCU_TRAFFIC["config"] == args.config
            and one_launch and NCU_TRAFFIC["dram_bytes_per_algorithmic_byte"]):
        traffic = int(NCU_TRAFFIC["dram_bytes_per_algorithmic_byte"] * kernel_bytes)
    bucket_mb = [round(n * esz / 2 ** 20, 2) for n in red.bucket_numel]
    nb = len(red.buckets)
    table_kernel = ("k_bucket_table_staged (tiles staged in shared memory by bulk copies)" if red.staged()
                    else "k_bucket_allreduce_table (register fold)")
    kernel_name = (f"{table_kernel}: every bucket's flatten + ring-order all-reduce + unflatten and the "
                   "buffers' broadcast in one launch" if one_launch
                   else "flatten, fused all-reduce, unflatten per bucket (whole sync timed)")

    # The same step as two launches (coalesced broadcast, then the in-place
    # sync), for comparison with the one-launch form.
    two_launch = None
    if one_launch and bsync:
        for _ in range(3):
            bsync(bc_algo, stream)
            red.sync_gradients(divisor, algo, mode, 1.0, stream)
        torch.cuda.synchronize()
        r0.record(stream)
        for _ in range(roof_launches):
            bsync(bc_algo, stream)
            red.sync_gradients(divisor, algo, mode, 1.0, stream)
        r1.record(stream)
        torch.cuda.synchronize()
        two_launch = {"ms_per_step": round(r0.elapsed_time(r1) / roof_launches, 5), "steps": roof_launches,
                      "note": "ddp_broadcast_coalesced then ddp_reducer_sync(in place): two launches per step"}

    # End to end through the public API: every step copies every replica's
    # gradients in from pinned host memory, synchronises them and copies the
    # result out. Three device copies of the workload rotate, so step i+1's
    # copy-in (H2D stream) never waits for step i's sync: it only needs the
    # copy-out of step i-2, long done. Both link directions stay busy; the
    # step runs on the compute stream between them.
    NSETS = 3
    sets = [(arenas, red)]
    for _ in range(NSETS - 1):
        g_x, a_x = W.make_grads(cfg, f"cuda:{dev}")
        r_x = Reducer(g_x, cfg["first_cap"], cfg["cap"])
        if bufs and one_launch:
            r_x.set_buffers(bufs, 0)
        sets.append((a_x, r_x))
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
        step(red_k)
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

    # the same step body captured once as a CUDA graph and replayed: what host
    # launch overhead costs the eager step
    graph = None
    if one_launch and ranks.world == 1:
        cg = torch.cuda.CUDAGraph()
        with torch.cuda.graph(cg):
            red.step(divisor, None)
        for _ in range(3):
            cg.replay()
        torch.cuda.synchronize()
        k_g = max(roof_launches, min(args.steps, 2000))
        g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        g0.record(stream)
        for _ in range(k_g):
            cg.replay()
        g1.record(stream)
        torch.cuda.synchronize()
        graph = {"ms_per_step": round(g0.elapsed_time(g1) / k_g, 5), "steps": k_g,
                 "note": "the one-launch step replayed from a CUDA graph (bucket assignment stays on the host)"}
        del cg

    # the flatten form of the same step, for comparison (not the headline)
    other = None
    if one_launch:
        k2 = max(10, min(args.steps, 200))

        def flat_step():
            if bsync:
                bsync(bc_algo, stream)
            red.sync_gradients(divisor, algo, D.DDP_SYNC_FLATTEN, 1.0, stream)

        for _ in range(3):
            flat_step()
        torch.cuda.synchronize()
        g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        g0.record(stream)
        for _ in range(k2):
            flat_step()
        g1.record(stream)
        torch.cuda.synchronize()
        fl = red.algorithmic_bytes(D.DDP_SYNC_FLATTEN)["total"] + bc_bytes
        ms2 = g0.elapsed_time(g1) / k2
        other = {"mode": "broadcast, then flatten + all-reduce + unflatten per bucket", "ms_per_step": round(ms2, 5),
                 "gbs": round(fl / (ms2 / 1e3) / 1e9, 1), "steps": k2}

    extras = {}
    if one_launch and ranks.world == 1 and args.config == "resnet50" and not args.no_extras:
        del red, grads, arenas
        torch.cuda.empty_cache()
        extras["sweep"] = bench_sweep_points(peak)
        extras["configs"] = bench_config_points(peak)

    cpu = None
    if ranks.rank == 0 and ranks.world == 1 and not args.no_cpu_baseline:
        cpu = oracle_baseline(cfg, args.cpu_budget_s)

    line = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": ranks.world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": cfg["dtype"], "data": "synthetic",
        "config": {"workload": WORKLOAD_TEXT[args.config], "p": p, "buckets": nb, "bucket_mb": bucket_mb,
                   "buffer_bytes": buf_bytes, "algo": args.algo,
                   "sync": "in_place, one launch with the buffer broadcast" if one_launch else "flatten",
                   "divisor": divisor,
                   "l2": l2_note(sum(a.numel() * a.element_size() for a in host_in), dev),
                   "parallelism": f"replicas only: {ranks.world} independent GPU(s)"},
        "roofline": {"bound": "hbm", "kernel": kernel_name, "achieved": round(achieved, 1),
                     "peak": peak, "peak_kind": peak_kind, "unit": "GB/s", "frac": round(achieved / peak, 4),
                     "traffic": traffic, "algorithmic_bytes_per_launch": int(kernel_bytes),
                     "avg_launch_us": round(avg_us, 2), "event_timed_launches": roof_launches,
                     "timing": "CUDA events around the launches, back to back on the launching stream"},
        "allreduce_gbs": round(ab["allreduce"] / (avg_us / 1e6) / 1e9, 1),
        "buckets_per_s": round(nb * args.steps * ranks.world / (ms_max / 1e3), 1),
        "busbw_gbs": round(sum(n * esz for n in red_bucket_numel(cfg)) / (avg_us / 1e6) / 1e9 * 2 * (p - 1) / p, 1),
        "two_launch_form": two_launch,
        "flatten_form": other,
        "cuda_graph": graph,
        **extras,
        "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": launches, "clocks": clocks,
    }
    if ranks.rank == 0:
        print(json.dumps(line), flush=True)


def red_bucket_numel(cfg):
    """Elements of every bucket of the workload (the oracle's plan, which the
    library's equals: checked by the tests)."""
    from oracle import buckets as ob
    from synth import workloads as W
    numel = W.numels(cfg)
    _, _, bnumel = ob.bucket_layout(numel, ob.assign_buckets(numel, W.esize(cfg), cfg["first_cap"], cfg["cap"]))
    return bnumel


def make_flush():
    """An L2 flush: a 512 MiB write, then a 512 MiB read of another buffer, so
    the next launch starts with clean lines that belong to neither."""
    import torch
    wflush = torch.empty(512 << 20, dtype=torch.uint8, device="cuda")
    rflush = torch.ones(128 << 20, dtype=torch.float32, device="cuda")

    def flush():
        wflush.fill_(1)
        rflush.sum()
    return flush


def time_point(call, nsets, reps, batches, flush, graph=True):
    """Batches of launches call(0), call(1), ... (call(i) uses input copy
    i mod nsets), L2 flushed before each batch. Returns (seconds per launch:
    graph-replayed if graph else eager, eager seconds per launch, launches per
    batch, batches). A batch has up to `reps` launches, fewer when one launch
    is long (about 5 ms of work per batch is enough)."""
    import torch
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

    def batch():
        for i in range(nrep):
            call(i)

    def timed(run):
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
    if graph:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            batch()
        g.replay()
        torch.cuda.synchronize()
        t_graph = timed(g.replay)
        del g
    return (t_graph if t_graph is not None else t_eager), t_eager, nrep, nbat


def sweep_sets(p, n, with_outs, reps, out_elems=None):
    """Input copies for one sweep point: enough copies that no launch of a
    batch finds its inputs in L2 when one copy is under 2x L2 (at most 4 GiB
    of copies), values uniform on [-1, 1)."""
    import torch

    import synth
    l2 = torch.cuda.get_device_properties(0).L2_cache_size
    out_elems = out_elems or n
    set_bytes = p * n * 4 + (p * out_elems * 4 if with_outs else 0)
    nsets = 1
    if set_bytes < 2 * l2:
        nsets = max(1, min(reps, (4 << 30) // set_bytes))
    sets = []
    for _ in range(nsets):
        bufs = []
        for r in range(p):
            t = torch.empty(n, dtype=torch.float32, device="cuda")
            synth.fill_(t, "uniform", 1005, r)
            bufs.append(t)
        outs = [torch.empty(out_elems, dtype=torch.float32, device="cuda") for _ in range(p)] if with_outs else []
        sets.append((bufs, outs))
    return sets


def bench_sweep_points(peak, ps=(2, 8, 64), sizes_mib=(1, 25, 256), reps=20, batches=5):
    """The metric's two axes for the bench line: the fused all-reduce of one
    fp32 buffer of M MiB on each of p replicas, graph-replayed batches after an
    L2 flush (as --sweep times them)."""
    import torch

    import ring_all_reduce_ddp_gb300 as D
    flush = make_flush()
    out = []
    for p in ps:
        for mib in sizes_mib:
            M = mib << 20
            n = M // 4
            sets = sweep_sets(p, n, False, reps)
            call = lambda i, sets=sets, n=n, p=p: D.ddp_allreduce(sets[i % len(sets)][0], n, D.DDP_FLOAT32,
                                                                  float(p), D.DDP_ALGO_FUSED)
            t, t_eager, nrep, nbat = time_point(call, len(sets), reps, batches, flush)
            gbs = 2 * p * M / t / 1e9
            out.append({"op": "allreduce", "algo": "fused", "p": p, "bytes": M, "us": round(t * 1e6, 2),
                        "us_eager": round(t_eager * 1e6, 2), "gbs": round(gbs, 1), "frac": round(gbs / peak, 4),
                        "input_copies": len(sets), "reps": nrep, "batches": nbat})
            del sets
            torch.cuda.empty_cache()
    return {"timing": "CUDA graph of a batch of launches, L2 flushed before each batch, median of batches",
            "points": out}


def bench_config_points(peak, reps=20):
    """The other model-shaped gradient sets of the metric: GPT-2 small (fp32,
    token-count divisor) and Llama-1B (bf16, with its 64 per-forward buffers),
    each as the one-launch step, back-to-back launches timed by events."""
    import torch

    from ring_all_reduce_ddp_gb300.reducer import Reducer
    from synth import workloads as W
    out = {}
    for name in ("gpt2_small", "llama_1b"):
        cfg = W.CONFIGS[name]
        p = cfg["p"]
        grads, arenas = W.make_grads(cfg)
        red = Reducer(grads, cfg["first_cap"], cfg["cap"])
        buf_bytes = 0
        if cfg.get("buffers"):
            bufs = W.buffer_set(cfg)
            buf_bytes = red.set_buffers(bufs, 0)
        Dv = W.divisor(cfg)
        nbytes = red.algorithmic_bytes()["allreduce"] + p * buf_bytes
        for _ in range(3):
            red.step(Dv)
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        n_l = reps if name == "gpt2_small" else max(8, reps // 2)
        a.record()
        for _ in range(n_l):
            red.step(Dv)
        b.record()
        torch.cuda.synchronize()
        us = 1e3 * a.elapsed_time(b) / n_l
        gbs = nbytes / (us / 1e6) / 1e9
        out[name] = {"workload": WORKLOAD_TEXT[name], "p": p, "dtype": cfg["dtype"], "buckets": len(red.buckets),
                     "algorithmic_bytes": int(nbytes), "us": round(us, 2), "gbs": round(gbs, 1),
                     "frac": round(gbs / peak, 4), "buckets_per_s": round(len(red.buckets) / (us / 1e6), 1),
                     "launches": n_l}
        red.destroy()
        del red, grads, arenas
        torch.cuda.empty_cache()
    return out


# --------------------------------------------------------------- reference arm
def run_reference(args, ranks: Ranks):
    """The CPU oracle as it stands, on rank 0 only, on the GPU arm's step:
    bucket assignment, the coalesced broadcast of the buffers, flatten +
    literal ring all-reduce + unflatten of every bucket, all replicas, every
    element. If --steps + --warmup whole steps would take more than about
    two minutes, every step is the same sample of it instead: each bucket's
    all-reduce on its leading fraction of elements (same_config is then
    false). Inputs are generated once, outside the timed region."""
    if ranks.rank != 0:
        return
    from synth import workloads as W
    cfg = W.CONFIGS[args.config]
    p = cfg["p"]
    grads, bufs = oracle_inputs(cfg)
    t0 = time.perf_counter()
    oracle_step(cfg, grads, bufs)  # one whole step, untimed, sizes the run
    t_full = time.perf_counter() - t0
    budget = 120.0
    frac = min(1.0, budget / max(1e-9, (args.steps + args.warmup) * t_full))
    for _ in range(max(args.warmup, 0)):
        oracle_step(cfg, grads, bufs, frac)
    t_tot = 0.0
    for _ in range(args.steps):
        t0 = time.perf_counter()
        oracle_step(cfg, grads, bufs, frac)
        t_tot += time.perf_counter() - t0
    nbytes = oracle_step_bytes(cfg, frac) * args.steps
    value = nbytes / t_tot / 1e9
    ms_step = 1e3 * t_tot / max(args.steps, 1)
    if frac >= 1:
        desc = (f"the whole step in the oracle every step: bucket assignment, coalesced broadcast of the buffers, "
                f"flatten + literal ring all-reduce + unflatten of every bucket (p={p}, every element); "
                f"single thread; bytes counted as the GPU arm counts them (2pM + pB)")
    else:
        desc = (f"a sample of the step in the oracle every step: the buffers' broadcast and each bucket's literal "
                f"ring all-reduce on its leading {frac:.4f} of elements (p={p}); single thread")
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": UNIT, "n_gpus": ranks.world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": cfg["dtype"],
        "data": "synthetic",
        "config": {"workload": WORKLOAD_TEXT[args.config], "p": p, "algo": "oracle literal ring",
                   "same_config": frac >= 1, "sample_fraction": round(frac, 6)},
        "cpu_baseline": {"value": round(value, 4), "unit": UNIT, "kind": "oracle", "cores": 1, "sample": desc,
                         "ms_per_step": round(ms_step, 3), "host_cores_available": cores_used(),
                         "cpu_model": cpu_model()},
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
    flush = make_flush()

    for p in ps:
        for k in range(min_k, max_k + 1):
            M = 1024 * 4 ** k
            if p * M > 64 << 30:
                continue
            n = M // 4
            m = n // p
            with_outs = ops != "allreduce"
            sets = sweep_sets(p, n, with_outs, reps, max(n, p * m))
            nsets = len(sets)
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
                    # the persistent ring (a cooperative launch) is timed eagerly only
                    t, t_eager, nrep, nbat = time_point(call, nsets, reps, batches, flush,
                                                        graph=(an != "persistent"))
                    t_graph = t if an != "persistent" else None
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
    """Exposed communication against bucket cap and the comm kernels' grid,
    with readiness-driven firing.

    A synthetic backward walks the parameters last-registered first on the
    compute stream; each weight gradient costs two bf16 GEMMs with
    4 * numel * n_tok FLOPs in all (backward is about 4N FLOPs per token);
    after each gradient an event is recorded and the Reducer is told the
    gradient is ready, which launches every newly complete bucket's in-place
    all-reduce on a communication stream. A step ends when the compute stream
    has waited for the communication stream (the optimizer needs the reduced
    gradients). For each cap, comm-stream priority and grid cap of the bucket
    launches (0: one block per 2 KB tile; N > 0: N blocks striding over the
    tiles, so the all-reduces hold at most about N/9 SMs at p = 8): the backward alone,
    backward + overlapped sync (with the time the compute stream took inside
    it), and backward followed by the sync. One JSON line per point."""
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

    ready_events = [torch.cuda.Event() for _ in range(k)]

    def backward(red=None, comm=None):
        for t in range(k - 1, -1, -1):
            cols = (numel[t] + kdim - 1) // kdim
            if numel[t] >= 4096:  # 2 GEMMs: 2 * (2 * n_tok * kdim * cols) ~ 4 * numel * n_tok FLOPs
                torch.mm(x, w[:, :cols], out=y[:, :cols])
                torch.mm(x, w[:, :cols], out=y[:, :cols])
            if red is not None:
                ready_events[t].record(compute)
                red.mark_ready(t, divisor, ready_events[t], comm)

    def timed(fn, reps, comm=None):
        """Mean per step of (compute-stream time, time until both streams are done)."""
        def one():
            fn()
            c = torch.cuda.Event(enable_timing=True)
            c.record(compute)
            if comm is not None:
                compute.wait_stream(comm)
            return c
        for _ in range(3):
            one()
        torch.cuda.synchronize()
        ev = []
        for _ in range(reps):
            s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            s0.record(compute)
            c = one()
            s1.record(compute)
            ev.append((s0, c, s1))
        torch.cuda.synchronize()
        return (statistics.mean(a.elapsed_time(c) for a, c, _ in ev),
                statistics.mean(a.elapsed_time(b) for a, _, b in ev))

    reps = max(5, min(args.steps, 20))
    _, t_bwd = timed(lambda: backward(None), reps)
    flops = 4.0 * sum(n for n in numel if n >= 4096) * n_tok
    caps = [int(float(c) * (1 << 20)) for c in os.environ.get("OVERLAP_CAPS_MB", "1,5,25").split(",")]
    prios = os.environ.get("OVERLAP_PRIORITIES", "normal,high").split(",")
    blocks = [int(b) for b in os.environ.get("OVERLAP_COMM_BLOCKS", "0,24,48,96,192,384").split(",")]
    for cap in caps:
        red = Reducer(grads, min(cfg["first_cap"], cap), cap)
        _, t_comm = timed(lambda: red.sync_gradients(divisor, D.DDP_ALGO_FUSED, D.DDP_SYNC_IN_PLACE, 1.0, compute),
                          reps)

        def serial():
            backward(None)
            red.sync_gradients(divisor, D.DDP_ALGO_FUSED, D.DDP_SYNC_IN_PLACE, 1.0, compute)

        _, t_se = timed(serial, reps)
        for prio in prios:
            comm = comm_streams[prio]
            for nblk in blocks:
                red.set_comm_blocks(nblk)

                def overlapped():
                    red.prepare()
                    backward(red, comm)

                def fired_alone():  # the same bucket launches with no backward beside them
                    red.prepare()
                    comm.wait_stream(compute)
                    for t in range(k - 1, -1, -1):
                        red.mark_ready(t, divisor, None, comm)

                _, t_fire = timed(fired_alone, reps, comm)
                t_cmp, t_ov = timed(overlapped, reps, comm)
                exposed = t_ov - t_bwd
                print(json.dumps({"overlap": args.config, "p": cfg["p"], "bucket_cap_mb": cap / (1 << 20),
                                  "comm_stream_priority": prio, "comm_blocks": nblk,
                                  # 9 blocks of the per-bucket kernel fit on an SM at p = 8 fp32
                                  # (56 registers x 128 threads)
                                  "comm_sm_equivalent": round(nblk / 9, 1) if nblk else None,
                                  "buckets": len(red.buckets), "n_tok": n_tok,
                                  "backward_ms": round(t_bwd, 4),
                                  "backward_tflops": round(flops / (t_bwd / 1e3) / 1e12, 1),
                                  "sync_alone_ms": round(t_comm, 4), "fired_alone_ms": round(t_fire, 4),
                                  "serial_ms": round(t_se, 4),
                                  "overlapped_ms": round(t_ov, 4), "backward_in_overlap_ms": round(t_cmp, 4),
                                  "gemm_slowdown_ms": round(t_cmp - t_bwd, 4), "tail_ms": round(t_ov - t_cmp, 4),
                                  "exposed_ms": round(exposed, 4),
                                  "hidden_frac": round(1 - exposed / (t_se - t_bwd), 3) if t_se > t_bwd else None}),
                      flush=True)
        red.set_comm_blocks(0)
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
