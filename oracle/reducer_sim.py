"""Bucket readiness and communication overlap, simulated (oracle; test infrastructure).

Sources (titles and sections of the pages):
  * "PyTorch DDP Deep Dive", Part 2 "Step 2: backward": mark_variable_ready
    decrements the bucket's pending count; mark_bucket_ready walks forward from
    next_bucket_ and reduces every contiguous bucket whose pending count is
    zero -- "buckets are reduced in sequence", a complete bucket waits for its
    turn. Part 2 forward: _rebuild_buckets rebuilds the buckets from the order
    in which gradients were observed to become ready.
  * "Data parallelism", "Overlapping communication with the backward pass":
    gradients appear from the last layer to the first; a bucket's all-reduce
    starts on a separate stream once all its gradients are ready; tiny buckets
    pay the latency many times, huge buckets start late and the last one sticks
    out past the end of the backward pass. Its ddp_step_time cell (marked "no
    overlap at all") costs t = end_bwd + 2(p-1) alpha + 2(p-1)/p * total * beta.
  * Same page, "Ring all-reduce, derived": one ring all-reduce of M bytes costs
    2(p-1) alpha + 2(p-1)/p M beta.

Readings where the pages leave a step open:
  * One communication stream: bucket b's all-reduce starts at the later of
    (the time its last gradient is ready, the end of bucket b-1's all-reduce)
    -- in-order firing makes the stream sequential in bucket index.
  * Exposed communication = max(0, end of the last all-reduce - end of backward).
"""
from __future__ import annotations

from .buckets import assign_buckets, bucket_layout
from .costs import ring_time


def fire_sequence(buckets: list[list[int]], ready_order: list[int]) -> list[tuple[int, int]]:
    """Replay mark_variable_ready for tensors in ready_order. Returns
    (index in ready_order of the call that fired it, bucket) for every bucket,
    in firing order. A tensor marked twice raises ValueError."""
    bucket_of = {}
    for b, members in enumerate(buckets):
        for t in members:
            bucket_of[t] = b
    pending = [len(m) for m in buckets]
    seen = set()
    nxt = 0
    fired = []
    for pos, t in enumerate(ready_order):
        if t in seen:
            raise ValueError(f"tensor {t} marked ready twice")
        seen.add(t)
        pending[bucket_of[t]] -= 1
        while nxt < len(buckets) and pending[nxt] == 0:  # mark_bucket_ready
            fired.append((pos, nxt))
            nxt += 1
    return fired


def overlap(ready_time: list[float], comm_time: list[float]) -> dict:
    """Bucket b is ready at ready_time[b] (all its gradients done) and its
    all-reduce takes comm_time[b]; all-reduces run one at a time in bucket
    order. Returns per-bucket start / end and the exposed communication
    against end_bwd = max(ready_time)."""
    start, end = [], []
    t = 0.0
    for b in range(len(ready_time)):
        s = max(ready_time[b], t)
        t = s + comm_time[b]
        start.append(s)
        end.append(t)
    end_bwd = max(ready_time) if ready_time else 0.0
    last = end[-1] if end else 0.0
    return {"start": start, "end": end, "end_bwd": end_bwd, "step": max(end_bwd, last),
            "exposed": max(0.0, last - end_bwd)}


def ddp_step_time(grads: list[tuple[int, float]], bucket_cap: int, p: int, alpha: float, beta: float,
                  first_cap: int | None = None) -> dict:
    """grads: (bytes, time the gradient is ready) per tensor, in registration
    order (backward produces them last-first). Buckets by the reversed walk
    with the given caps; each bucket's all-reduce is one ring all-reduce of its
    bytes. Returns the overlap() result plus the buckets."""
    nbytes = [g[0] for g in grads]
    buckets = assign_buckets(nbytes, 1, bucket_cap if first_cap is None else first_cap, bucket_cap)
    _, _, bsize = bucket_layout(nbytes, buckets)
    ready = [max(grads[t][1] for t in members) for members in buckets]
    comm = [ring_time(M, p, alpha, beta) for M in bsize]
    out = overlap(ready, comm)
    out["buckets"] = buckets
    return out


def rebuild(numel: list[int], elem_size: int, first_cap: int, cap: int, observed_order: list[int]):
    """Buckets rebuilt from the order in which gradients became ready: the walk
    follows observed_order (first ready first), bucket 0 gets the first cap, a
    bucket closes once it reaches its cap."""
    buckets, current, size = [], [], 0
    for t in observed_order:
        current.append(t)
        size += numel[t] * elem_size
        if size >= (first_cap if not buckets else cap):
            buckets.append(current)
            current, size = [], 0
    if current:
        buckets.append(current)
    return buckets
