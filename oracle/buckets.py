"""Bucket assignment, flatten/unflatten and broadcast coalescing (oracle; test infrastructure).

Sources (titles and sections of the pages):
  * "PyTorch DDP Deep Dive", Part 1, "What _ddp_init_helper actually does":
    buckets are computed by byte size, handed to the Reducer reversed so that
    bucket 0 holds the parameters whose gradients are ready first in backward,
    and the first bucket may have a smaller cap (1 MB by default).
  * Same page, Part 3, DDPOptimizer's compile_fn: the walk over the graph is in
    reverse order; a new bucket opens once the current one reaches its cap, the
    first bucket's cap being first_bucket_cap.
  * "Data parallelism", "Overlapping communication with the backward pass":
    ~25 MB buckets, parameters assigned in roughly the reverse of model order.
  * "PyTorch DDP Deep Dive", Part 2 backward, mark_variable_ready: each bucket
    holds one flat gradients tensor; each parameter owns a slice, filled by a
    copy that may pre-divide by the world size; finalize_backward copies the
    reduced flat tensor back into the per-parameter gradients.
  * Same page, Part 2 forward, the annotated trace: _broadcast_coalesced packs
    tensors into buckets of at most 250 * 1024 * 1024 bytes, flattens each,
    broadcasts it from the root, unflattens and copies back.

Readings where the pages leave a step open:
  * Walk order "reversed" (default): walk tensors from the last registered to
    the first; bucket 0 (the first to fire) gets first_cap. "registration":
    walk in registration order with bucket 0 capped at first_cap, then reverse
    the list of buckets (members keep registration order).
  * A bucket closes as soon as its byte size is >= its cap, tested after adding
    a tensor; tensors are never split, so a bucket may exceed its cap by its
    last tensor. No empty bucket is produced.
  * Inside a bucket tensors lie in walk order; offsets are exclusive prefix sums.
  * Broadcast coalescing: tensors in the given order; a new bucket starts when
    adding the next tensor would take the current one over the cap (a tensor
    larger than the cap travels alone).
"""
from __future__ import annotations

import numpy as np

MiB = 1024 * 1024


def assign_buckets(numel: list[int], elem_size: int, first_cap_bytes: int, cap_bytes: int,
                   order: str = "reversed") -> list[list[int]]:
    """Buckets as lists of tensor indices, bucket 0 first to be reduced."""
    k = len(numel)
    if order == "reversed":
        walk = list(range(k - 1, -1, -1))
    elif order == "registration":
        walk = list(range(k))
    else:
        raise ValueError(order)
    buckets: list[list[int]] = []
    current: list[int] = []
    size = 0
    for t in walk:
        current.append(t)
        size += numel[t] * elem_size
        cap = first_cap_bytes if not buckets else cap_bytes
        if size >= cap:
            buckets.append(current)
            current, size = [], 0
    if current:
        buckets.append(current)
    if order == "registration":
        buckets.reverse()
    return buckets


def bucket_layout(numel: list[int], buckets: list[list[int]]):
    """Per tensor: bucket index and element offset inside it; per bucket: element count."""
    bucket_of = [-1] * len(numel)
    offset = [0] * len(numel)
    bucket_numel = []
    for b, members in enumerate(buckets):
        pos = 0
        for t in members:
            bucket_of[t] = b
            offset[t] = pos
            pos += numel[t]
        bucket_numel.append(pos)
    return bucket_of, offset, bucket_numel


def flatten(grads: list[np.ndarray], members: list[int], offset: list[int], n: int,
            predivide: float = 1.0) -> np.ndarray:
    """One replica's flat bucket: grads[t] copied to [offset[t], offset[t]+numel).
    With predivide != 1 each element is divided by it during the copy (in the
    gradients' own precision)."""
    dt = grads[members[0]].dtype if members else np.float32
    flat = np.zeros(n, dtype=dt)
    for t in members:
        g = grads[t].reshape(-1)
        if predivide != 1.0:
            g = g / dt.type(predivide)
        flat[offset[t]:offset[t] + g.size] = g
    return flat


def unflatten(flat: np.ndarray, members: list[int], offset: list[int], numel: list[int]) -> dict:
    """The per-tensor slices of a flat bucket, as copies."""
    return {t: flat[offset[t]:offset[t] + numel[t]].copy() for t in members}


def coalesce(nbytes: list[int], cap_bytes: int = 250 * MiB) -> list[list[int]]:
    """Group tensors (in order) into broadcast buckets of at most cap_bytes."""
    groups: list[list[int]] = []
    current: list[int] = []
    size = 0
    for t, nb in enumerate(nbytes):
        if current and size + nb > cap_bytes:
            groups.append(current)
            current, size = [], 0
        current.append(t)
        size += nb
    if current:
        groups.append(current)
    return groups
