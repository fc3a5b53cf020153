"""A Reducer for p simulated replicas: sequences the C-ABI calls of one
gradient synchronisation, the way DDP's Reducer does in backward.

"PyTorch DDP Deep Dive", Part 1 (buckets computed at construction, handed to
the Reducer in reverse) and Part 2 (each gradient is copied into its bucket
slice, a full bucket is all-reduced, finalize_backward copies the reduced flat
buckets back into the gradients); "Data parallelism", "Overlapping
communication with the backward pass" (the sum is divided by the number of
ranks, or, with unequal token counts, by the global count).

Only sequencing: every byte is moved and every sum is taken by the library's
kernels. Gradients become ready in reverse registration order, so buckets are
processed in index order (bucket 0 first).
"""
from __future__ import annotations

from . import (DDP_ALGO_FUSED, DDP_BFLOAT16, DDP_FLOAT32, DDP_ORDER_REVERSED, ddp_allreduce, ddp_bucket_assign,
               ddp_bucket_flatten, ddp_bucket_unflatten, ddp_broadcast_coalesced)

MiB = 1 << 20


class Reducer:
    def __init__(self, grads, first_bucket_cap_bytes: int = 1 * MiB, bucket_cap_bytes: int = 25 * MiB,
                 order: int = DDP_ORDER_REVERSED):
        """grads: p lists of k gradient tensors (same shapes and dtype on every
        replica, registration order)."""
        import torch
        self.p = len(grads)
        self.k = len(grads[0])
        self.grads = grads
        t0 = grads[0][0]
        self.torch_dtype = t0.dtype
        self.dtype = DDP_FLOAT32 if t0.dtype == torch.float32 else DDP_BFLOAT16
        self.esize = t0.element_size()
        self.numel = [g.numel() for g in grads[0]]
        self._caps = (first_bucket_cap_bytes, bucket_cap_bytes, order)
        plan = ddp_bucket_assign(self.numel, self.esize, *self._caps)
        self.plan = plan
        self.buckets = plan["buckets"]
        self.bucket_numel = plan["bucket_numel"]
        self.offset = plan["offset"]
        self.flat = [[torch.empty(n, dtype=t0.dtype, device=t0.device) for n in self.bucket_numel]
                     for _ in range(self.p)]
        # per bucket: the argument lists of flatten / allreduce / unflatten
        self._bucket_args = []
        for b, members in enumerate(self.buckets):
            numel = [self.numel[t] for t in members]
            offset = [self.offset[t] for t in members]
            g = [[grads[r][t] for t in members] for r in range(self.p)]
            flat = [self.flat[r][b] for r in range(self.p)]
            self._bucket_args.append((numel, offset, g, flat))

    def assign(self) -> bool:
        """Recompute the bucket assignment (host only); True if it is unchanged."""
        return ddp_bucket_assign(self.numel, self.esize, *self._caps)["buckets"] == self.buckets

    def sync_gradients(self, divisor: float, algo: int = DDP_ALGO_FUSED, predivide: float = 1.0,
                       stream=None, allreduce_events=None):
        """Flatten and all-reduce every bucket in order, then copy every bucket back.
        allreduce_events: optional list that receives (start, end) CUDA events
        recorded around each all-reduce on `stream`."""
        import torch
        for numel, offset, g, flat in self._bucket_args:
            ddp_bucket_flatten(g, numel, offset, flat, self.dtype, predivide, stream)
            if allreduce_events is not None:
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
            ddp_allreduce(flat, flat[0].numel(), self.dtype, divisor, algo, stream)
            if allreduce_events is not None:
                e1.record(stream)
                allreduce_events.append((e0, e1))
        for numel, offset, g, flat in self._bucket_args:
            ddp_bucket_unflatten(flat, numel, offset, g, self.dtype, stream)

    def algorithmic_bytes(self) -> dict:
        """Bytes each op must move per synchronisation: all-reduce p*M read +
        p*M written per bucket; flatten and unflatten the same again each."""
        M = sum(self.bucket_numel) * self.esize
        ar = 2 * self.p * M
        copies = 2 * (2 * self.p * M)
        return {"allreduce": ar, "flatten_unflatten": copies, "total": ar + copies}


def broadcast_buffers(buffers, root: int = 0, bucket_cap_bytes: int = 0, algo: int = DDP_ALGO_FUSED,
                      stream=None):
    """DDP's per-forward buffer sync: p lists of k buffer tensors, root's copied
    to every other replica ("PyTorch DDP Deep Dive", Part 2, _sync_buffers)."""
    nbytes = [t.numel() * t.element_size() for t in buffers[0]]
    ddp_broadcast_coalesced(buffers, nbytes, root, bucket_cap_bytes, algo, stream)
    return sum(nbytes)
