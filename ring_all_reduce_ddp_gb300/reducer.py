"""The Reducer of p simulated replicas and the per-forward buffer sync, over
the library's native handles.

"PyTorch DDP Deep Dive", Part 1 (buckets computed at construction, handed to
the Reducer in reverse) and Part 2 (each gradient goes into its bucket slice,
a full bucket is all-reduced, finalize_backward copies the reduced buckets
back; the forward's _sync_buffers broadcasts the buffers from rank 0);
"Data parallelism", "Overlapping communication with the backward pass" (the
sum is divided by the number of ranks, or by the global token count).

Only sequencing and argument marshalling, done once at construction: every
byte is moved and every sum is taken by the library's kernels.
"""
from __future__ import annotations

import ctypes

from . import (DDP_ALGO_FUSED, DDP_ORDER_REVERSED, DDP_SYNC_IN_PLACE, DDPReducer, _check, _ptrs, _i64s,
               ddp_broadcast_coalesced, ddp_bucket_assign, ddp_bucket_assign_order, lib)

MiB = 1 << 20


class Reducer(DDPReducer):
    """A ddp_reducer over p lists of k gradient tensors (registration order),
    plus the bucket plan ddp_bucket_assign gives for the same arguments."""

    def __init__(self, grads, first_bucket_cap_bytes: int = 1 * MiB, bucket_cap_bytes: int = 25 * MiB,
                 order: int = DDP_ORDER_REVERSED):
        super().__init__(grads, first_bucket_cap_bytes, bucket_cap_bytes, order)
        self.grads = grads
        self.esize = grads[0][0].element_size()
        self.numel = [g.numel() for g in grads[0]]
        self._caps = (first_bucket_cap_bytes, bucket_cap_bytes, order)
        self._walk = None
        plan = ddp_bucket_assign(self.numel, self.esize, *self._caps)
        self.plan = plan
        self.buckets = plan["buckets"]
        self.bucket_numel = plan["bucket_numel"]
        self.offset = plan["offset"]
        assert self.num_buckets() == len(self.buckets)
        self._prepare_assign()

    def _prepare_assign(self):
        """The argument and result arrays of the per-step assignment call, made
        once, and the plan's CSR arrays to compare its result with."""
        k = len(self.numel)
        self._a_numel = _i64s(self.numel)
        self._a_nb = ctypes.c_int32(0)
        self._a_of = (ctypes.c_int32 * max(1, k))()
        self._a_off = (ctypes.c_int64 * max(1, k))()
        self._a_ptr = (ctypes.c_int32 * (k + 1))()
        self._a_tens = (ctypes.c_int32 * max(1, k))()
        self._a_bn = (ctypes.c_int64 * max(1, k))()
        self._a_walk = None if self._walk is None else (ctypes.c_int32 * max(1, k))(*[int(x) for x in self._walk])
        ptr, tens = [0], []
        for b in self.buckets:
            tens += b
            ptr.append(len(tens))
        self._want = (len(self.buckets), bytes((ctypes.c_int32 * (k + 1))(*ptr))[:4 * (len(self.buckets) + 1)],
                      bytes((ctypes.c_int32 * max(1, k))(*tens))[:4 * len(tens)])

    def assign(self) -> bool:
        """Recompute the bucket assignment (host only, ddp_bucket_assign or,
        after a rebuild, ddp_bucket_assign_order); True if it is unchanged."""
        k = len(self.numel)
        head = (k, self._a_numel, self.esize, self._caps[0], self._caps[1])
        tail = (ctypes.byref(self._a_nb), self._a_of, self._a_off, self._a_ptr, self._a_tens, self._a_bn)
        if self._a_walk is not None:
            _check(lib().ddp_bucket_assign_order(*head, self._a_walk, *tail))
        else:
            _check(lib().ddp_bucket_assign(*head, self._caps[2], *tail))
        nb = self._a_nb.value
        return (nb == self._want[0] and bytes(self._a_ptr)[:4 * (nb + 1)] == self._want[1]
                and bytes(self._a_tens)[:len(self._want[2])] == self._want[2])

    def rebuild(self, order=None):
        """Rebuild the buckets along `order`, or along the ready order observed
        since the last prepare(), and refresh the host-side plan."""
        walk = list(order) if order is not None else self.observed()
        super().rebuild(order)
        self._walk = walk
        plan = ddp_bucket_assign_order(self.numel, self.esize, self._caps[0], self._caps[1], walk)
        self.plan = plan
        self.buckets = plan["buckets"]
        self.bucket_numel = plan["bucket_numel"]
        self.offset = plan["offset"]
        assert self.num_buckets() == len(self.buckets)
        self._prepare_assign()

    def sync_gradients(self, divisor: float, algo: int = DDP_ALGO_FUSED, mode: int = DDP_SYNC_IN_PLACE,
                       predivide: float = 1.0, stream=None):
        self.sync(divisor, algo, mode, predivide, stream)

    def algorithmic_bytes(self, mode: int = DDP_SYNC_IN_PLACE) -> dict:
        """Bytes a synchronisation must move: the all-reduce reads p*M and writes
        p*M; in the flatten mode the copies in and out add 2*p*M each."""
        M = sum(self.bucket_numel) * self.esize
        ar = 2 * self.p * M
        copies = 0 if mode == DDP_SYNC_IN_PLACE else 2 * (2 * self.p * M)
        return {"allreduce": ar, "flatten_unflatten": copies, "total": ar + copies}


class BufferSync:
    """DDP's per-forward buffer sync: root's buffers copied to every other
    replica by ddp_broadcast_coalesced. Pointer tables are built once."""

    def __init__(self, buffers, root: int = 0, bucket_cap_bytes: int = 0):
        self.p = len(buffers)
        self.nbytes = [t.numel() * t.element_size() for t in buffers[0]]
        self._ptrs = _ptrs([t for row in buffers for t in row])
        self._nbytes = _i64s(self.nbytes)
        self.root = root
        self.cap = bucket_cap_bytes
        self.buffers = buffers

    def __call__(self, algo: int = DDP_ALGO_FUSED, stream=None) -> int:
        ddp_broadcast_coalesced(self._ptrs, self._nbytes, self.root, self.cap, algo, stream, p=self.p)
        return sum(self.nbytes)


def broadcast_buffers(buffers, root: int = 0, bucket_cap_bytes: int = 0, algo: int = DDP_ALGO_FUSED,
                      stream=None):
    """One-shot form of BufferSync."""
    return BufferSync(buffers, root, bucket_cap_bytes)(algo, stream)
