"""Python binding of libddp_ring.so: bucketed ring all-reduce over p simulated
ranks in one GPU's memory (the hot path of PyTorch DDP's Reducer).

Argument marshalling only: every function has the name of a C entry point in
include/ddp_ring.h, turns tensors / lists into pointer and size arrays, calls
it, and raises DDPError on a non-zero status. All work on the data runs in the
library's CUDA kernels; torch provides device memory and streams.

Pointers may be given as torch tensors (their data_ptr) or plain ints. A
stream may be a torch.cuda.Stream, an int handle, or None for torch's current
stream. dtype may be DDP_FLOAT32 / DDP_BFLOAT16 or torch.float32 / torch.bfloat16.
"""
from __future__ import annotations

import ctypes
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libddp_ring.so")

# ddp_status
DDP_OK, DDP_ERR_ARG, DDP_ERR_DTYPE, DDP_ERR_NOT_DIVISIBLE, DDP_ERR_ALIGN = 0, 1, 2, 3, 4
DDP_ERR_NOMEM, DDP_ERR_CUDA, DDP_ERR_TIMEOUT, DDP_ERR_STATE = 5, 6, 7, 8
# ddp_dtype
DDP_FLOAT32, DDP_BFLOAT16 = 0, 1
# ddp_algo
DDP_ALGO_FUSED, DDP_ALGO_RING_STEPS, DDP_ALGO_FUSED_LDST, DDP_ALGO_FUSED_TMA = 0, 1, 2, 3
DDP_ALGO_RECURSIVE_DOUBLING, DDP_ALGO_RABENSEIFNER, DDP_ALGO_TREE = 4, 5, 6
# ddp_own
DDP_OWN_RANK, DDP_OWN_RING = 0, 1
# ddp_border
DDP_ORDER_REVERSED, DDP_ORDER_REGISTRATION = 0, 1
# flags of ddp_allreduce_ex
DDP_FLAG_ROUND_EACH_HOP = 1
# ddp_sync_mode
DDP_SYNC_FLATTEN, DDP_SYNC_IN_PLACE = 0, 1
# ddp_op
DDP_OP_ALLREDUCE, DDP_OP_REDUCE_SCATTER, DDP_OP_ALLGATHER, DDP_OP_BROADCAST = 0, 1, 2, 3
DDP_MAX_P = 256

_c_i32, _c_i64, _c_f32, _c_vp = ctypes.c_int32, ctypes.c_int64, ctypes.c_float, ctypes.c_void_p
_P_i64 = ctypes.POINTER(ctypes.c_int64)
_P_i32 = ctypes.POINTER(ctypes.c_int32)
_P_vp = ctypes.POINTER(ctypes.c_void_p)

_SIGS = {
    "ddp_bucket_assign": [_c_i32, _P_i64, _c_i32, _c_i64, _c_i64, _c_i32, _P_i32, _P_i32, _P_i64, _P_i32,
                          _P_i32, _P_i64],
    "ddp_bucket_flatten": [_c_i32, _c_i32, _P_vp, _P_i64, _P_i64, _P_vp, _c_i32, _c_f32, _c_vp],
    "ddp_bucket_unflatten": [_c_i32, _c_i32, _P_vp, _P_i64, _P_i64, _P_vp, _c_i32, _c_vp],
    "ddp_allreduce": [_P_vp, _c_i32, _c_i64, _c_i32, _c_f32, _c_i32, _c_vp],
    "ddp_allreduce_persistent": [_P_vp, _c_i32, _c_i64, _c_i32, _c_f32, _c_i64, _c_i32, _c_i32, _c_vp, _c_vp],
    "ddp_allreduce_ex": [_P_vp, _c_i32, _c_i64, _c_i32, _c_f32, _c_i32, ctypes.c_uint32, _c_vp],
    "ddp_reduce_scatter": [_P_vp, _P_vp, _c_i32, _c_i64, _c_i32, _c_f32, _c_i32, _c_i32, _c_vp],
    "ddp_allgather": [_P_vp, _P_vp, _c_i32, _c_i64, _c_i32, _c_i32, _c_i32, _c_vp],
    "ddp_bucket_allreduce": [_c_i32, _c_i32, _P_vp, _P_i64, _P_i64, _c_i32, _c_f32, _c_vp],
    "ddp_reducer_create": [ctypes.POINTER(_c_vp), _c_i32, _c_i32, _P_vp, _P_i64, _c_i32, _c_i64, _c_i64, _c_i32],
    "ddp_reducer_num_buckets": [_c_vp],
    "ddp_reducer_staged": [_c_vp],
    "ddp_reducer_bucket": [_c_vp, _c_i32, _P_i64, _P_vp],
    "ddp_reducer_sync": [_c_vp, _c_f32, _c_f32, _c_i32, _c_i32, _c_vp],
    "ddp_reducer_destroy": [_c_vp],
    "ddp_reducer_set_buffers": [_c_vp, _c_i32, _P_vp, _P_i64, _c_i32],
    "ddp_reducer_step": [_c_vp, _c_f32, _c_vp],
    "ddp_reducer_set_comm_blocks": [_c_vp, _c_i32],
    "ddp_reducer_prepare": [_c_vp],
    "ddp_reducer_mark_ready": [_c_vp, _c_i32, _c_f32, _c_vp, _c_vp, _P_i32],
    "ddp_reducer_observed": [_c_vp, _P_i32],
    "ddp_reducer_rebuild": [_c_vp, _P_i32],
    "ddp_bucket_assign_order": [_c_i32, _P_i64, _c_i32, _c_i64, _c_i64, _P_i32, _P_i32, _P_i32, _P_i64, _P_i32,
                                _P_i32, _P_i64],
    "ddp_reduce_scatter_noalloc": [_P_vp, _P_vp, _c_i32, _c_i64, _c_i32, _c_f32, _c_i32, _c_vp],
    "ddp_broadcast": [_P_vp, _c_i32, _c_i64, _c_i32, _c_i32, _c_vp],
    "ddp_broadcast_coalesced": [_c_i32, _c_i32, _P_vp, _P_i64, _c_i32, _c_i64, _c_i32, _c_vp],
    "ddp_ring_create": [ctypes.POINTER(_c_vp), _c_i32, _P_vp, _P_vp, _c_i32, _c_i64, _c_i32, _c_f32, _c_i32,
                        _c_i32, _c_vp],
    "ddp_ring_num_steps": [_c_vp],
    "ddp_ring_steps_done": [_c_vp],
    "ddp_ring_step": [_c_vp],
    "ddp_ring_workspace": [_c_vp, ctypes.POINTER(_c_vp), _P_i64],
    "ddp_ring_bytes_sent": [_c_vp, _c_i32, _P_i64],
    "ddp_ring_sync": [_c_vp],
    "ddp_ring_destroy": [_c_vp],
    "ddp_device_error": [_c_vp, _P_i32],
    "ddp_kernel_launches": [],
    "ddp_last_error": [],
    "ddp_status_string": [_c_i32],
}
_RESTYPES = {"ddp_reducer_observed": _c_i32, "ddp_reducer_num_buckets": _c_i32, "ddp_reducer_staged": _c_i32, "ddp_ring_num_steps": _c_i32, "ddp_ring_steps_done": _c_i32, "ddp_kernel_launches": _c_i64,
             "ddp_last_error": ctypes.c_char_p, "ddp_status_string": ctypes.c_char_p}

_lib = None


class DDPError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{status_string(status)}: {message}")
        self.status = status


def lib() -> ctypes.CDLL:
    """The loaded library. Fails loudly if it has not been built: there is no fallback."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is not built; run ring_all_reduce_ddp_gb300.build.build_library()")
        L = ctypes.CDLL(LIB_PATH)
        for name, args in _SIGS.items():
            fn = getattr(L, name)
            fn.argtypes = args
            fn.restype = _RESTYPES.get(name, _c_i32)
        _lib = L
    return _lib


def exported_symbols() -> list[str]:
    return sorted(_SIGS)


def status_string(s: int) -> str:
    return lib().ddp_status_string(int(s)).decode()


def _check(rc: int):
    if rc != DDP_OK:
        raise DDPError(rc, lib().ddp_last_error().decode())


def _ptr(x) -> int:
    """A device address: an int is passed through (the caller vouches for it);
    a tensor must be a contiguous device tensor, since the library sees only
    its first byte and its element count."""
    if x is None:
        return 0
    if isinstance(x, int):
        return x
    if not x.is_cuda:
        raise ValueError("tensors passed to the library must live on a CUDA device")
    if not x.is_contiguous():
        raise ValueError("tensors passed to the library must be contiguous")
    return int(x.data_ptr())


def _ptrs(seq):
    """A ctypes array of pointers (passed through if it already is one)."""
    if isinstance(seq, ctypes.Array):
        return seq
    arr = (ctypes.c_void_p * max(1, len(seq)))()
    for i, x in enumerate(seq):
        arr[i] = _ptr(x)
    return arr


def _i64s(seq):
    if isinstance(seq, ctypes.Array):
        return seq
    arr = (ctypes.c_int64 * max(1, len(seq)))()
    for i, x in enumerate(seq):
        arr[i] = int(x)
    return arr


def _stream(s) -> int:
    if s is None:
        import torch
        return int(torch.cuda.current_stream().cuda_stream)
    if isinstance(s, int):
        return s
    return int(s.cuda_stream)


def _dtype(dt) -> int:
    if isinstance(dt, int):
        return dt
    import torch
    if dt == torch.float32:
        return DDP_FLOAT32
    if dt == torch.bfloat16:
        return DDP_BFLOAT16
    raise DDPError(DDP_ERR_DTYPE, f"unsupported dtype {dt}")


# ------------------------------------------------------------------ buckets
def ddp_bucket_assign(numel, elem_size: int, first_bucket_cap_bytes: int, bucket_cap_bytes: int,
                      order: int = DDP_ORDER_REVERSED) -> dict:
    """Returns {'buckets': [[tensor indices in walk order] per bucket], 'bucket_of',
    'offset', 'bucket_numel'}."""
    k = len(numel)
    nb = ctypes.c_int32(0)
    bucket_of = (ctypes.c_int32 * max(1, k))()
    offset = (ctypes.c_int64 * max(1, k))()
    bptr = (ctypes.c_int32 * (k + 1))()
    btens = (ctypes.c_int32 * max(1, k))()
    bnumel = (ctypes.c_int64 * max(1, k))()
    _check(lib().ddp_bucket_assign(k, _i64s(numel), elem_size, first_bucket_cap_bytes, bucket_cap_bytes,
                                   order, ctypes.byref(nb), bucket_of, offset, bptr, btens, bnumel))
    B = nb.value
    buckets = [[btens[i] for i in range(bptr[b], bptr[b + 1])] for b in range(B)]
    return {"buckets": buckets, "bucket_of": list(bucket_of)[:k], "offset": list(offset)[:k],
            "bucket_numel": list(bnumel)[:B]}


def ddp_bucket_assign_order(numel, elem_size: int, first_bucket_cap_bytes: int, bucket_cap_bytes: int,
                            walk) -> dict:
    """Buckets along an explicit walk (first-ready first); same result dict as ddp_bucket_assign."""
    k = len(numel)
    nb = ctypes.c_int32(0)
    bucket_of = (ctypes.c_int32 * max(1, k))()
    offset = (ctypes.c_int64 * max(1, k))()
    bptr = (ctypes.c_int32 * (k + 1))()
    btens = (ctypes.c_int32 * max(1, k))()
    bnumel = (ctypes.c_int64 * max(1, k))()
    w = (ctypes.c_int32 * max(1, k))(*[int(x) for x in walk])
    _check(lib().ddp_bucket_assign_order(k, _i64s(numel), elem_size, first_bucket_cap_bytes, bucket_cap_bytes, w,
                                         ctypes.byref(nb), bucket_of, offset, bptr, btens, bnumel))
    B = nb.value
    buckets = [[btens[i] for i in range(bptr[b], bptr[b + 1])] for b in range(B)]
    return {"buckets": buckets, "bucket_of": list(bucket_of)[:k], "offset": list(offset)[:k],
            "bucket_numel": list(bnumel)[:B]}


def ddp_bucket_flatten(grads, numel, offset, bucket, dtype=DDP_FLOAT32, predivide: float = 1.0, stream=None):
    """grads: p lists of k tensors (or a flat list of p*k pointers, replica-major);
    bucket: p flat buckets."""
    p = len(bucket)
    k = len(numel)
    flat = [g for row in grads for g in row] if grads and isinstance(grads[0], (list, tuple)) else list(grads)
    _check(lib().ddp_bucket_flatten(p, k, _ptrs(flat), _i64s(numel), _i64s(offset), _ptrs(bucket),
                                    _dtype(dtype), float(predivide), _stream(stream)))


def ddp_bucket_unflatten(bucket, numel, offset, grads, dtype=DDP_FLOAT32, stream=None):
    p = len(bucket)
    k = len(numel)
    flat = [g for row in grads for g in row] if grads and isinstance(grads[0], (list, tuple)) else list(grads)
    _check(lib().ddp_bucket_unflatten(p, k, _ptrs(bucket), _i64s(numel), _i64s(offset), _ptrs(flat),
                                      _dtype(dtype), _stream(stream)))


# -------------------------------------------------------------- collectives
def ddp_allreduce(bufs, n: int, dtype=DDP_FLOAT32, divisor: float = 1.0, algo: int = DDP_ALGO_FUSED,
                  stream=None):
    _check(lib().ddp_allreduce(_ptrs(bufs), len(bufs), int(n), _dtype(dtype), float(divisor), algo,
                               _stream(stream)))


def ddp_allreduce_ex(bufs, n: int, dtype=DDP_FLOAT32, divisor: float = 1.0, algo: int = DDP_ALGO_FUSED,
                     flags: int = 0, stream=None):
    _check(lib().ddp_allreduce_ex(_ptrs(bufs), len(bufs), int(n), _dtype(dtype), float(divisor), algo,
                                  int(flags), _stream(stream)))


def ddp_allreduce_persistent(bufs, n: int, dtype=DDP_FLOAT32, divisor: float = 1.0, timeout_ns: int = 0,
                             fault_rank: int = -1, fault_step: int = 0, status=None, stream=None):
    """status: None or a device int32 tensor of 4 words (zeroed and written by the call)."""
    _check(lib().ddp_allreduce_persistent(_ptrs(bufs), len(bufs), int(n), _dtype(dtype), float(divisor),
                                          int(timeout_ns), int(fault_rank), int(fault_step), _ptr(status),
                                          _stream(stream)))


def ddp_reduce_scatter(ins, outs, n: int, dtype=DDP_FLOAT32, divisor: float = 1.0, own: int = DDP_OWN_RANK,
                       algo: int = DDP_ALGO_FUSED, stream=None):
    _check(lib().ddp_reduce_scatter(_ptrs(ins), _ptrs(outs), len(ins), int(n), _dtype(dtype), float(divisor),
                                    own, algo, _stream(stream)))


def ddp_reduce_scatter_noalloc(ins, outs, n: int, dtype=DDP_FLOAT32, divisor: float = 1.0,
                               own: int = DDP_OWN_RANK, stream=None):
    """The literal ring reduce-scatter with its partials in the library's fixed
    scratch array: for callers that cannot allocate device memory mid-step."""
    _check(lib().ddp_reduce_scatter_noalloc(_ptrs(ins), _ptrs(outs), len(ins), int(n), _dtype(dtype),
                                            float(divisor), own, _stream(stream)))


def ddp_allgather(ins, outs, m: int, dtype=DDP_FLOAT32, own: int = DDP_OWN_RANK, algo: int = DDP_ALGO_FUSED,
                  stream=None):
    _check(lib().ddp_allgather(_ptrs(ins), _ptrs(outs), len(ins), int(m), _dtype(dtype), own, algo,
                               _stream(stream)))


def ddp_broadcast(bufs, nbytes: int, root: int = 0, algo: int = DDP_ALGO_FUSED, stream=None):
    _check(lib().ddp_broadcast(_ptrs(bufs), len(bufs), int(nbytes), int(root), algo, _stream(stream)))


def ddp_broadcast_coalesced(tensors, nbytes, root: int = 0, bucket_cap_bytes: int = 0,
                            algo: int = DDP_ALGO_FUSED, stream=None, p: int | None = None):
    """tensors: p lists of k tensors, a flat replica-major list of p*k pointers,
    or (with p given) a prebuilt ctypes pointer array."""
    k = len(nbytes)
    if isinstance(tensors, ctypes.Array):
        flat = tensors
    elif tensors and isinstance(tensors[0], (list, tuple)):
        p = len(tensors)
        flat = [t for row in tensors for t in row]
    else:
        p = len(tensors) // max(1, k)
        flat = list(tensors)
    _check(lib().ddp_broadcast_coalesced(p, k, _ptrs(flat), _i64s(nbytes), int(root), int(bucket_cap_bytes),
                                         algo, _stream(stream)))


def ddp_bucket_allreduce(grads, numel, offset, dtype=DDP_FLOAT32, divisor: float = 1.0, stream=None):
    """One bucket's all-reduce straight on the gradients. grads: p lists of the
    bucket's k tensors (walk order), or a flat replica-major list of p*k pointers."""
    k = len(numel)
    if grads and isinstance(grads[0], (list, tuple)):
        p = len(grads)
        flat = [g for row in grads for g in row]
    else:
        p = len(grads) // max(1, k)
        flat = list(grads)
    _check(lib().ddp_bucket_allreduce(p, k, _ptrs(flat), _i64s(numel), _i64s(offset), _dtype(dtype),
                                      float(divisor), _stream(stream)))


class DDPReducer:
    """ddp_reducer_create / sync / destroy: a whole gradient synchronisation per call."""

    def __init__(self, grads, first_bucket_cap_bytes: int = 1 << 20, bucket_cap_bytes: int = 25 << 20,
                 order: int = DDP_ORDER_REVERSED):
        self.p = len(grads)
        self.k = len(grads[0])
        self.dtype = _dtype(grads[0][0].dtype)
        numel = [g.numel() for g in grads[0]]
        for r, row in enumerate(grads):  # one dtype and one shape list for every replica
            if len(row) != self.k or [g.numel() for g in row] != numel:
                raise ValueError(f"replica {r} does not have replica 0's tensor sizes")
            if any(g.dtype != grads[0][0].dtype for g in row):
                raise ValueError("all gradient tensors of a Reducer must share one dtype")
        h = ctypes.c_void_p(0)
        self._grads = _ptrs([g for row in grads for g in row])
        _check(lib().ddp_reducer_create(ctypes.byref(h), self.p, self.k, self._grads, _i64s(numel), self.dtype,
                                        int(first_bucket_cap_bytes), int(bucket_cap_bytes), int(order)))
        self.h = h

    def num_buckets(self) -> int:
        return lib().ddp_reducer_num_buckets(self.h)

    def staged(self) -> bool:
        """True if step() and the default in-place sync take the shared-memory staged form."""
        return lib().ddp_reducer_staged(self.h) == 1

    def bucket(self, b: int):
        """(element count, [p flat-buffer device pointers]) of bucket b."""
        n = ctypes.c_int64(0)
        flat = (ctypes.c_void_p * self.p)()
        _check(lib().ddp_reducer_bucket(self.h, int(b), ctypes.byref(n), flat))
        return n.value, [flat[r] for r in range(self.p)]

    def sync(self, divisor: float, algo: int = DDP_ALGO_FUSED, mode: int = DDP_SYNC_IN_PLACE,
             predivide: float = 1.0, stream=None):
        _check(lib().ddp_reducer_sync(self.h, float(divisor), float(predivide), int(algo), int(mode),
                                      _stream(stream)))

    def set_buffers(self, buffers, root: int = 0):
        """Attach the per-forward buffers (p lists of k tensors, replica-major)
        that ddp_reducer_step broadcasts from `root`; an empty list detaches."""
        k = len(buffers[0]) if buffers else 0
        if buffers and len(buffers) != self.p:
            raise ValueError(f"need buffers for {self.p} replicas, got {len(buffers)}")
        nbytes = [t.numel() * t.element_size() for t in buffers[0]] if k else []
        self._bufs = _ptrs([t for row in buffers for t in row]) if k else None
        _check(lib().ddp_reducer_set_buffers(self.h, k, self._bufs, _i64s(nbytes), int(root)))
        return sum(nbytes)

    def step(self, divisor: float, stream=None):
        """The attached buffers' broadcast and the in-place sync, one launch."""
        _check(lib().ddp_reducer_step(self.h, float(divisor), _stream(stream)))

    def set_comm_blocks(self, max_blocks: int):
        """Grid cap of the bucket launches mark_ready fires (0: one block per tile)."""
        _check(lib().ddp_reducer_set_comm_blocks(self.h, int(max_blocks)))

    def prepare(self):
        _check(lib().ddp_reducer_prepare(self.h))

    def mark_ready(self, tensor: int, divisor: float, ready_event=None, comm_stream=None) -> int:
        """Mark gradient `tensor` ready; returns how many buckets this fired.
        ready_event: a torch.cuda.Event (or raw handle) the comm stream waits on."""
        fired = ctypes.c_int32(0)
        ev = 0 if ready_event is None else (ready_event if isinstance(ready_event, int)
                                            else int(ready_event.cuda_event))
        _check(lib().ddp_reducer_mark_ready(self.h, int(tensor), float(divisor), ev, _stream(comm_stream),
                                            ctypes.byref(fired)))
        return fired.value

    def observed(self) -> list[int]:
        n = lib().ddp_reducer_observed(self.h, None)
        arr = (ctypes.c_int32 * max(1, n))()
        lib().ddp_reducer_observed(self.h, arr)
        return [arr[i] for i in range(n)]

    def rebuild(self, order=None):
        arr = None if order is None else (ctypes.c_int32 * len(order))(*[int(x) for x in order])
        _check(lib().ddp_reducer_rebuild(self.h, arr))

    def destroy(self):
        if self.h:
            _check(lib().ddp_reducer_destroy(self.h))
            self.h = None

    def __del__(self):
        try:
            self.destroy()
        except Exception:
            pass


# ------------------------------------------------------- literal schedule
class DDPRing:
    """ddp_ring_create / step / sync / destroy: the literal schedule, stepwise."""

    def __init__(self, op: int, ins, outs, n: int, dtype=DDP_FLOAT32, divisor: float = 1.0,
                 own: int = DDP_OWN_RANK, root: int = 0, stream=None):
        h = ctypes.c_void_p(0)
        self.p = len(ins)
        _check(lib().ddp_ring_create(ctypes.byref(h), op, _ptrs(ins), _ptrs(outs) if outs is not None else None,
                                     self.p, int(n), _dtype(dtype), float(divisor), own, int(root),
                                     _stream(stream)))
        self.h = h

    def num_steps(self) -> int:
        return lib().ddp_ring_num_steps(self.h)

    def steps_done(self) -> int:
        return lib().ddp_ring_steps_done(self.h)

    def step(self):
        _check(lib().ddp_ring_step(self.h))

    def workspace(self):
        ptr = ctypes.c_void_p(0)
        n = ctypes.c_int64(0)
        _check(lib().ddp_ring_workspace(self.h, ctypes.byref(ptr), ctypes.byref(n)))
        return (ptr.value or 0), n.value

    def bytes_sent(self, rank: int) -> int:
        b = ctypes.c_int64(0)
        _check(lib().ddp_ring_bytes_sent(self.h, int(rank), ctypes.byref(b)))
        return b.value

    def sync(self):
        _check(lib().ddp_ring_sync(self.h))

    def destroy(self):
        if self.h:
            _check(lib().ddp_ring_destroy(self.h))
            self.h = None

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.destroy()


def ddp_ring_create(op, ins, outs, n, dtype=DDP_FLOAT32, divisor=1.0, own=DDP_OWN_RANK, root=0, stream=None):
    return DDPRing(op, ins, outs, n, dtype, divisor, own, root, stream)


def ddp_device_error(stream=None) -> int:
    code = ctypes.c_int32(0)
    rc = lib().ddp_device_error(_stream(stream), ctypes.byref(code))
    if rc not in (DDP_OK, DDP_ERR_TIMEOUT):
        _check(rc)
    return code.value


def ddp_kernel_launches() -> int:
    return int(lib().ddp_kernel_launches())


def ddp_last_error() -> str:
    return lib().ddp_last_error().decode()
