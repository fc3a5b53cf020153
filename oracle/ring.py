"""The two-pass ring all-reduce and its collectives, simulated literally (oracle; test infrastructure).

Sources (titles and sections of the pages):
  * "Collective Ops From Scratch", "Ring allreduce in two passes": split the
    tensor into N chunks; zero-pad to the next multiple of N and trim at the
    end. Reduce-scatter: at step s rank r sends chunk (r - s) mod N to rank
    r + 1, which accumulates it into its local copy; after N - 1 steps rank r
    owns the full sum of chunk (r + 1) mod N. All-gather: N - 1 more steps
    rotate the finished chunks. Same page, the code/main.py list: reduce_scatter
    pre-rotates the chunks so that rank r returns the sum of chunk r and raises
    ValueError when the element count is not divisible by the world size;
    broadcast is a doubling tree; all-gather is N - 1 rotations.
  * "Data parallelism", "Ring all-reduce, derived": the same two phases with
    steps k = 0 .. p - 2; in the all-gather rank r sends chunk (r + 1 - k) mod p
    and the receiver overwrites its copy. "The collective operations": an
    all-reduce is a reduce-scatter followed by an all-gather. "Overlapping
    communication with the backward pass": DDP divides the summed gradients by
    the number of ranks. "Why averaging gradients is exactly large-batch
    training": with unequal token counts, sum over tokens, sum the counts,
    divide once. Same section's neighbour "Ring all-reduce, derived": the naive
    algorithm sends everything to one rank, adds, sends the result back.

Readings where the pages leave a step open:
  * Chunk size cs = ceil(n / p); chunk c covers [c*cs, min(n, (c+1)*cs)); the
    zero padding sits at the tail of the last chunks and is trimmed.
  * All sends of a step happen at once: every payload is taken before any
    receiver adds (send-buffer semantics). The receiver computes
    local + received in the working precision (fp32; fp64 for fp64 inputs).
  * The division by D happens once, on the owner's finished chunk, as part of
    the last reduce-scatter step: y = fl(sum / D). With p == 1 there are no
    ring steps and the scale is the one step.
  * bf16 buffers: widened to fp32 working copies; all hops accumulate in fp32;
    the owner rounds fl32(sum / D) to bf16 once; the all-gather copies it.
  * reduce_scatter "rank" ownership (the torch contract): ring chunk label L
    stands for real chunk (L - 1) mod p, so real chunk c starts at rank
    (c + 1) mod p and ends, summed, on rank c. "ring" ownership: rank q gets
    chunk (q + 1) mod p, as pass 1 leaves it.
  * Byte counters count every payload at the buffer's element size, padding
    included (each reduce-scatter / all-reduce send is one cs-element chunk).
  * Per-hop bf16 rounding (hop_round=True, bf16 only): the variant in which
    partials travel as bf16, as a bf16 wire format would carry them: after
    every local + received the receiver rounds the fp32 sum to bf16 (nearest
    even); the owner then rounds fl32(sum / D) to bf16 as usual.
"""
from __future__ import annotations

import numpy as np

from .bf16 import bf16_to_f32, f32_to_bf16

_ESIZE = {"f32": 4, "bf16": 2, "f64": 8}


def chunk_size(n: int, p: int) -> int:
    """Elements per chunk after zero-padding n up to a multiple of p."""
    return -(-n // p) if n > 0 else 0


def chunk_bounds(n: int, p: int) -> list[tuple[int, int]]:
    """[start, end) of each chunk's real (unpadded) elements."""
    cs = chunk_size(n, p)
    return [(min(n, c * cs), min(n, (c + 1) * cs)) for c in range(p)]


class _Chunks:
    """Which columns of the working arrays hold chunk c.

    Full mode: working arrays have p * cs columns (the zero-padded tensor) and
    chunk c is a contiguous slice. Sampled mode: working arrays hold only the
    element indices `idx` of the tensor, and chunk c is the set of columns whose
    element index falls in it; every step then does, on those columns, exactly
    what it does on the full tensor."""

    def __init__(self, n: int, p: int, idx: np.ndarray | None = None):
        self.n, self.p = n, p
        self.cs = chunk_size(n, p)
        self.sampled = idx is not None
        if idx is None:
            self.width = p * self.cs
            self.cols = [slice(c * self.cs, (c + 1) * self.cs) for c in range(p)]
        else:
            idx = np.asarray(idx, dtype=np.int64)
            self.width = idx.size
            which = idx // max(self.cs, 1)
            self.cols = [np.flatnonzero(which == c) for c in range(p)]


def _widen(b: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == "f32":
        return np.asarray(b, dtype=np.float32).copy()
    if dtype == "bf16":
        return bf16_to_f32(b).copy()
    if dtype == "f64":
        return np.asarray(b, dtype=np.float64).copy()
    raise ValueError(dtype)


def _work_dtype(dtype: str):
    return np.float64 if dtype == "f64" else np.float32


def _working_copies(bufs, n, chunks, dtype):
    """Per-rank working arrays; in full mode zero-padded to p * cs."""
    out = []
    for b in bufs:
        w = _widen(b, dtype)
        if not chunks.sampled:
            padded = np.zeros(chunks.width, dtype=_work_dtype(dtype))
            padded[:n] = w[:n]
            w = padded
        out.append(w)
    return out


def _narrow(w: np.ndarray, dtype: str) -> np.ndarray:
    return f32_to_bf16(w) if dtype == "bf16" else w


def _reduce_scatter_pass(work, chunks, p, divisor, dtype, shift, counter, snaps, hop_round=False):
    """Pass 1: p - 1 steps; the owner's finished chunk is scaled in the last step.

    shift = 0: ring ownership; shift = 1: chunks pre-rotated (torch contract).
    Returns the real chunk each rank owns afterwards."""
    wdt = _work_dtype(dtype)
    esize = _ESIZE[dtype]
    owned = [(q + 1 - shift) % p for q in range(p)]

    def scale_owned():
        for q in range(p):
            cols = chunks.cols[owned[q]]
            y = work[q][cols] / wdt(divisor)
            if dtype == "bf16":
                y = bf16_to_f32(f32_to_bf16(y))
            work[q][cols] = y

    if p == 1:
        scale_owned()
        if snaps is not None:
            snaps.append([w.copy() for w in work])
        return owned
    for s in range(p - 1):
        payloads = []
        for r in range(p):
            c = (r - s - shift) % p
            payloads.append((r, c, work[r][chunks.cols[c]].copy()))
        for r, c, data in payloads:
            d = (r + 1) % p
            cols = chunks.cols[c]
            acc = work[d][cols] + data
            if hop_round:
                acc = bf16_to_f32(f32_to_bf16(acc))
            work[d][cols] = acc
            counter[r] += chunks.cs * esize
        if s == p - 2:
            scale_owned()
        if snaps is not None:
            snaps.append([w.copy() for w in work])
    return owned


def _allgather_pass(work, chunks, p, owned, esize, counter, snaps):
    """Pass 2: at step k rank r sends chunk (owned[r] - k) mod p; the receiver overwrites."""
    for k in range(p - 1):
        payloads = []
        for r in range(p):
            c = (owned[r] - k) % p
            payloads.append((r, c, work[r][chunks.cols[c]].copy()))
        for r, c, data in payloads:
            work[(r + 1) % p][chunks.cols[c]] = data
            counter[r] += chunks.cs * esize
        if snaps is not None:
            snaps.append([w.copy() for w in work])


def allreduce(bufs, n: int, divisor: float = 1.0, dtype: str = "f32", idx=None,
              snapshots: bool = False, hop_round: bool = False):
    """Ring all-reduce of p replica buffers (in place in the method; here on copies).

    bufs: p arrays of n elements (fp32 / fp64 values or uint16 bf16 patterns), or,
    in sampled mode, of len(idx) elements holding the values at element indices idx.
    Returns (outputs, info): outputs are the p results in the input's storage type;
    info has 'bytes_sent' per rank, 'owned' chunks and, if asked, 'snapshots' (the
    p working arrays after each of the steps, zero-padded, working precision).
    hop_round: round every partial to bf16 at each hop (bf16 buffers only)."""
    if hop_round and dtype != "bf16":
        raise ValueError("per-hop rounding is a bf16 variant")
    p = len(bufs)
    chunks = _Chunks(n, p, idx)
    work = _working_copies(bufs, n, chunks, dtype)
    counter = [0] * p
    snaps = [] if snapshots else None
    owned = _reduce_scatter_pass(work, chunks, p, divisor, dtype, 0, counter, snaps, hop_round)
    _allgather_pass(work, chunks, p, owned, _ESIZE[dtype], counter, snaps)
    width = n if not chunks.sampled else chunks.width
    outs = [_narrow(w[:width], dtype) for w in work]
    return outs, {"bytes_sent": counter, "owned": owned, "snapshots": snaps, "cs": chunks.cs}


def reduce_scatter(bufs, n: int, divisor: float = 1.0, dtype: str = "f32",
                   ownership: str = "rank", snapshots: bool = False):
    """Pass 1 alone. ownership 'rank': rank r receives the sum of chunk r (the
    torch contract; ValueError unless p divides n). 'ring': rank q receives chunk
    (q + 1) mod p, only its real (unpadded) elements.
    Returns (outs, info): outs[r] holds the valid elements of rank r's chunk."""
    p = len(bufs)
    if ownership == "rank":
        if n % p != 0:
            raise ValueError(f"reduce_scatter: {n} elements are not divisible by {p} ranks")
        shift = 1
    elif ownership == "ring":
        shift = 0
    else:
        raise ValueError(ownership)
    chunks = _Chunks(n, p)
    work = _working_copies(bufs, n, chunks, dtype)
    counter = [0] * p
    snaps = [] if snapshots else None
    owned = _reduce_scatter_pass(work, chunks, p, divisor, dtype, shift, counter, snaps)
    bounds = chunk_bounds(n, p)
    outs = []
    for q in range(p):
        lo, hi = bounds[owned[q]]
        outs.append(_narrow(work[q][lo:hi].copy(), dtype))
    return outs, {"bytes_sent": counter, "owned": owned, "snapshots": snaps, "cs": chunks.cs}


def allgather(ins, dtype: str = "f32", ownership: str = "rank", snapshots: bool = False):
    """Pass 2 alone: ins[r] (m elements each) is rank r's finished chunk: chunk r
    ('rank') or chunk (r + 1) mod p ('ring'). Every rank ends with all p chunks
    in chunk order (p * m elements). No scaling."""
    p = len(ins)
    m = len(ins[0]) if p else 0
    owned = [r if ownership == "rank" else (r + 1) % p for r in range(p)]
    chunks = _Chunks(p * m, p)
    wdt = np.uint16 if dtype == "bf16" else _work_dtype(dtype)
    work = [np.zeros(p * m, dtype=wdt) for _ in range(p)]
    for r in range(p):
        work[r][chunks.cols[owned[r]]] = ins[r]
    counter = [0] * p
    snaps = [] if snapshots else None
    _allgather_pass(work, chunks, p, owned, _ESIZE[dtype], counter, snaps)
    return work, {"bytes_sent": counter, "owned": owned, "snapshots": snaps}


def naive_allreduce(bufs, divisor: float = 1.0, dtype: str = "f32"):
    """Send-to-root all-reduce: rank 0 adds the buffers in rank order, divides
    once and sends the result back to every rank."""
    acc = _widen(bufs[0], dtype)
    for b in bufs[1:]:
        acc = acc + _widen(b, dtype)
    y = acc / _work_dtype(dtype)(divisor)
    return [_narrow(y.copy(), dtype) for _ in bufs]


def broadcast_tree(bufs, root: int = 0, snapshots: bool = False):
    """Doubling-tree broadcast: with relative rank v = (r - root) mod p, at step j
    every v < 2^j that has a partner v + 2^j < p copies its buffer to it.
    Returns (outs, n_steps, snapshots)."""
    p = len(bufs)
    work = [np.array(b, copy=True) for b in bufs]
    snaps = [] if snapshots else None
    span, steps = 1, 0
    while span < p:
        for v in range(span):
            if v + span < p:
                work[(root + v + span) % p] = work[(root + v) % p].copy()
        span *= 2
        steps += 1
        if snaps is not None:
            snaps.append([w.copy() for w in work])
    return work, steps, snaps


def broadcast_coalesced(tensors, root: int = 0, cap_bytes: int = 250 * 1024 * 1024):
    """tensors[r][t]: uint8 byte arrays of rank r's tensor t. Root's tensors are
    grouped into buckets of at most cap_bytes, each bucket flattened, broadcast
    by the doubling tree and unflattened into every rank's tensors.
    Returns (new tensors, groups)."""
    from .buckets import coalesce
    p = len(tensors)
    k = len(tensors[0]) if p else 0
    nbytes = [int(tensors[root][t].size) for t in range(k)]
    groups = coalesce(nbytes, cap_bytes)
    out = [[np.array(tensors[r][t], copy=True) for t in range(k)] for r in range(p)]
    for g in groups:
        total = sum(nbytes[t] for t in g)
        flats = [np.zeros(total, dtype=np.uint8) for _ in range(p)]
        pos = 0
        for t in g:
            flats[root][pos:pos + nbytes[t]] = tensors[root][t]
            pos += nbytes[t]
        flats, _, _ = broadcast_tree(flats, root)
        for r in range(p):
            pos = 0
            for t in g:
                out[r][t] = flats[r][pos:pos + nbytes[t]].copy()
                pos += nbytes[t]
    return out, groups
