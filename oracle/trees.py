"""Tree-shaped all-reduces, simulated literally (oracle; test infrastructure).

Sources (titles and sections of the pages):
  * "Data parallelism", "Latency, trees, and choosing an algorithm": recursive
    doubling -- at step j = 0 .. log2 p - 1 rank r exchanges its whole current
    buffer with rank r XOR 2^j and both add; log2 p steps, M log2 p bytes per
    rank. Recursive halving and doubling (Rabenseifner's algorithm) exchanges
    half of the remaining data at each step: 2 log2 p latency terms and the
    optimal 2(p-1)M/p bytes when p is a power of two.
  * "Collective Ops From Scratch", intro: tree all-reduce has depth log2 N;
    the exercise adds a tree all-reduce beside the ring; the same page's
    broadcast is a doubling tree.

Readings where the pages leave a step open:
  * Recursive doubling and Rabenseifner need p to be a power of two
    (ValueError otherwise); the tree works for any p.
  * Rabenseifner's halving: chunks as in the ring (cs = ceil(n/p), virtual
    tail padding). At halving step k the partner distance is d = p / 2^(k+1);
    of the pair (r, r ^ d) the rank with bit d clear keeps the lower half of
    their common segment and the other the upper half, each adding the
    partner's copy of the half it keeps. Rank r ends owning chunk r. The
    all-gather then doubles back (d = 1, 2, ..., p/2), each pair swapping
    the segments they own.
  * The tree all-reduce: a binomial reduce to rank 0 (at step j every rank
    r with r mod 2^(j+1) == 0 adds rank r + 2^j's partial, if that rank
    exists), the division by D on rank 0, then the doubling-tree broadcast.
  * Every add is local + received in fp32 (commutative: both partners of an
    exchange hold the same bits); the division by D is applied once at the end
    of the reduction, on every copy holding a finished sum.
"""
from __future__ import annotations

import numpy as np

from .bf16 import bf16_to_f32, f32_to_bf16
from .ring import _ESIZE, _narrow, _widen, _work_dtype, chunk_size


def _pow2(p: int) -> bool:
    return p >= 1 and (p & (p - 1)) == 0


def _log2(p: int) -> int:
    return p.bit_length() - 1


def _scale(w, divisor, dtype):
    y = w / _work_dtype(dtype)(divisor)
    if dtype == "bf16":
        y = bf16_to_f32(f32_to_bf16(y))
    return y


def recursive_doubling(bufs, n: int, divisor: float = 1.0, dtype: str = "f32", snapshots: bool = False):
    """log2 p steps; at step j every pair (r, r ^ 2^j) swaps whole buffers and adds."""
    p = len(bufs)
    if not _pow2(p):
        raise ValueError(f"recursive doubling needs p a power of two, got {p}")
    work = [_widen(b, dtype)[:n].copy() for b in bufs]
    sent = [0] * p
    snaps = [] if snapshots else None
    for j in range(_log2(p)):
        d = 1 << j
        payloads = [work[r].copy() for r in range(p)]
        for r in range(p):
            work[r] = work[r] + payloads[r ^ d]
            sent[r] += n * _ESIZE[dtype]
        if snaps is not None:
            snaps.append([w.copy() for w in work])
    outs = [_narrow(_scale(w, divisor, dtype), dtype) for w in work]
    return outs, {"bytes_sent": sent, "steps": _log2(p), "snapshots": snaps}


def rabenseifner(bufs, n: int, divisor: float = 1.0, dtype: str = "f32", snapshots: bool = False):
    """Recursive-halving reduce-scatter (log2 p steps) then recursive-doubling
    all-gather (log2 p steps)."""
    p = len(bufs)
    if not _pow2(p):
        raise ValueError(f"Rabenseifner's algorithm needs p a power of two, got {p}")
    cs = chunk_size(n, p)
    L = p * cs
    work = []
    for b in bufs:
        w = np.zeros(L, dtype=_work_dtype(dtype))
        w[:n] = _widen(b, dtype)[:n]
        work.append(w)
    seg = [(0, p) for _ in range(p)]  # chunk range each rank still reduces
    sent = [0] * p
    snaps = [] if snapshots else None
    steps = _log2(p)
    es = _ESIZE[dtype]
    for k in range(steps):
        d = p >> (k + 1)
        payloads = [w.copy() for w in work]
        new_seg = list(seg)
        for r in range(p):
            lo, hi = seg[r]
            mid = (lo + hi) // 2
            keep = (lo, mid) if (r & d) == 0 else (mid, hi)
            give = (mid, hi) if (r & d) == 0 else (lo, mid)
            a, b = keep[0] * cs, keep[1] * cs
            work[r][a:b] = work[r][a:b] + payloads[r ^ d][a:b]
            new_seg[r] = keep
            sent[r] += (give[1] - give[0]) * cs * es
        seg = new_seg
        if snaps is not None:
            snaps.append([w.copy() for w in work])
    for r in range(p):  # each rank now owns one finished chunk
        a, b = seg[r][0] * cs, seg[r][1] * cs
        work[r][a:b] = _scale(work[r][a:b], divisor, dtype)
    owned = [seg[r][0] for r in range(p)]
    for k in range(steps):
        d = 1 << k
        payloads = [(seg[r], work[r].copy()) for r in range(p)]
        new_seg = list(seg)
        for r in range(p):
            (plo, phi), pw = payloads[r ^ d]
            work[r][plo * cs:phi * cs] = pw[plo * cs:phi * cs]
            new_seg[r] = (min(seg[r][0], plo), max(seg[r][1], phi))
            sent[r] += (seg[r][1] - seg[r][0]) * cs * es
        seg = new_seg
        if snaps is not None:
            snaps.append([w.copy() for w in work])
    outs = [_narrow(w[:n], dtype) for w in work]
    return outs, {"bytes_sent": sent, "steps": 2 * steps, "owned": owned, "snapshots": snaps, "cs": cs}


def tree(bufs, n: int, divisor: float = 1.0, dtype: str = "f32", snapshots: bool = False):
    """Binomial reduce to rank 0, scale there, then the doubling-tree broadcast."""
    p = len(bufs)
    work = [_widen(b, dtype)[:n].copy() for b in bufs]
    sent = [0] * p
    snaps = [] if snapshots else None
    es = _ESIZE[dtype]
    span, steps = 1, 0
    while span < p:
        payloads = [w.copy() for w in work]
        for r in range(0, p, 2 * span):
            if r + span < p:
                work[r] = work[r] + payloads[r + span]
                sent[r + span] += n * es
        span *= 2
        steps += 1
        if snaps is not None:
            snaps.append([w.copy() for w in work])
    work[0] = _scale(work[0], divisor, dtype)
    span = 1
    while span < p:
        for v in range(span):
            if v + span < p:
                work[v + span] = work[v].copy()
                sent[v] += n * es
        span *= 2
        steps += 1
        if snaps is not None:
            snaps.append([w.copy() for w in work])
    outs = [_narrow(w, dtype) for w in work]
    return outs, {"bytes_sent": sent, "steps": steps, "snapshots": snaps}
