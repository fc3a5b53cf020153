"""Cost-model closed forms of the pages (oracle; test infrastructure).

Sources:
  * "Data parallelism", "Ring all-reduce, derived": the naive send-to-root
    all-reduce takes at least 2(p-1)M/B; each ring step costs alpha + (M/p)/B
    (Hockney's model, beta = 1/B), for 2(p-1) steps; any all-reduce has a rank
    that sends at least 2(p-1)M/p bytes (Patarasuk and Yuan); reduce-scatter or
    all-gather alone is one pass, (p-1)M/p bytes per rank.
  * Same page, "Latency, trees, and choosing an algorithm": recursive doubling
    takes log2 p steps, each exchanging the whole buffer; setting the two times
    equal gives the crossover message size.
  * Same page, "The hardware the messages run on": bus bandwidth is algorithm
    bandwidth times 2(p-1)/p; the hierarchical all-reduce's per-GPU network
    traffic is 2(n-1)/n * M/g instead of 2(ng-1)/(ng) * M.
  * Same page, "When data parallelism stops scaling": backward costs 4N FLOPs
    per token, the bf16 all-reduce moves about 2 x 2N bytes per GPU, so comm
    hides under backward when n_tok >= F/B.
  * "Collective Ops From Scratch", intro: per-rank bytes of the ring are
    2T(N-1)/N.
The formulas that the extracted text lost are rebuilt from the words around
them; each reproduces the numbers the pages print.
"""
from __future__ import annotations

import math


def naive_time(M: float, p: int, bw: float) -> float:
    """Send-to-root all-reduce: rank 0 receives and sends (p-1)M bytes."""
    return 2 * (p - 1) * M / bw


def ring_time(M: float, p: int, alpha: float, beta: float) -> float:
    """2(p-1) steps of alpha + (M/p) beta."""
    return 2 * (p - 1) * (alpha + (M / p) * beta)


def ring_bytes_per_rank(T: float, p: int) -> float:
    """Bytes each rank sends in a ring all-reduce of a T-byte tensor."""
    return 2 * T * (p - 1) / p


def lower_bound_bytes(M: float, p: int) -> float:
    """Some rank must send at least this many bytes in any all-reduce."""
    return 2 * (p - 1) * M / p


def half_bytes_per_rank(M: float, p: int) -> float:
    """Reduce-scatter or all-gather alone (M = the full gathered size)."""
    return (p - 1) * M / p


def recursive_doubling_time(M: float, p: int, alpha: float, beta: float) -> float:
    return math.log2(p) * (alpha + M * beta)


def ring_rd_crossover(p: int, alpha: float, beta: float) -> float:
    """M* where ring_time == recursive_doubling_time; the ring is faster above it."""
    lg = math.log2(p)
    return (2 * (p - 1) - lg) * alpha / ((lg - 2 * (p - 1) / p) * beta)


def bus_bandwidth(algbw: float, p: int) -> float:
    return algbw * 2 * (p - 1) / p


def hierarchical_net_bytes(M: float, n: int, g: int) -> float:
    return 2 * (n - 1) / n * M / g


def flat_ring_net_bytes(M: float, n: int, g: int) -> float:
    return 2 * (n * g - 1) / (n * g) * M


def overlap_tokens(flops: float, bw: float) -> float:
    """Tokens per GPU per step at which a bf16 gradient all-reduce (4N bytes)
    fits under the backward pass (4N FLOPs per token): F/B."""
    return flops / bw
