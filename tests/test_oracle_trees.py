"""Pins for the oracle's tree-shaped all-reduces (CPU only): contribution sets
after every step, exact integer sums against the naive send-to-root sum,
bytes and step counts against the closed forms of "Data parallelism",
"Latency, trees, and choosing an algorithm", and the tree summation bound."""
import math

import numpy as np
import pytest

from oracle import ring as orc
from oracle import trees as ot
from oracle.bf16 import bf16_to_f32, f32_to_bf16

POW2 = [1, 2, 4, 8, 16, 32]


def _bits(p, n):
    return [np.full(n, float(2 ** r)) for r in range(p)]


def _mask(ranks):
    return sum(2 ** q for q in ranks)


@pytest.mark.parametrize("p", POW2)
def test_recursive_doubling_contribution_sets(p):
    """After step j rank r holds exactly the ranks that agree with it above bit j."""
    n = 13
    outs, info = ot.recursive_doubling(_bits(p, n), n, 1.0, "f64", snapshots=True)
    assert info["steps"] == int(math.log2(p))
    for j, snap in enumerate(info["snapshots"]):
        for r in range(p):
            group = [q for q in range(p) if q >> (j + 1) == r >> (j + 1)]
            assert np.all(snap[r] == _mask(group))
    assert all(np.all(o == 2 ** p - 1) for o in outs)


@pytest.mark.parametrize("p", POW2)
@pytest.mark.parametrize("n", [1, 7, 64, 101])
def test_rabenseifner_contribution_sets_and_ownership(p, n):
    """After halving step k (distance d = p / 2^(k+1)) the half rank r keeps holds
    the ranks congruent to r modulo d; rank r ends owning chunk r; the
    all-gather leaves every rank with every finished chunk."""
    outs, info = ot.rabenseifner(_bits(p, n), n, 1.0, "f64", snapshots=True)
    L = int(math.log2(p))
    assert info["steps"] == 2 * L
    cs = info["cs"]
    assert info["owned"] == list(range(p))
    seg = [(0, p)] * p
    for k in range(L):
        d = p >> (k + 1)
        snap = info["snapshots"][k]
        new = []
        for r in range(p):
            lo, hi = seg[r]
            mid = (lo + hi) // 2
            keep = (lo, mid) if (r & d) == 0 else (mid, hi)
            new.append(keep)
            group = [q for q in range(p) if q % d == r % d]
            a, b = keep[0] * cs, min(n, keep[1] * cs)
            if b > a:
                assert np.all(snap[r][a:b] == _mask(group)), (p, n, k, r)
        seg = new
    assert all(np.all(o == 2 ** p - 1) for o in outs)


@pytest.mark.parametrize("p", [1, 2, 3, 5, 6, 8, 13])
def test_tree_reduce_then_broadcast(p):
    n = 11
    outs, info = ot.tree(_bits(p, n), n, 1.0, "f64", snapshots=True)
    up = (p - 1).bit_length()
    assert info["steps"] == 2 * up
    for j in range(up):
        snap = info["snapshots"][j]
        for r in range(0, p, 2 ** (j + 1)):
            assert np.all(snap[r] == _mask(range(r, min(p, r + 2 ** (j + 1)))))
    assert all(np.all(o == 2 ** p - 1) for o in outs)


@pytest.mark.parametrize("algo", ["rd", "rab", "tree"])
@pytest.mark.parametrize("p", [2, 4, 8, 16])
def test_exact_integers_equal_naive_sum(algo, p):
    rng = np.random.default_rng(p)
    n = 1000 + 3
    bufs = [rng.integers(-1000, 1000, size=n).astype(np.float32) for _ in range(p)]
    f = {"rd": ot.recursive_doubling, "rab": ot.rabenseifner, "tree": ot.tree}[algo]
    outs, _ = f(bufs, n, 1.0)
    naive = orc.naive_allreduce(bufs, 1.0)
    for o in outs:
        assert np.array_equal(o, naive[0])


@pytest.mark.parametrize("p", [2, 4, 8, 32])
def test_bytes_on_the_wire(p):
    """Recursive doubling sends the whole buffer every step: M log2 p per rank.
    Rabenseifner sends the optimal 2(p-1)M/p per rank. The tree sends
    2(p-1)M in all (p-1 partials up, p-1 copies down)."""
    n = 64 * p
    M = 4 * n
    bufs = [np.zeros(n, np.float32) for _ in range(p)]
    _, rd = ot.recursive_doubling(bufs, n)
    assert all(b == M * math.log2(p) for b in rd["bytes_sent"])
    _, rab = ot.rabenseifner(bufs, n)
    assert all(b == 2 * (p - 1) * M / p for b in rab["bytes_sent"])
    _, tr = ot.tree(bufs, n)
    assert sum(tr["bytes_sent"]) == 2 * (p - 1) * M


@pytest.mark.parametrize("algo", ["rd", "rab", "tree"])
@pytest.mark.parametrize("p", [2, 8, 64])
def test_tree_summation_bound(algo, p):
    """A balanced pairwise sum errs by at most ceil(log2 p) u sum|x|."""
    rng = np.random.default_rng(7 + p)
    n = 2001
    bufs = [rng.standard_normal(n).astype(np.float32) for _ in range(p)]
    f = {"rd": ot.recursive_doubling, "rab": ot.rabenseifner, "tree": ot.tree}[algo]
    outs, _ = f(bufs, n, 1.0)
    st = np.stack(bufs).astype(np.float64)
    exact = np.array([math.fsum(st[:, i]) for i in range(n)])
    bound = math.ceil(math.log2(p)) * 2.0 ** -24 * np.abs(st).sum(axis=0) + 1e-45
    for o in outs:
        assert np.all(np.abs(o.astype(np.float64) - exact) <= bound)
    for o in outs[1:]:
        assert np.array_equal(o.view(np.uint32), outs[0].view(np.uint32))


@pytest.mark.parametrize("p", [2, 4, 8, 16])
def test_recursive_doubling_and_tree_pair_the_same_way(p):
    """For p a power of two both pair distance 1 first, so their bits agree."""
    rng = np.random.default_rng(p)
    bufs = [rng.standard_normal(333).astype(np.float32) for _ in range(p)]
    a, _ = ot.recursive_doubling(bufs, 333, float(p))
    b, _ = ot.tree(bufs, 333, float(p))
    assert np.array_equal(a[0].view(np.uint32), b[0].view(np.uint32))


def test_non_power_of_two_is_refused():
    bufs = [np.zeros(4, np.float32)] * 6
    with pytest.raises(ValueError):
        ot.recursive_doubling(bufs, 4)
    with pytest.raises(ValueError):
        ot.rabenseifner(bufs, 4)


def test_bf16_rounds_once():
    p, n = 8, 100
    rng = np.random.default_rng(0)
    vals = [rng.integers(-50, 50, size=n).astype(np.float32) for _ in range(p)]
    bufs = [f32_to_bf16(v) for v in vals]
    exact = np.sum(np.stack(vals), axis=0, dtype=np.float64)
    want = f32_to_bf16((exact.astype(np.float32) / np.float32(3.0)))
    for f in (ot.recursive_doubling, ot.rabenseifner, ot.tree):
        outs, _ = f(bufs, n, 3.0, "bf16")
        assert all(np.array_equal(o, want) for o in outs)
        assert np.array_equal(bf16_to_f32(outs[0]), bf16_to_f32(want))
