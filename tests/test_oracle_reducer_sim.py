"""Pins for the readiness / overlap simulation (CPU only)."""
import pytest

from oracle import buckets as ob
from oracle import reducer_sim as rs
from oracle.costs import ring_time


def test_buckets_fire_in_order_and_a_complete_bucket_waits_its_turn():
    buckets = [[5, 4], [3, 2], [1, 0]]
    # bucket 1 completes first (tensors 3, 2) but must wait for bucket 0
    seq = rs.fire_sequence(buckets, [3, 2, 5, 1, 4, 0])
    assert seq == [(4, 0), (4, 1), (5, 2)]
    # reverse registration order: each bucket fires on its own last tensor
    assert rs.fire_sequence(buckets, [5, 4, 3, 2, 1, 0]) == [(1, 0), (3, 1), (5, 2)]
    with pytest.raises(ValueError):
        rs.fire_sequence(buckets, [5, 5])


def test_every_bucket_fires_exactly_once_for_any_order():
    import itertools
    buckets = [[4], [3, 2], [1, 0]]
    for order in itertools.permutations(range(5)):
        seq = rs.fire_sequence(buckets, list(order))
        assert [b for _, b in seq] == [0, 1, 2]
        # a bucket never fires before all its tensors are ready
        for pos, b in seq:
            assert all(order.index(t) <= pos for t in buckets[b])


def test_one_bucket_at_the_end_is_the_no_overlap_formula():
    """The page's no-overlap cell: t = end_bwd + 2(p-1) alpha + 2(p-1)/p total beta."""
    p, alpha, beta = 8, 10e-6, 1 / 50e9
    grads = [(4_000_000, 0.010), (1_000_000, 0.020), (2_000_000, 0.030)]
    total = sum(g[0] for g in grads)
    out = rs.ddp_step_time(grads, bucket_cap=10 ** 12, p=p, alpha=alpha, beta=beta)
    end_bwd = 0.030
    assert len(out["buckets"]) == 1
    assert out["step"] == pytest.approx(end_bwd + 2 * (p - 1) * alpha + 2 * (p - 1) / p * total * beta)
    assert out["exposed"] == pytest.approx(ring_time(total, p, alpha, beta))


def test_bucket_size_trade_off():
    """Many small gradients produced last-first over the backward: tiny buckets
    pay alpha many times, one huge bucket starts only at the end; a middle cap
    hides the most."""
    p, alpha, beta = 8, 20e-6, 1 / 50e9
    k = 200
    grads = [(250_000, (k - t) * 50e-6) for t in range(k)]  # tensor t ready at (k - t) * 50 us
    exposed = {cap: rs.ddp_step_time(grads, cap, p, alpha, beta)["exposed"]
               for cap in (250_000, 2_500_000, 25_000_000, 10 ** 10)}
    best = min(exposed.values())
    assert exposed[2_500_000] == best
    assert exposed[250_000] > best and exposed[10 ** 10] > best
    assert exposed[10 ** 10] == pytest.approx(ring_time(k * 250_000, p, alpha, beta))


def test_overlap_timeline():
    out = rs.overlap([1.0, 1.5, 4.0], [1.0, 1.0, 0.5])
    assert out["start"] == [1.0, 2.0, 4.0] and out["end"] == [2.0, 3.0, 4.5]
    assert out["exposed"] == pytest.approx(0.5)
    assert rs.overlap([3.0], [0.0])["exposed"] == 0.0


def test_rebuild_from_observed_order_matches_the_reversed_walk():
    numel = [15, 7, 2112, 33, 8192, 128, 17000, 17, 249856, 61]
    observed = list(range(len(numel)))[::-1]  # gradients ready last-registered first
    assert rs.rebuild(numel, 4, 16384, 262144, observed) == ob.assign_buckets(numel, 4, 16384, 262144)
    # a different observed order gives buckets in that order
    odd = [9, 0, 8, 1, 7, 2, 6, 3, 5, 4]
    b = rs.rebuild(numel, 4, 16384, 262144, odd)
    assert [t for g in b for t in g] == odd
