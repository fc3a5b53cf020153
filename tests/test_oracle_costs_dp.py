"""Pins for the oracle's closed forms (printed numbers) and the data-parallel
averaging claims on a linear model (CPU only)."""
import json
import math
import os

import numpy as np
import pytest

from oracle import costs, linear_dp
from oracle import ring as orc

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "cost_model.json")))


def _round_sig(x, digits):
    return float(f"{x:.{digits}g}")


def test_naive_allreduce_five_seconds():
    g = GOLD["naive_allreduce"]
    t = costs.naive_time(g["M_bytes"], g["p"], g["bw_Bps"])
    assert round(t) == g["printed_seconds"] and abs(t - 5.04) < 1e-9


def test_ring_recursive_doubling_crossover():
    g = GOLD["ring_rd_crossover"]
    beta = 1.0 / g["bw_Bps"]
    assert g["alpha_s"] / beta == pytest.approx(g["printed_alpha_over_beta_bytes"])
    for case in g["cases"]:
        m = costs.ring_rd_crossover(case["p"], g["alpha_s"], beta)
        assert _round_sig(m, case["printed_digits"]) == case["printed_bytes"]
        # the two times really are equal there, and the ring wins above it
        a = costs.ring_time(m, case["p"], g["alpha_s"], beta)
        b = costs.recursive_doubling_time(m, case["p"], g["alpha_s"], beta)
        assert a == pytest.approx(b, rel=1e-12)
        assert costs.ring_time(2 * m, case["p"], g["alpha_s"], beta) < \
            costs.recursive_doubling_time(2 * m, case["p"], g["alpha_s"], beta)


def test_overlap_token_thresholds():
    g = GOLD["overlap_tokens"]
    peak = costs.overlap_tokens(g["flops_peak"], g["ib_Bps"])
    assert round(peak, -2) == g["printed_peak"]
    assert round(costs.overlap_tokens(0.4 * g["flops_peak"], g["ib_Bps"]), -2) == g["printed_40pct"]
    assert round(costs.overlap_tokens(g["flops_peak"], g["nvlink_Bps"]), -2) == g["printed_nvlink"]


def test_link_speed_units():
    g = GOLD["link_speeds"]
    assert g["ib_Gbps"] / 8 == g["ib_GBps_printed"]
    assert g["nvswitch_GBps"] / g["ib_GBps_printed"] == 9


@pytest.mark.parametrize("p", [2, 3, 8, 64, 1024])
def test_ring_bandwidth_term_meets_lower_bound(p):
    M = 1e9
    beta = 1e-9
    assert costs.ring_time(M, p, 0.0, beta) == pytest.approx(costs.lower_bound_bytes(M, p) * beta)
    assert costs.ring_bytes_per_rank(M, p) == pytest.approx(costs.lower_bound_bytes(M, p))
    assert costs.ring_bytes_per_rank(M, p) < 2 * M
    assert 2 * costs.half_bytes_per_rank(M, p) == pytest.approx(costs.ring_bytes_per_rank(M, p))
    assert costs.bus_bandwidth(1.0, p) == pytest.approx(2 * (p - 1) / p)


def test_hierarchical_traffic_is_smaller():
    M, n, g = 1e9, 16, 8
    assert costs.hierarchical_net_bytes(M, n, g) < costs.flat_ring_net_bytes(M, n, g)
    assert costs.hierarchical_net_bytes(M, 1, g) == 0


def test_hierarchical_traffic_hand_worked():
    """2 nodes of 8 GPUs, 1 GB: after the in-node reduce-scatter each GPU holds
    M/8 = 125 MB and runs a 2-rank ring across nodes, sending 2(2-1)/2 of it:
    125 MB. The flat ring over all 16 GPUs sends 2 * 15/16 GB = 1.875 GB."""
    assert costs.hierarchical_net_bytes(1e9, 2, 8) == pytest.approx(125e6, rel=1e-15)
    assert costs.flat_ring_net_bytes(1e9, 2, 8) == pytest.approx(1.875e9, rel=1e-15)
    assert costs.hierarchical_net_bytes(1e9, 4, 8) == pytest.approx(187.5e6, rel=1e-15)


@pytest.mark.parametrize("n,g", [(2, 8), (4, 8), (3, 4), (8, 2)])
def test_hierarchical_traffic_equals_the_simulated_cross_node_ring(n, g):
    """The cross-node phase of the hierarchical all-reduce is a ring all-reduce
    of each GPU's M/g shard among the n nodes: the oracle's simulated ring
    counts the bytes one rank sends, which must equal the closed form."""
    M_elems = 1024 * n * g  # fp32 elements, so M/g divides into n chunks
    shard = M_elems // g
    bufs = [np.ones(shard, np.float32) for _ in range(n)]
    _, info = orc.allreduce(bufs, shard, 1.0, "f32")
    per_rank = set(info["bytes_sent"])
    assert per_rank == {costs.hierarchical_net_bytes(4 * M_elems, n, g)}
    flat = [np.ones(M_elems, np.float32) for _ in range(n * g)]
    _, finfo = orc.allreduce(flat, M_elems, 1.0, "f32")
    assert set(finfo["bytes_sent"]) == {costs.flat_ring_net_bytes(4 * M_elems, n, g)}


@pytest.mark.parametrize("p", [2, 3, 8, 16])
def test_bus_bandwidth_is_the_simulated_per_rank_send_rate(p):
    """Bus bandwidth is what one rank's link carries: the bytes the simulated
    ring makes a rank send, divided by the time. Given the algorithm bandwidth
    M / t of the same all-reduce, bus_bandwidth must reproduce it."""
    n = 96 * p  # divisible by p: no padding on the wire
    M = 4 * n
    bufs = [np.full(n, r, np.float32) for r in range(p)]
    _, info = orc.allreduce(bufs, n, 1.0, "f32")
    for t in (1e-6, 3.7e-3, 2.0):
        for sent in info["bytes_sent"]:
            assert costs.bus_bandwidth(M / t, p) == pytest.approx(sent / t, rel=1e-12)


def test_example_gradient_hand_worked():
    """x = (1, 2), w = (3, 4), y = 5: the residual is 11 - 5 = 6, so the
    gradient of 0.5 (x.w - y)^2 is 6 x = (6, 12)."""
    g = linear_dp.example_grads(np.array([[1.0, 2.0]]), np.array([5.0]), np.array([3.0, 4.0]))
    assert np.array_equal(g, np.array([[6.0, 12.0]]))


def test_example_gradients_are_the_loss_derivative():
    """Central finite differences of each example's loss 0.5 (x.w - y)^2 give
    its gradient row; the batch mean gradient is zero at the least-squares
    solution (the normal equations)."""
    rng = np.random.default_rng(7)
    X = rng.standard_normal((9, 5))
    y = rng.standard_normal(9)
    w = rng.standard_normal(5)
    G = linear_dp.example_grads(X, y, w)
    h = 1e-6
    for i in range(X.shape[0]):
        for j in range(X.shape[1]):
            e = np.zeros(5)
            e[j] = h
            lp = 0.5 * (X[i] @ (w + e) - y[i]) ** 2
            lm = 0.5 * (X[i] @ (w - e) - y[i]) ** 2
            assert G[i, j] == pytest.approx((lp - lm) / (2 * h), rel=1e-6, abs=1e-8)
    w_star = np.linalg.lstsq(X, y, rcond=None)[0]
    assert np.allclose(linear_dp.batch_mean_grad(X, y, w_star), 0.0, atol=1e-12)


def _shards(rng, counts, d=6):
    w = rng.standard_normal(d)
    shards = []
    for c in counts:
        X = rng.standard_normal((c, d))
        y = rng.standard_normal(c)
        shards.append((X, y))
    return shards, w


def test_equal_shards_mean_of_means_is_the_batch_gradient():
    rng = np.random.default_rng(0)
    shards, w = _shards(rng, [32] * 8)
    X = np.concatenate([s[0] for s in shards])
    y = np.concatenate([s[1] for s in shards])
    full = linear_dp.batch_mean_grad(X, y, w)
    assert np.allclose(linear_dp.mean_of_means(shards, w), full, rtol=1e-12, atol=1e-14)


def test_unequal_token_counts_need_sum_then_divide_once():
    rng = np.random.default_rng(1)
    shards, w = _shards(rng, [100, 10000, 731, 4000])
    X = np.concatenate([s[0] for s in shards])
    y = np.concatenate([s[1] for s in shards])
    full = linear_dp.batch_mean_grad(X, y, w)
    assert np.allclose(linear_dp.sum_then_divide_once(shards, w), full, rtol=1e-12, atol=1e-14)
    assert not np.allclose(linear_dp.mean_of_means(shards, w), full, rtol=1e-3)


def test_ring_with_token_count_divisor_gives_the_batch_gradient():
    """The fp64 ring over per-rank summed gradients with D = sum of counts."""
    rng = np.random.default_rng(2)
    counts = [100, 2500, 731, 9999, 4000]
    shards, w = _shards(rng, counts, d=23)
    X = np.concatenate([s[0] for s in shards])
    y = np.concatenate([s[1] for s in shards])
    full = linear_dp.batch_mean_grad(X, y, w)
    bufs = linear_dp.shard_sum_grads(shards, w)
    outs, _ = orc.allreduce(bufs, 23, float(sum(counts)), "f64")
    for o in outs:
        assert np.allclose(o, full, rtol=1e-12, atol=1e-14)


@pytest.mark.parametrize("p", [2, 3, 4, 8, 16])
def test_per_rank_byte_forms_equal_the_simulated_schedules(p):
    """The closed forms of what one rank sends, against the oracle's simulated
    byte counters (n divisible by p, so no padding goes on the wire): the
    two-pass ring sends 2(p-1)/p of the tensor per rank and meets the lower
    bound; each of its halves sends (p-1)/p; recursive doubling's time with
    no latency term is its per-rank bytes, M log2 p, times beta."""
    from oracle import trees
    n = 40 * p
    M = 4 * n
    bufs = [np.full(n, r + 1, np.float32) for r in range(p)]
    _, ar = orc.allreduce(bufs, n)
    assert set(ar["bytes_sent"]) == {costs.ring_bytes_per_rank(M, p)} == {costs.lower_bound_bytes(M, p)}
    _, rs = orc.reduce_scatter(bufs, n, 1.0, "f32", "ring")
    assert set(rs["bytes_sent"]) == {costs.half_bytes_per_rank(M, p)}
    _, ag = orc.allgather([np.full(n // p, r, np.float32) for r in range(p)])
    assert set(ag["bytes_sent"]) == {costs.half_bytes_per_rank(M, p)}
    if p & (p - 1) == 0:
        _, rd = trees.recursive_doubling(bufs, n)
        beta = 1e-9
        for sent in rd["bytes_sent"]:
            assert costs.recursive_doubling_time(M, p, 0.0, beta) == pytest.approx(sent * beta, rel=1e-12)
