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
