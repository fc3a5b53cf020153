"""Pins for the oracle's bucket assignment, flatten/unflatten and coalescing (CPU only)."""
import itertools
import json
import os

import numpy as np
import pytest

from oracle import buckets as ob
from oracle.ring import chunk_size
from synth import shapes

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "tiny_buckets.json")))


def test_tiny_reversed_matches_hand_worked_table():
    g = GOLD
    b = ob.assign_buckets(g["numel"], g["elem_size"], g["first_cap_bytes"], g["cap_bytes"], "reversed")
    assert b == g["reversed"]["buckets"]
    bucket_of, offset, bnumel = ob.bucket_layout(g["numel"], b)
    assert bnumel == g["reversed"]["bucket_numel"]
    for t, off in g["reversed"]["offset"].items():
        assert offset[int(t)] == off
    cs = [chunk_size(n, g["p"]) for n in bnumel]
    assert cs == g["reversed"]["chunk_size"]
    assert [g["p"] * c - n for c, n in zip(cs, bnumel)] == g["reversed"]["pad"]


def test_tiny_registration_reading_matches_hand_worked_table():
    g = GOLD
    b = ob.assign_buckets(g["numel"], g["elem_size"], g["first_cap_bytes"], g["cap_bytes"], "registration")
    assert b == g["registration"]["buckets"]
    assert ob.bucket_layout(g["numel"], b)[2] == g["registration"]["bucket_numel"]


def _valid_partition(groups, numel, esize, first_cap, cap):
    """The characterisation of the close rule: every bucket but the last reaches
    its cap with its last tensor and not before; the last never reaches it before
    its last tensor."""
    for i, g in enumerate(groups):
        c = first_cap if i == 0 else cap
        sizes = [numel[t] * esize for t in g]
        prefix = np.cumsum(sizes)
        if i < len(groups) - 1:
            if not (prefix[-1] >= c and (len(g) == 1 or prefix[-2] < c)):
                return False
        if any(prefix[j] >= c for j in range(len(g) - 1)):
            return False
    return True


@pytest.mark.parametrize("seed", range(40))
def test_assignment_is_the_unique_partition_the_close_rule_allows(seed):
    """Brute force over every split of the reversed walk into contiguous buckets."""
    rng = np.random.default_rng(seed)
    k = int(rng.integers(0, 8))
    numel = [int(x) for x in rng.integers(0, 12, size=k)]
    first_cap, cap = int(rng.integers(1, 30)) * 4, int(rng.integers(1, 60)) * 4
    walk = list(range(k - 1, -1, -1))
    valid = []
    for cuts in itertools.product([0, 1], repeat=max(k - 1, 0)):
        groups, cur = [], [walk[0]] if k else []
        for j, cut in enumerate(cuts):
            if cut:
                groups.append(cur)
                cur = []
            cur.append(walk[j + 1])
        if cur:
            groups.append(cur)
        if _valid_partition(groups, numel, 4, first_cap, cap):
            valid.append(groups)
    got = ob.assign_buckets(numel, 4, first_cap, cap, "reversed")
    if k == 0:
        assert got == []
    else:
        assert valid == [got]


def test_edge_cases():
    # exactly at the cap closes; a tensor larger than the cap travels alone
    assert ob.assign_buckets([2, 2, 2], 4, 16, 16) == [[2, 1], [0]]
    assert ob.assign_buckets([100, 1, 1], 4, 16, 16) == [[2, 1, 0]]
    assert ob.assign_buckets([1, 100, 1], 4, 4, 16) == [[2], [1], [0]]
    # zero-element tensors join the open bucket and never close one
    assert ob.assign_buckets([0, 0, 0], 4, 16, 16) == [[2, 1, 0]]
    assert ob.assign_buckets([], 4, 16, 16) == []


@pytest.mark.parametrize("builder", [shapes.resnet50, shapes.gpt2_small, shapes.llama_1b])
def test_model_sized_sets_partition_and_respect_caps(builder):
    numel = [shapes.numel(s) for _, s in builder()]
    first, cap = 1 << 20, 25 << 20
    esize = 2 if builder is shapes.llama_1b else 4
    b = ob.assign_buckets(numel, esize, first, cap)
    assert sorted(t for g in b for t in g) == list(range(len(numel)))
    assert _valid_partition(b, numel, esize, first, cap)
    # the first bucket to fire holds the last-registered tensors
    assert b[0][0] == len(numel) - 1


def test_resnet50_bucket_count():
    numel = [shapes.numel(s) for _, s in shapes.resnet50()]
    b = ob.assign_buckets(numel, 4, 1 << 20, 25 << 20)
    sizes = ob.bucket_layout(numel, b)[2]
    assert len(b) == 5 and sum(sizes) == 25557032


def test_flatten_unflatten_round_trip_and_predivide():
    rng = np.random.default_rng(3)
    numel = [5, 0, 17, 3]
    grads = [rng.standard_normal(n).astype(np.float32) for n in numel]
    members = [3, 2, 1, 0]
    _, offset, bn = ob.bucket_layout(numel, [members])
    flat = ob.flatten(grads, members, offset, bn[0])
    assert flat.size == sum(numel)
    assert np.array_equal(flat[:3], grads[3]) and np.array_equal(flat[3:20], grads[2])
    back = ob.unflatten(flat, members, offset, numel)
    for t in members:
        assert np.array_equal(back[t], grads[t])
    # pre-dividing by a power of two is exact: equal to scaling afterwards
    pre = ob.flatten(grads, members, offset, bn[0], predivide=8.0)
    assert np.array_equal(pre, flat / np.float32(8.0))


def test_coalesce_groups():
    nb = [10, 20, 30, 500, 5, 5]
    g = ob.coalesce(nb, 60)
    assert g == [[0, 1, 2], [3], [4, 5]]
    assert [t for grp in g for t in grp] == list(range(len(nb)))
    for grp in g:
        assert sum(nb[t] for t in grp) <= 60 or len(grp) == 1
    # greedy: the next tensor would not have fitted
    for a, b in zip(g, g[1:]):
        assert sum(nb[t] for t in a) + nb[b[0]] > 60
    assert ob.coalesce([], 60) == []
