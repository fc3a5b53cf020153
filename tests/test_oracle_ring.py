"""Pins for the oracle's ring collectives (CPU only).

Each test checks the literal simulation against something other than itself:
contribution sets (the "dots" of the ring widget), exact integer sums, the naive
send-to-root definition, error bounds of fp32 summation, the closed forms for
bytes on the wire, the all-reduce = reduce-scatter + all-gather identity, and
an independent bf16 rounding routine.
"""
import math

import numpy as np
import pytest
import torch

from oracle import ring as orc
from oracle.bf16 import bf16_to_f32, f32_to_bf16


def _rank_bits(p, n):
    """Rank r holds 2^r everywhere (fp64, exact): a sum's bits name its contributors."""
    return [np.full(n, float(2 ** r)) for r in range(p)]


def _arc_mask(start, length, p):
    return sum(2 ** ((start + j) % p) for j in range(length))


@pytest.mark.parametrize("p", range(1, 10))
def test_contribution_sets_every_step(p):
    """After reduce-scatter step s, the chunk rank d just received holds exactly
    the arc of ranks d-1-s .. d; after the pass rank q owns chunk (q+1) mod p
    complete; after the all-gather every element holds every rank."""
    full = 2 ** p - 1
    for n in range(0, 71):
        outs, info = orc.allreduce(_rank_bits(p, n), n, 1.0, "f64", snapshots=True)
        cs = info["cs"]
        snaps = info["snapshots"]
        assert len(snaps) == max(2 * (p - 1), 1)
        for s in range(p - 1):
            for d in range(p):
                c = (d - 1 - s) % p
                lo, hi = c * cs, c * cs + cs
                want = _arc_mask(c, s + 2, p)
                # padded columns carry zeros: only real elements hold the arc
                real = max(0, min(hi, n) - lo)
                assert np.all(snaps[s][d][lo:lo + real] == want), (p, n, s, d)
        assert info["owned"] == [(q + 1) % p for q in range(p)]
        if p > 1:
            rs_end = snaps[p - 2]
            for q in range(p):
                c = (q + 1) % p
                lo, hi = c * cs, min(n, c * cs + cs)
                assert np.all(rs_end[q][lo:max(lo, hi)] == full)
        for o in outs:
            assert o.shape == (n,) and np.all(o == full)


@pytest.mark.parametrize("p", [1, 2, 3, 5, 8])
def test_allgather_steps_send_chunk_r_plus_1_minus_k(p):
    """Step k of the all-gather: rank r+1 receives chunk (r+1-k) mod p of rank r."""
    n = 7 * p
    outs, info = orc.allreduce(_rank_bits(p, n), n, 1.0, "f64", snapshots=True)
    snaps = info["snapshots"]
    full = 2 ** p - 1
    cs = info["cs"]
    for k in range(p - 1):
        snap = snaps[p - 1 + k]
        for r in range(p):
            c = (r + 1 - k) % p
            assert np.all(snap[(r + 1) % p][c * cs:(c + 1) * cs] == full)


@pytest.mark.parametrize("p", [2, 3, 4, 8, 16])
def test_small_integers_are_exact_and_equal_naive(p):
    rng = np.random.default_rng(p)
    n = 1000 + p
    bufs = [rng.integers(-1000, 1000, size=n).astype(np.float32) for _ in range(p)]
    ring, _ = orc.allreduce(bufs, n, 1.0)
    naive = orc.naive_allreduce(bufs, 1.0)
    exact = np.sum(np.stack(bufs).astype(np.int64), axis=0)
    for a, b in zip(ring, naive):
        assert np.array_equal(a, b) and np.array_equal(a.astype(np.int64), exact)


@pytest.mark.parametrize("p", [2, 4, 8, 64])
def test_random_sum_within_fp32_summation_bound(p):
    rng = np.random.default_rng(10 + p)
    n = 777
    bufs = [rng.standard_normal(n).astype(np.float32) for _ in range(p)]
    outs, _ = orc.allreduce(bufs, n, float(p))
    stack = np.stack(bufs).astype(np.float64)
    exact = np.array([math.fsum(stack[:, i]) for i in range(n)]) / p
    u = 2.0 ** -24
    bound = (p - 1) * u * np.abs(stack).sum(axis=0) / p + u * np.abs(exact) + 1e-45
    for o in outs:
        assert np.all(np.abs(o.astype(np.float64) - exact) <= bound)
    # and all replicas are bit-identical: the data-parallel invariant
    for o in outs[1:]:
        assert np.array_equal(o.view(np.uint32), outs[0].view(np.uint32))


@pytest.mark.parametrize("p", [3, 4, 8])
def test_origin_rank_is_added_first(p):
    """Rank c sends chunk c first (it 'starts by sending the chunk whose index
    equals its rank'), so chunk c's fold starts at x_c. Put 1.0 on rank c and
    2^-24 (half an ulp of 1) on every other rank: added to 1 first, each tiny
    term rounds away (ties to even); any other start accumulates them."""
    n = 6 * p
    cs = orc.chunk_size(n, p)
    bufs = [np.full(n, 2.0 ** -24, dtype=np.float32) for _ in range(p)]
    for c in range(p):
        bufs[c][c * cs:(c + 1) * cs] = 1.0
    outs, _ = orc.allreduce(bufs, n, 1.0)
    assert np.all(outs[0] == 1.0)

    def with_big_at(j):
        b = [np.full(n, 2.0 ** -24, dtype=np.float32) for _ in range(p)]
        for c in range(p):
            b[(c + j) % p][c * cs:(c + 1) * cs] = 1.0
        return orc.allreduce(b, n, 1.0)[0][0]

    # x_c and x_{c+1} are the first pair added; the owner c-1 adds last, after
    # the tiny terms have summed to a representable 1 + (p-1) 2^-24
    assert np.all(with_big_at(1) == 1.0)
    assert np.all(with_big_at(p - 1) > 1.0)


@pytest.mark.parametrize("p,n", [(2, 10), (4, 1024), (8, 4096), (5, 35), (16, 160)])
def test_allreduce_is_reduce_scatter_then_allgather(p, n):
    rng = np.random.default_rng(p * n)
    bufs = [rng.standard_normal(n).astype(np.float32) for _ in range(p)]
    ar, _ = orc.allreduce(bufs, n, float(p))
    rs, _ = orc.reduce_scatter(bufs, n, float(p), ownership="ring")
    ag, _ = orc.allgather(rs, ownership="ring")
    for a, b in zip(ar, ag):
        assert np.array_equal(a.view(np.uint32), b.view(np.uint32))
    # the torch contract's pre-rotated order reaches the same sum up to rounding
    rs2, _ = orc.reduce_scatter(bufs, n, float(p), ownership="rank")
    ag2, _ = orc.allgather(rs2, ownership="rank")
    for a, b in zip(ar, ag2):
        assert np.allclose(a, b, rtol=1e-5, atol=1e-6)


@pytest.mark.parametrize("p", [1, 2, 3, 4, 7])
def test_reduce_scatter_torch_contract(p):
    """Rank r returns the (complete) sum of chunk r; ValueError when p does not divide n."""
    n = 5 * p
    outs, info = orc.reduce_scatter(_rank_bits(p, n), n, 1.0, "f64", ownership="rank")
    m = n // p
    for r in range(p):
        assert outs[r].shape == (m,) and np.all(outs[r] == 2 ** p - 1)
    assert info["owned"] == list(range(p))
    if p > 1:
        with pytest.raises(ValueError):
            orc.reduce_scatter(_rank_bits(p, n + 1), n + 1, ownership="rank")
    # pre-rotation: real chunk c starts at rank c+1, so 1.0 there is added first
    bufs = [np.full(n, 2.0 ** -24, dtype=np.float32) for _ in range(p)]
    for c in range(p):
        bufs[(c + 1) % p][c * m:(c + 1) * m] = 1.0
    outs, _ = orc.reduce_scatter(bufs, n, 1.0, ownership="rank")
    assert all(np.all(o == 1.0) for o in outs)


def test_reduce_scatter_ring_ownership_trims_padding():
    p, n = 4, 10  # cs = 3, chunk 3 holds one real element
    outs, info = orc.reduce_scatter(_rank_bits(p, n), n, 1.0, "f64", ownership="ring")
    lens = [len(o) for o in outs]
    assert info["owned"] == [1, 2, 3, 0]
    assert lens == [3, 3, 1, 3]


@pytest.mark.parametrize("p,n", [(2, 8), (4, 1000), (8, 8192), (3, 999)])
def test_bytes_on_the_wire(p, n):
    """Per rank 2T(p-1)/p for the all-reduce, (p-1)M/p for each half; the ring
    meets the lower bound 2(p-1)M/p. With padding, a chunk is ceil(n/p)."""
    bufs = [np.zeros(n, dtype=np.float32) for _ in range(p)]
    _, info = orc.allreduce(bufs, n)
    T = 4 * n
    cs = orc.chunk_size(n, p)
    assert all(b == 2 * (p - 1) * cs * 4 for b in info["bytes_sent"])
    if n % p == 0:
        assert all(b == 2 * T * (p - 1) / p for b in info["bytes_sent"])
        _, rs = orc.reduce_scatter(bufs, n, ownership="rank")
        assert all(b == (p - 1) * T / p for b in rs["bytes_sent"])
        _, ag = orc.allgather([np.zeros(n // p, np.float32)] * p)
        assert all(b == (p - 1) * T / p for b in ag["bytes_sent"])


@pytest.mark.parametrize("p", [1, 2, 4, 8])
def test_divisor_applied_once(p):
    """p = 1 is a scale-only pass; D may be a global token count."""
    n = 100
    rng = np.random.default_rng(p)
    bufs = [rng.integers(-50, 50, size=n).astype(np.float32) for _ in range(p)]
    D = 12345.0
    outs, _ = orc.allreduce(bufs, n, D)
    exact_sum = np.sum(np.stack(bufs), axis=0, dtype=np.float64)  # exact: small integers
    assert np.array_equal(outs[0], (exact_sum.astype(np.float32) / np.float32(D)))


def test_bf16_rounding_matches_torch():
    """Round-to-nearest-even narrowing against torch's own cast, on edge patterns
    and a wide sample of fp32 bit patterns; widening is exact."""
    rng = np.random.default_rng(0)
    pats = rng.integers(0, 2 ** 32, size=2_000_000, dtype=np.uint64).astype(np.uint32)
    edges = np.array([0, 0x80000000, 0x00008000, 0x00018000, 0x3F808000, 0x3F818000, 0x3F807FFF,
                      0x7F7F8000, 0x7F7FFFFF, 0x7F800000, 0xFF800000, 0x00000001, 0x807FFFFF],
                     dtype=np.uint32)
    pats = np.concatenate([pats, edges])
    x = pats.view(np.float32)
    finite = np.isfinite(x) | np.isinf(x)
    mine = f32_to_bf16(x[finite])
    ref = torch.from_numpy(x[finite].copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(mine, ref)
    nan = f32_to_bf16(np.array([np.nan], dtype=np.float32))
    assert np.isnan(bf16_to_f32(nan))[0]
    b = rng.integers(0, 2 ** 16, size=10000).astype(np.uint16)
    wid = bf16_to_f32(b)
    ok = ~np.isnan(wid)
    assert np.array_equal(torch.from_numpy(b.view(np.int16)).view(torch.bfloat16).float().numpy()[ok], wid[ok])


@pytest.mark.parametrize("p", [2, 4, 8])
def test_bf16_allreduce_rounds_once(p):
    """Small-integer bf16 inputs: the fp32 sum is exact, so the result must be
    the single rounding of exact_sum / D to bf16 (torch's cast as the check)."""
    n = 333
    rng = np.random.default_rng(p)
    vals = [rng.integers(-100, 100, size=n).astype(np.float32) for _ in range(p)]
    bufs = [f32_to_bf16(v) for v in vals]
    D = 3.0
    outs, _ = orc.allreduce(bufs, n, D, "bf16")
    exact = np.sum(np.stack(vals).astype(np.float64), axis=0)
    want = torch.from_numpy((exact.astype(np.float32) / np.float32(D))).to(torch.bfloat16)
    want = want.view(torch.int16).numpy().view(np.uint16)
    for o in outs:
        assert o.dtype == np.uint16 and np.array_equal(o, want)


@pytest.mark.parametrize("p,root", [(1, 0), (2, 1), (5, 3), (8, 0), (9, 4)])
def test_doubling_tree_broadcast(p, root):
    bufs = [np.full(4, r, dtype=np.int32) for r in range(p)]
    outs, steps, _ = orc.broadcast_tree(bufs, root)
    assert steps == (math.ceil(math.log2(p)) if p > 1 else 0)
    assert all(np.array_equal(o, bufs[root]) for o in outs)


def test_broadcast_coalesced_copies_root_tensors():
    rng = np.random.default_rng(1)
    p, k = 5, 9
    sizes = [int(s) for s in rng.integers(0, 40, size=k)]
    tensors = [[rng.integers(0, 255, size=s).astype(np.uint8) for s in sizes] for _ in range(p)]
    out, groups = orc.broadcast_coalesced(tensors, root=2, cap_bytes=64)
    assert all(sum(sizes[t] for t in g) <= 64 or len(g) == 1 for g in groups)
    for r in range(p):
        for t in range(k):
            assert np.array_equal(out[r][t], tensors[2][t])


def test_sampled_mode_equals_full_mode():
    """Running the steps on a subset of element indices gives those elements' full-run results."""
    p, n = 8, 5003
    rng = np.random.default_rng(7)
    bufs = [rng.standard_normal(n).astype(np.float32) for _ in range(p)]
    full, _ = orc.allreduce(bufs, n, 8.0)
    idx = np.sort(rng.choice(n, size=300, replace=False))
    samp, _ = orc.allreduce([b[idx] for b in bufs], n, 8.0, idx=idx)
    for a, b in zip(full, samp):
        assert np.array_equal(a[idx], b)


@pytest.mark.parametrize("p", [2, 4, 8])
def test_per_hop_bf16_equals_accumulate_when_every_partial_is_exact(p):
    """Small integers: every partial sum is a bf16 value, so rounding at each hop
    changes nothing."""
    rng = np.random.default_rng(p)
    n = 257
    vals = [rng.integers(-16, 16, size=n).astype(np.float32) for _ in range(p)]
    bufs = [f32_to_bf16(v) for v in vals]
    a, _ = orc.allreduce(bufs, n, 1.0, "bf16")
    b, _ = orc.allreduce(bufs, n, 1.0, "bf16", hop_round=True)
    for x, y in zip(a, b):
        assert np.array_equal(x, y)


def test_per_hop_bf16_worked_example():
    """p = 8, 256 on the origin rank and 1 on the seven others. Near 256 the
    bf16 spacing is 2, so each hop's 256 + 1 is a tie and rounds to the even
    256: the per-hop ring ends at 256. Accumulating in fp32 gives the exact
    263, whose single rounding (a tie between 262 and 264) goes to the even 264."""
    p, n = 8, 8
    bufs = []
    for r in range(p):
        v = np.ones(n, dtype=np.float32)
        v[r] = 256.0  # chunk r (one element each) starts at rank r
        bufs.append(f32_to_bf16(v))
    hop, _ = orc.allreduce(bufs, n, 1.0, "bf16", hop_round=True)
    acc, _ = orc.allreduce(bufs, n, 1.0, "bf16")
    assert np.all(bf16_to_f32(hop[0]) == 256.0)
    assert np.all(bf16_to_f32(acc[0]) == 264.0)


def test_per_hop_bf16_error_grows_with_p():
    """Against the exact sum, rounding every hop errs more than rounding once,
    and more so as p grows (the error-growth study, on normal gradients)."""
    rng = np.random.default_rng(0)
    n = 20000
    errs = {}
    for p in (2, 8, 32):
        vals = [rng.standard_normal(n).astype(np.float32) for _ in range(p)]
        bufs = [f32_to_bf16(v) for v in vals]
        exact = np.sum(np.stack([bf16_to_f32(b) for b in bufs]).astype(np.float64), axis=0)
        once, _ = orc.allreduce(bufs, n, 1.0, "bf16")
        hop, _ = orc.allreduce(bufs, n, 1.0, "bf16", hop_round=True)
        e1 = np.mean(np.abs(bf16_to_f32(once[0]) - exact))
        e2 = np.mean(np.abs(bf16_to_f32(hop[0]) - exact))
        errs[p] = (e1, e2)
        # one rounding of the exact sum: within half an ulp of bf16
        assert np.all(np.abs(bf16_to_f32(once[0]) - exact) <= 2.0 ** -8 * np.abs(exact) + 1e-30)
    assert errs[2][1] >= errs[2][0] and errs[8][1] > 1.5 * errs[8][0] and errs[32][1] > 2 * errs[32][0]
    assert errs[32][1] / errs[32][0] > errs[8][1] / errs[8][0]
