"""What a whole gradient synchronisation must give, computed by the CPU oracle
from its own bucket plan, for the GPU parity tests.

The plan (which tensors share a bucket, their offsets, each bucket's size)
comes from oracle.buckets, never from the Reducer under test; each helper
first asserts that the Reducer's plan equals it. Values come from the
oracle's literal ring on inputs regenerated on the host by the seeded
generator."""
from __future__ import annotations

import numpy as np

from oracle import buckets as ob
from oracle import ring as orc
from oracle.bf16 import bf16_to_f32, f32_to_bf16
from synth import workloads as W
from tests.helpers import assert_bf16_close, assert_bit_equal, to_host


def oracle_plan(cfg, red=None, order: str = "reversed"):
    """(buckets, offset per tensor, elements per bucket) by the oracle's walk;
    if a Reducer is given, its plan must be the same."""
    numel = W.numels(cfg)
    plan = ob.assign_buckets(numel, W.esize(cfg), cfg["first_cap"], cfg["cap"], order)
    _, offset, bnumel = ob.bucket_layout(numel, plan)
    if red is not None:
        assert red.buckets == plan, "the library's buckets differ from the oracle's"
        assert list(red.bucket_numel) == list(bnumel), "bucket sizes differ from the oracle's"
        assert all(red.offset[t] == offset[t] for b in plan for t in b), "offsets differ from the oracle's"
    return plan, offset, bnumel


def flat_inputs(cfg, members, offset, n, p=None):
    """Every replica's flat bucket of `members`, from host-regenerated inputs."""
    p = p or cfg["p"]
    numel = W.numels(cfg)
    starts = W.tensor_starts(cfg)
    ins = []
    for r in range(p):
        hv = {t: W.host_values(cfg, r, np.arange(starts[t], starts[t] + numel[t])) for t in members}
        if cfg["dtype"] == "bf16":
            hv = {t: bf16_to_f32(v) for t, v in hv.items()}
        flat = ob.flatten([hv.get(t, np.zeros(0, np.float32)) for t in range(len(numel))], members, offset, n)
        ins.append(f32_to_bf16(flat) if cfg["dtype"] == "bf16" else flat)
    return ins


def whole_set_expected(cfg, red=None, plan=None):
    """Oracle: flatten, literal ring all-reduce, unflatten, per bucket of the
    oracle's plan (or of `plan` = (buckets, offset, bnumel)); returns, per
    replica, tensor -> values."""
    p = cfg["p"]
    numel = W.numels(cfg)
    buckets, offset, bnumel = plan if plan is not None else oracle_plan(cfg, red)
    out = [dict() for _ in range(p)]
    for b, members in enumerate(buckets):
        ins = flat_inputs(cfg, members, offset, bnumel[b])
        want, _ = orc.allreduce(ins, bnumel[b], W.divisor(cfg), cfg["dtype"])
        for r in range(p):
            out[r].update(ob.unflatten(want[r], members, offset, numel))
    return out


def check_whole_set(cfg, red, grads, plan=None):
    """Every element of every replica's gradients against the oracle."""
    want = whole_set_expected(cfg, red, plan)
    for r in range(cfg["p"]):
        for t in range(len(grads[r])):
            assert_bit_equal(to_host(grads[r][t]), want[r][t], f"tensor {t} replica {r}")


def sample_indices(n, cs, p, tensor_bounds, rng, k=2000):
    """Every chunk and tensor boundary +-2, the first and last 64 elements,
    and k random indices of an n-element bucket."""
    idx = set(range(min(n, 64))) | set(range(max(0, n - 64), n))
    for c in range(p + 1):
        for d in (-2, -1, 0, 1, 2):
            i = c * cs + d
            if 0 <= i < n:
                idx.add(i)
    for b in tensor_bounds:
        for d in (-2, -1, 0, 1, 2):
            if 0 <= b + d < n:
                idx.add(b + d)
    idx |= set(int(x) for x in rng.integers(0, n, size=min(k, n)))
    return np.array(sorted(idx), dtype=np.int64)


def check_sync_sampled(cfg, red, grads, rng, per_bucket=2000):
    """Compare the synchronised gradients with the oracle on sampled elements
    of every bucket of the oracle's plan."""
    import torch
    p = cfg["p"]
    starts = W.tensor_starts(cfg)
    Dv = W.divisor(cfg)
    buckets, offset, bnumel = oracle_plan(cfg, red)
    for b, members in enumerate(buckets):
        n = bnumel[b]
        offs = [offset[t] for t in members]
        idx = sample_indices(n, orc.chunk_size(n, p), p, offs, rng, per_bucket)
        # element i of the bucket is element i - offset[t] of tensor t
        which = np.searchsorted(np.array(offs), idx, side="right") - 1
        tens = np.array(members)[which]
        within = idx - np.array(offs)[which]
        flat_idx = np.array(starts)[tens] + within
        ins = [W.host_values(cfg, r, flat_idx) for r in range(p)]
        want, _ = orc.allreduce(ins, n, Dv, cfg["dtype"], idx=idx)
        for r in range(p):
            got = np.empty(idx.size, dtype=want[r].dtype)
            for t in np.unique(tens):
                sel = tens == t
                vals = grads[r][t].view(-1)[torch.from_numpy(within[sel]).cuda()]
                got[sel] = to_host(vals)
            assert_bit_equal(got, want[r], f"bucket {b} replica {r}")
            if cfg["dtype"] == "bf16":
                assert_bf16_close(got, want[r])
    return True
