"""Subnormal inputs through every reduction form (GPU).

The library is built without flush-to-zero and with IEEE division, so sums
and quotients that fall in the subnormal range must keep their bits, as the
oracle's numpy arithmetic does: the reading that denormals are preserved on
both sides. Inputs mix normal values, subnormal values and exact zeros of
both signs; every result is compared with the oracle bit for bit."""
import numpy as np
import pytest

import ring_all_reduce_ddp_gb300 as D
import synth
from oracle import buckets as ob
from oracle import ring as orc
from tests.helpers import assert_bit_equal, to_host

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def _tiny_values(p, n, seed):
    """p host arrays: uniforms scaled into the subnormal range (2^-130 and
    below), a few normal values, and signed zeros."""
    out = []
    for r in range(p):
        u = synth.values_np("uniform", seed, r, np.arange(n))
        x = (u.astype(np.float64) * 2.0 ** -130).astype(np.float32)  # subnormal: below 2^-126
        x[::17] = u[::17]                      # some normal values
        x[5::23] = np.float32(0.0)
        x[7::29] = np.float32(-0.0)
        out.append(x)
    return out


def _device(hosts):
    return [torch.from_numpy(h.copy()).cuda() for h in hosts]


@pytest.mark.parametrize("p", [2, 3, 8])
@pytest.mark.parametrize("algo", [D.DDP_ALGO_FUSED, D.DDP_ALGO_RING_STEPS, D.DDP_ALGO_TREE])
def test_flat_allreduce_keeps_subnormals(p, algo):
    n = 4099
    hosts = _tiny_values(p, n, 3100 + p)
    assert np.any((hosts[0] != 0) & (np.abs(hosts[0]) < np.finfo(np.float32).tiny))
    devs = _device(hosts)
    D.ddp_allreduce(devs, n, D.DDP_FLOAT32, float(p), algo)
    torch.cuda.synchronize()
    if algo == D.DDP_ALGO_TREE:
        from oracle import trees
        want, _ = trees.tree(hosts, n, float(p))
    else:
        want, _ = orc.allreduce(hosts, n, float(p))
    for r in range(p):
        assert_bit_equal(to_host(devs[r]), want[r], f"rank {r}")


@pytest.mark.parametrize("p", [2, 8])
def test_in_place_bucket_keeps_subnormals(p):
    """The in-place bucket all-reduce (the one-launch step's kernel body) on
    three tensors whose values sit in the subnormal range."""
    sizes = [1000, 37, 5001]
    n = sum(sizes)
    flat_hosts = _tiny_values(p, n, 3200 + p)
    grads, hosts = [], []
    for r in range(p):
        row, hrow, pos = [], [], 0
        for sz in sizes:
            h = flat_hosts[r][pos:pos + sz].copy()
            row.append(torch.from_numpy(h).cuda())
            hrow.append(h)
            pos += sz
        grads.append(row)
        hosts.append(hrow)
    members = [2, 1, 0]  # reversed registration order, as the Reducer walks
    offset = [0] * 3
    pos = 0
    for t in members:
        offset[t] = pos
        pos += sizes[t]
    D.ddp_bucket_allreduce([[grads[r][t] for t in members] for r in range(p)], [sizes[t] for t in members],
                           [offset[t] for t in members], D.DDP_FLOAT32, float(p))
    torch.cuda.synchronize()
    ins = [ob.flatten(hosts[r], members, offset, n) for r in range(p)]
    want, _ = orc.allreduce(ins, n, float(p))
    for r in range(p):
        back = ob.unflatten(want[r], members, offset, sizes)
        for t in members:
            assert_bit_equal(to_host(grads[r][t]), back[t], f"tensor {t} replica {r}")
    assert D.ddp_device_error() == 0


@pytest.mark.parametrize("algo", [D.DDP_ALGO_FUSED_LDST, D.DDP_ALGO_FUSED_TMA])
@pytest.mark.parametrize("p", [2, 4, 8, 16])
def test_reducer_table_forms_keep_subnormals(p, algo):
    """The whole-Reducer in-place sync, register and shared-memory staged
    forms, on three tensors whose values sit in the subnormal range."""
    from ring_all_reduce_ddp_gb300.reducer import Reducer
    sizes = [1000, 37, 5001]
    n = sum(sizes)
    flat_hosts = _tiny_values(p, n, 3300 + p)
    grads, hosts = [], []
    for r in range(p):
        row, hrow, pos = [], [], 0
        for sz in sizes:
            h = flat_hosts[r][pos:pos + sz].copy()
            row.append(torch.from_numpy(h).cuda())
            hrow.append(h)
            pos += sz
        grads.append(row)
        hosts.append(hrow)
    red = Reducer(grads, 1 << 20, 25 << 20)
    plan = ob.assign_buckets(sizes, 4, 1 << 20, 25 << 20, "reversed")
    _, offset, bnumel = ob.bucket_layout(sizes, plan)
    assert red.buckets == plan == [[2, 1, 0]]
    red.sync_gradients(float(p), algo, D.DDP_SYNC_IN_PLACE)
    torch.cuda.synchronize()
    members = plan[0]
    ins = [ob.flatten(hosts[r], members, offset, bnumel[0]) for r in range(p)]
    want, _ = orc.allreduce(ins, bnumel[0], float(p))
    for r in range(p):
        back = ob.unflatten(want[r], members, offset, sizes)
        for t in members:
            assert_bit_equal(to_host(grads[r][t]), back[t], f"tensor {t} replica {r}")
    red.destroy()
    assert D.ddp_device_error() == 0
