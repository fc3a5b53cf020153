"""The Reducer's one-launch step (GPU): the attached per-forward buffers
copied from the root to every other replica, and every bucket's in-place
sync, in one launch.

Gradients are checked against the oracle's flatten + literal ring +
unflatten on the oracle's own bucket plan; buffers against the oracle's
coalesced broadcast of the same bytes. The root's buffers must stay as they
were, and every buffer sits inside an allocation with sentinel margins that
must stay intact."""
import numpy as np
import pytest

import ring_all_reduce_ddp_gb300 as D
import synth
from oracle import ring as orc
from ring_all_reduce_ddp_gb300.reducer import Reducer
from synth import workloads as W
from tests.oracle_sync import check_sync_sampled, check_whole_set

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

GUARD = 4096
SENTINEL = 0x5A
# (dtype, elements): BatchNorm-like running stats and counters, odd sizes, an
# empty one, a few that span several tiles
BUFFER_SPECS = [("f32", 64), ("f32", 64), ("i64", 1), ("f32", 1), ("f32", 3), ("i64", 5), ("f32", 1000),
                ("f32", 0), ("f32", 5000), ("i64", 2049), ("f32", 70001)]
BF16_EXTRA = [("bf16", 3), ("bf16", 1), ("bf16", 4099)]  # 2-byte multiples, for bf16 gradient sets
TDT = {"f32": torch.float32, "i64": torch.int64, "bf16": torch.bfloat16}
ESZ = {"f32": 4, "i64": 8, "bf16": 2}


class GuardedBuffer:
    """A buffer of `n` elements inside a sentinel-filled allocation, holding
    replica r's own seeded bytes."""

    def __init__(self, dt, n, r, j, seed):
        nb = n * ESZ[dt]
        self.raw = torch.full((2 * GUARD + nb,), SENTINEL, dtype=torch.uint8, device="cuda")
        self.t = self.raw[GUARD:GUARD + nb].view(TDT[dt])
        self.nbytes = nb
        vals = synth.values_np("uniform", seed, 5000 + 100 * r + j, np.arange(max(1, nb // 4)))
        host = np.frombuffer(vals.tobytes(), dtype=np.uint8)[:nb].copy()
        if host.size < nb:
            host = np.resize(host, nb)
        self.raw[GUARD:GUARD + nb].copy_(torch.from_numpy(host))
        self.host = host

    def bytes_now(self):
        return self.raw[GUARD:GUARD + self.nbytes].cpu().numpy()

    def margins_intact(self):
        raw = self.raw.cpu().numpy()
        return bool((raw[:GUARD] == SENTINEL).all() and (raw[GUARD + self.nbytes:] == SENTINEL).all())


def _buffers(p, specs, seed=71):
    return [[GuardedBuffer(dt, n, r, j, seed) for j, (dt, n) in enumerate(specs)] for r in range(p)]


def _check_buffers(bufs, root):
    p = len(bufs)
    want, _ = orc.broadcast_coalesced([[b.host for b in row] for row in bufs], root)
    for r in range(p):
        for j, b in enumerate(bufs[r]):
            assert b.margins_intact(), f"buffer {j} of replica {r}: margin written"
            assert np.array_equal(b.bytes_now(), want[r][j]), f"buffer {j} of replica {r}"
    for j, b in enumerate(bufs[root]):
        assert np.array_equal(b.bytes_now(), b.host), f"root buffer {j} changed"


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("p", [1, 2, 3, 4, 8, 16, 17, 256])
def test_step_on_the_tiny_set_with_buffers(p, dtype):
    cfg = dict(W.CONFIGS["tiny"], dtype=dtype, p=p)
    grads, _ = W.make_grads(cfg, p=p)
    red = Reducer(grads, cfg["first_cap"], cfg["cap"])
    specs = BUFFER_SPECS + (BF16_EXTRA if dtype == "bf16" else [])
    for root in sorted({0, p - 1, p // 2}):
        fresh, _ = W.make_grads(cfg, p=p)  # the seeded inputs again, for every root
        for r in range(p):
            for t, g in enumerate(fresh[r]):
                grads[r][t].copy_(g)
        bufs = _buffers(p, specs, seed=71 + root)
        red.set_buffers([[b.t for b in row] for row in bufs], root)
        red.step(W.divisor(cfg))
        torch.cuda.synchronize()
        check_whole_set(cfg, red, grads)
        _check_buffers(bufs, root)
    assert D.ddp_device_error() == 0


def test_in_place_sync_leaves_attached_buffers_alone():
    cfg = W.CONFIGS["tiny"]
    p = cfg["p"]
    grads, _ = W.make_grads(cfg)
    red = Reducer(grads, cfg["first_cap"], cfg["cap"])
    bufs = _buffers(p, BUFFER_SPECS)
    red.set_buffers([[b.t for b in row] for row in bufs], 0)
    red.sync_gradients(W.divisor(cfg))
    torch.cuda.synchronize()
    check_whole_set(cfg, red, grads)
    for r in range(p):
        for j, b in enumerate(bufs[r]):
            assert np.array_equal(b.bytes_now(), b.host) and b.margins_intact(), (r, j)
    # detached again, the step is the in-place sync alone
    red.set_buffers([], 0)
    red.step(W.divisor(cfg))
    torch.cuda.synchronize()
    for r in range(p):
        for j, b in enumerate(bufs[r]):
            assert np.array_equal(b.bytes_now(), b.host), (r, j)


def test_step_on_the_resnet50_set_with_its_batchnorm_buffers():
    """The bench's step: 161 gradients on 8 replicas and the 159 BatchNorm
    buffers (fp32 running statistics, int64 counters) from replica 0."""
    cfg = W.CONFIGS["resnet50"]
    p = cfg["p"]
    grads, _ = W.make_grads(cfg)
    bufs = W.buffer_set(cfg)
    host = [[b.detach().cpu().view(-1).view(torch.uint8).numpy().copy() for b in row] for row in bufs]
    red = Reducer(grads, cfg["first_cap"], cfg["cap"])
    nbytes = red.set_buffers(bufs, 0)
    assert nbytes == sum(h.size for h in host[0])
    red.step(W.divisor(cfg))
    torch.cuda.synchronize()
    check_sync_sampled(cfg, red, grads, np.random.default_rng(21), per_bucket=1000)
    want, _ = orc.broadcast_coalesced(host, 0)
    for r in range(p):
        for j, b in enumerate(bufs[r]):
            assert np.array_equal(b.detach().cpu().view(-1).view(torch.uint8).numpy(), want[r][j]), (r, j)
    assert D.ddp_device_error() == 0


def test_step_argument_errors():
    cfg = W.CONFIGS["tiny"]
    p = cfg["p"]
    grads, _ = W.make_grads(cfg)
    red = Reducer(grads, cfg["first_cap"], cfg["cap"])
    bufs = _buffers(p, BUFFER_SPECS[:3])
    rows = [[b.t for b in row] for row in bufs]

    def status(fn):
        with pytest.raises(D.DDPError) as e:
            fn()
        return e.value.status

    # a buffer that is a gradient of the reducer
    assert status(lambda: red.set_buffers([[grads[r][0]] for r in range(p)], 0)) == D.DDP_ERR_ARG
    # two replicas' buffers overlapping
    assert status(lambda: red.set_buffers([[rows[0][0]]] + [[rows[r][0]] for r in range(p - 1)], 0)) == D.DDP_ERR_ARG
    # root out of range
    assert status(lambda: red.set_buffers(rows, p)) == D.DDP_ERR_ARG
    # fp32 gradients: a buffer of 6 bytes is not a whole number of elements
    odd = [torch.zeros(3, dtype=torch.bfloat16, device="cuda") for _ in range(p)]
    assert status(lambda: red.set_buffers([[o] for o in odd], 0)) == D.DDP_ERR_ARG
    # a buffer 2 bytes off a 4-byte boundary
    base = [torch.zeros(9, dtype=torch.bfloat16, device="cuda") for _ in range(p)]
    assert status(lambda: red.set_buffers([[b[1:3]] for b in base], 0)) == D.DDP_ERR_ALIGN
    # nothing was attached by the failed calls: the step is the sync alone
    red.step(W.divisor(cfg))
    torch.cuda.synchronize()
    check_whole_set(cfg, red, grads)
    for r in range(p):
        for j, b in enumerate(bufs[r]):
            assert np.array_equal(b.bytes_now(), b.host), (r, j)


def test_step_buffers_survive_a_rebuild():
    cfg = W.CONFIGS["tiny"]
    p = cfg["p"]
    grads, _ = W.make_grads(cfg)
    red = Reducer(grads, cfg["first_cap"], cfg["cap"])
    bufs = _buffers(p, BUFFER_SPECS, seed=90)
    red.set_buffers([[b.t for b in row] for row in bufs], 1)
    order = [9, 0, 8, 1, 7, 2, 6, 3, 5, 4]
    red.rebuild(order)
    red.step(W.divisor(cfg))
    torch.cuda.synchronize()
    from oracle import buckets as ob
    from oracle import reducer_sim as rs
    plan = rs.rebuild(W.numels(cfg), 4, cfg["first_cap"], cfg["cap"], order)
    assert red.buckets == plan
    _, offset, bnumel = ob.bucket_layout(W.numels(cfg), plan)
    check_whole_set(cfg, red, grads, plan=(plan, offset, bnumel))
    _check_buffers(bufs, 1)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_step_buffers_misaligned_differently_per_replica(dtype):
    """Buffers whose replicas sit at different addresses mod 16 bytes: their
    copy tiles take the element-by-element path. The sizes leave ragged heads
    and tails around the 16-byte words."""
    cfg = dict(W.CONFIGS["tiny"], dtype=dtype)
    p = cfg["p"]
    grads, _ = W.make_grads(cfg)
    red = Reducer(grads, cfg["first_cap"], cfg["cap"])
    esz = 4 if dtype == "f32" else 2
    sizes = [1, 5, 1023, 1025, 4097]  # elements of the gradients' dtype
    keep, rows, hosts = [], [], []
    for r in range(p):
        row, hrow = [], []
        for j, n in enumerate(sizes):
            shift = (r + j) % 4  # elements off the allocation's start: a different offset mod 16 per replica
            raw = torch.zeros((n + 8) * esz, dtype=torch.uint8, device="cuda")
            h = np.frombuffer(synth.values_np("uniform", 77, 900 + 10 * r + j, np.arange(n + 4)).tobytes(),
                              dtype=np.uint8)[:n * esz].copy()
            raw[shift * esz:(shift + n) * esz].copy_(torch.from_numpy(h))
            keep.append(raw)
            row.append(raw[shift * esz:(shift + n) * esz].view(TDT[dtype]))
            hrow.append(h)
        rows.append(row)
        hosts.append(hrow)
    root = 2
    red.set_buffers(rows, root)
    red.step(W.divisor(cfg))
    torch.cuda.synchronize()
    check_whole_set(cfg, red, grads)
    want, _ = orc.broadcast_coalesced(hosts, root)
    for r in range(p):
        for j, t in enumerate(rows[r]):
            got = t.view(torch.uint8).cpu().numpy()
            assert np.array_equal(got, want[r][j]), (r, j)
    assert D.ddp_device_error() == 0


def test_step_with_empty_gradients_and_a_tiny_cap():
    """Zero-size gradient tensors (no storage) among others, a cap that
    closes a bucket after every tensor, p = 3: the in-place sync and the
    one-launch step skip the empty tensors and reduce the rest like the
    oracle."""
    p = 3
    sizes = [0, 5, 0, 1000, 0, 4097, 1]
    grads, hosts = [], []
    for r in range(p):
        row, hrow = [], []
        for j, n in enumerate(sizes):
            h = synth.values_np("normal", 3300, 10 * r + j, np.arange(n))
            row.append(torch.from_numpy(h.copy()).cuda())
            hrow.append(h)
        grads.append(row)
        hosts.append(hrow)
    red = Reducer(grads, 4, 4)  # every non-empty tensor closes its bucket
    bufs = _buffers(p, BUFFER_SPECS[:4], seed=95)
    red.set_buffers([[b.t for b in row] for row in bufs], 0)
    red.step(float(p))
    torch.cuda.synchronize()
    from oracle import buckets as ob
    plan = ob.assign_buckets(sizes, 4, 4, 4)
    assert red.buckets == plan
    _, offset, bnumel = ob.bucket_layout(sizes, plan)
    for b, members in enumerate(plan):
        ins = [ob.flatten(hosts[r], members, offset, bnumel[b]) for r in range(p)]
        want, _ = orc.allreduce(ins, bnumel[b], float(p))
        for r in range(p):
            back = ob.unflatten(want[r], members, offset, sizes)
            for t in members:
                got = grads[r][t].cpu().numpy()
                assert np.array_equal(got.view(np.uint32), back[t].view(np.uint32)), (b, t, r)
    _check_buffers(bufs, 0)
    assert D.ddp_device_error() == 0
