"""Readiness-driven bucket all-reduces on a communication stream (GPU).

Gradients are marked ready one by one, each with an event recorded on the
producing stream; the Reducer must fire buckets strictly in order exactly
when the oracle's replay of mark_variable_ready / mark_bucket_ready says,
and the result must be the bits of a whole-set sync. A rebuild from the
observed ready order must give the oracle's rebuilt buckets and still reduce
to the oracle's values."""
import numpy as np
import pytest

import ring_all_reduce_ddp_gb300 as D
from oracle import buckets as ob
from oracle import reducer_sim as rs
from oracle import ring as orc
from ring_all_reduce_ddp_gb300.reducer import Reducer
from synth import workloads as W
from tests.helpers import assert_bit_equal, to_host
from tests.oracle_sync import check_sync_sampled, check_whole_set, oracle_plan

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def _fire_positions(red, order, divisor, comm, compute):
    seq = []
    fired_total = 0
    for pos, t in enumerate(order):
        ev = torch.cuda.Event()
        ev.record(compute)
        n = red.mark_ready(t, divisor, ev, comm)
        seq += [(pos, fired_total + i) for i in range(n)]
        fired_total += n
    return seq


@pytest.mark.parametrize("comm_blocks", [0, 5, 96])
@pytest.mark.parametrize("name", ["tiny", "resnet50"])
@pytest.mark.parametrize("shuffle", [False, True])
def test_mark_ready_fires_like_the_reducer_and_reduces_like_the_oracle(name, shuffle, comm_blocks):
    """Firing positions against the oracle's replay; values against the
    oracle's ring on the oracle's own bucket plan (every element of the tiny
    set, sampled elements of the ResNet-50-shaped one) and against a
    whole-set sync of the same inputs. With a grid cap the bucket launches
    stride over their tiles with that many blocks: the same bits."""
    cfg = W.CONFIGS[name]
    grads, _ = W.make_grads(cfg)
    ref_grads, _ = W.make_grads(cfg)
    red = Reducer(grads, cfg["first_cap"], cfg["cap"])
    red.set_comm_blocks(comm_blocks)
    ref = Reducer(ref_grads, cfg["first_cap"], cfg["cap"])
    Dv = W.divisor(cfg)
    ref.sync_gradients(Dv, D.DDP_ALGO_FUSED, D.DDP_SYNC_IN_PLACE)
    k = len(grads[0])
    order = list(range(k))[::-1]
    if shuffle:
        order = [int(x) for x in np.random.default_rng(3).permutation(k)]
    comm = torch.cuda.Stream()
    compute = torch.cuda.current_stream()
    red.prepare()
    seq = _fire_positions(red, order, Dv, comm, compute)
    torch.cuda.synchronize()
    plan, _, _ = oracle_plan(cfg, red)
    assert seq == rs.fire_sequence(plan, order)
    assert red.observed() == order
    if name == "tiny":
        check_whole_set(cfg, red, grads)
    else:
        check_sync_sampled(cfg, red, grads, np.random.default_rng(4), per_bucket=1000)
    for r in range(cfg["p"]):
        for t in range(k):
            assert torch.equal(grads[r][t].view(torch.int32), ref_grads[r][t].view(torch.int32)), (r, t)
    with pytest.raises(D.DDPError) as e:
        red.mark_ready(order[0], Dv, None, comm)
    assert e.value.status == D.DDP_ERR_STATE
    assert D.ddp_device_error() == 0


def test_rebuild_from_the_observed_order():
    cfg = W.CONFIGS["tiny"]
    p = cfg["p"]
    grads, _ = W.make_grads(cfg)
    red = Reducer(grads, cfg["first_cap"], cfg["cap"])
    numel = W.numels(cfg)
    observed = [9, 0, 8, 1, 7, 2, 6, 3, 5, 4]
    red.prepare()
    comm = torch.cuda.Stream()
    for t in observed:  # readiness only: the in-place reduction of this pass is checked above
        red.mark_ready(t, 1.0, None, comm)
    torch.cuda.synchronize()
    assert red.assign()  # the per-step host check of the default plan
    red.rebuild()  # along the observed order
    want_buckets = rs.rebuild(numel, 4, cfg["first_cap"], cfg["cap"], observed)
    assert red.buckets == want_buckets
    assert red.assign()  # and of the rebuilt one
    # fresh gradients, one sync on the rebuilt buckets, every element against the oracle
    fresh, _ = W.make_grads(cfg)
    for r in range(p):
        for t in range(len(numel)):
            grads[r][t].copy_(fresh[r][t])
    red.sync_gradients(W.divisor(cfg), D.DDP_ALGO_FUSED, D.DDP_SYNC_IN_PLACE)
    torch.cuda.synchronize()
    starts = W.tensor_starts(cfg)
    _, offset, bnumel = ob.bucket_layout(numel, want_buckets)
    for b, members in enumerate(want_buckets):
        ins = []
        for r in range(p):
            hv = {t: W.host_values(cfg, r, np.arange(starts[t], starts[t] + numel[t])) for t in members}
            ins.append(ob.flatten([hv.get(t, np.zeros(0, np.float32)) for t in range(len(numel))], members,
                                  offset, bnumel[b]))
        want, _ = orc.allreduce(ins, bnumel[b], W.divisor(cfg))
        for r in range(p):
            back = ob.unflatten(want[r], members, offset, numel)
            for t in members:
                assert_bit_equal(to_host(grads[r][t]), back[t], f"tensor {t} replica {r}")


@pytest.mark.parametrize("name", ["tiny", "resnet50"])
def test_step_captured_in_a_cuda_graph_replays_bit_exactly(name):
    """The per-forward buffer broadcast and the in-place sync make no
    allocation and no synchronisation, so one step captures into a CUDA graph;
    replaying it gives the bits of the eager step."""
    from ring_all_reduce_ddp_gb300.reducer import BufferSync
    cfg = W.CONFIGS[name]
    p = cfg["p"]
    Dv = W.divisor(cfg)
    eager, _ = W.make_grads(cfg)
    graphed, _ = W.make_grads(cfg)
    red_e = Reducer(eager, cfg["first_cap"], cfg["cap"])
    red_g = Reducer(graphed, cfg["first_cap"], cfg["cap"])
    bufs_e = W.buffer_set(cfg) if cfg.get("buffers") else None
    bufs_g = W.buffer_set(cfg) if cfg.get("buffers") else None
    bs_e = BufferSync(bufs_e) if bufs_e else None
    bs_g = BufferSync(bufs_g) if bufs_g else None
    # warm up (first-use lookups happen outside the capture), then restore the inputs
    red_g.sync_gradients(Dv)
    fresh, _ = W.make_grads(cfg)
    torch.cuda.synchronize()
    for r in range(p):
        for t in range(len(fresh[r])):
            graphed[r][t].copy_(fresh[r][t])
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        if bs_g:
            bs_g()
        red_g.sync_gradients(Dv)
    for r in range(p):  # capture does not run the work: inputs are still the fresh ones
        for t in range(len(fresh[r])):
            assert torch.equal(graphed[r][t], fresh[r][t])
    g.replay()
    if bs_e:
        bs_e()
    red_e.sync_gradients(Dv)
    torch.cuda.synchronize()
    for r in range(p):
        for t in range(len(eager[r])):
            assert torch.equal(graphed[r][t].view(torch.int16 if graphed[r][t].dtype == torch.bfloat16
                                                  else torch.int32),
                               eager[r][t].view(torch.int16 if eager[r][t].dtype == torch.bfloat16 else torch.int32))
    if bufs_e:
        for r in range(p):
            for j in range(len(bufs_e[r])):
                assert torch.equal(bufs_g[r][j], bufs_e[r][j])


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_collectives_capture_into_cuda_graphs(dtype):
    """Every collective form captures into a CUDA graph (including the
    stream-ordered workspaces of the literal and bf16 paths, which become graph
    memory nodes) and a replay gives the bits of the same call run eagerly."""
    from tests.helpers import make_replicas
    p, n = 8, 100003
    tdt = D.DDP_FLOAT32 if dtype == "f32" else D.DDP_BFLOAT16
    cases = [("allreduce", a) for a in (D.DDP_ALGO_FUSED, D.DDP_ALGO_FUSED_TMA, D.DDP_ALGO_RING_STEPS,
                                        D.DDP_ALGO_RECURSIVE_DOUBLING, D.DDP_ALGO_RABENSEIFNER, D.DDP_ALGO_TREE)]
    cases += [("reduce_scatter", a) for a in (D.DDP_ALGO_FUSED, D.DDP_ALGO_RING_STEPS)]
    cases += [("allgather", a) for a in (D.DDP_ALGO_FUSED, D.DDP_ALGO_RING_STEPS)]
    view = torch.int32 if dtype == "f32" else torch.int16
    for op, algo in cases:
        eager, _, _ = make_replicas(p, n, dtype, "normal", seed=77)
        graphed, _, _ = make_replicas(p, n, dtype, "normal", seed=77)
        m = -(-n // p)
        outs_e = [torch.zeros(p * m, dtype=eager[0].dtype, device="cuda") for _ in range(p)]
        outs_g = [torch.zeros(p * m, dtype=eager[0].dtype, device="cuda") for _ in range(p)]

        def call(bufs, outs, stream=None):
            if op == "allreduce":
                D.ddp_allreduce(bufs, n, tdt, float(p), algo, stream)
            elif op == "reduce_scatter":
                D.ddp_reduce_scatter(bufs, outs, n, tdt, float(p), D.DDP_OWN_RING, algo, stream)
            else:
                D.ddp_allgather([b[:m] for b in bufs], outs, m, tdt, D.DDP_OWN_RANK, algo, stream)

        call(eager, outs_e)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            call(graphed, outs_g)
        g.replay()
        torch.cuda.synchronize()
        for r in range(p):
            assert torch.equal(graphed[r].view(view), eager[r].view(view)), (op, algo, r)
            assert torch.equal(outs_g[r].view(view), outs_e[r].view(view)), (op, algo, r)
        del g
    assert D.ddp_device_error() == 0


def test_comm_blocks_must_not_be_negative():
    cfg = W.CONFIGS["tiny"]
    grads, _ = W.make_grads(cfg)
    red = Reducer(grads, cfg["first_cap"], cfg["cap"])
    with pytest.raises(D.DDPError) as e:
        red.set_comm_blocks(-1)
    assert e.value.status == D.DDP_ERR_ARG


def test_first_use_of_the_staged_kernels_inside_a_capture():
    """In a fresh process, the staged in-place sync and the staged flat
    all-reduce are first launched inside a CUDA graph capture (they set no
    function attribute and allocate nothing on first use); the replay gives
    the eager bits."""
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    code = """
import torch
import ring_all_reduce_ddp_gb300 as D
from ring_all_reduce_ddp_gb300.reducer import Reducer
from synth import workloads as W
cfg = dict(W.CONFIGS["tiny"], p=8)
sets = [W.make_grads_from_host(cfg, p=8)[0] for _ in range(2)]
reds = [Reducer(g, cfg["first_cap"], cfg["cap"]) for g in sets]
assert reds[0].staged()
n = (1 << 20) + 3
flats = [[torch.arange(n, device="cuda", dtype=torch.float32) * (r + 1) / 7 for r in range(8)] for _ in range(2)]
torch.cuda.synchronize()
g = torch.cuda.CUDAGraph()
with torch.cuda.graph(g):
    reds[0].sync_gradients(8.0)
    D.ddp_allreduce(flats[0], n, D.DDP_FLOAT32, 8.0, D.DDP_ALGO_FUSED_TMA)
g.replay()
reds[1].sync_gradients(8.0)
D.ddp_allreduce(flats[1], n, D.DDP_FLOAT32, 8.0, D.DDP_ALGO_FUSED_TMA)
torch.cuda.synchronize()
for r in range(8):
    for a, b in zip(sets[0][r], sets[1][r]):
        assert torch.equal(a.view(torch.int32), b.view(torch.int32))
    assert torch.equal(flats[0][r].view(torch.int32), flats[1][r].view(torch.int32))
assert D.ddp_device_error() == 0
print("ok")
"""
    r = subprocess.run([sys.executable, "-c", code], cwd=root, capture_output=True, text=True, timeout=300,
                       env=dict(os.environ, PYTHONPATH=root))
    assert r.returncode == 0 and r.stdout.strip().endswith("ok"), r.stderr[-2000:]
