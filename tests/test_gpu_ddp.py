"""GPU parity of the DDP path: bucket flatten / unflatten, the literal schedule
step by step (state after every step, bytes on the wire), and whole gradient
synchronisations on the four gradient sets, against the CPU oracle.

Full-size sets are checked on sampled elements (every chunk and tensor
boundary +-2, the first and last 64 elements of each bucket, and random
indices), each computed by the oracle's own ring simulation restricted to
those elements, from inputs regenerated on the host by the seeded generator."""
import numpy as np
import pytest

import ring_all_reduce_ddp_gb300 as D
from oracle import buckets as ob
from oracle import ring as orc
from oracle.bf16 import bf16_to_f32
from ring_all_reduce_ddp_gb300.reducer import Reducer, broadcast_buffers
from synth import workloads as W
from tests.helpers import assert_bit_equal, make_replicas, to_host
from tests.oracle_sync import check_sync_sampled, check_whole_set, oracle_plan

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

DT = {"f32": D.DDP_FLOAT32, "bf16": D.DDP_BFLOAT16}


# ------------------------------------------------------------ flatten / unflatten
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("predivide", [1.0, 4.0, 3.0])
def test_flatten_unflatten_tiny(dtype, predivide):
    cfg = dict(W.CONFIGS["tiny"], dtype=dtype)
    p = cfg["p"]
    grads, _ = W.make_grads(cfg)
    numel = W.numels(cfg)
    starts = W.tensor_starts(cfg)
    plan = ob.assign_buckets(numel, W.esize(cfg), cfg["first_cap"], cfg["cap"])
    _, offset, bnumel = ob.bucket_layout(numel, plan)
    tdt = torch.float32 if dtype == "f32" else torch.bfloat16
    for b, members in enumerate(plan):
        flat = [torch.full((bnumel[b],), 5.0, dtype=tdt, device="cuda") for _ in range(p)]
        D.ddp_bucket_flatten([[grads[r][t] for t in members] for r in range(p)], [numel[t] for t in members],
                             [offset[t] for t in members], flat, DT[dtype], predivide)
        for r in range(p):
            host = {t: W.host_values(cfg, r, np.arange(starts[t], starts[t] + numel[t])) for t in members}
            if dtype == "f32":
                want = ob.flatten([host.get(t, np.zeros(0, np.float32)) for t in range(len(numel))], members,
                                  offset, bnumel[b], predivide)
            else:
                from oracle.bf16 import f32_to_bf16
                wide = [bf16_to_f32(host[t]) if t in host else np.zeros(0, np.float32) for t in range(len(numel))]
                want = f32_to_bf16(ob.flatten(wide, members, offset, bnumel[b], predivide))
            assert_bit_equal(to_host(flat[r]), want, f"bucket {b} replica {r}")
        # unflatten into fresh tensors gives the flat slices back
        outs = [[torch.zeros(numel[t], dtype=tdt, device="cuda") for t in members] for _ in range(p)]
        D.ddp_bucket_unflatten(flat, [numel[t] for t in members], [offset[t] for t in members], outs, DT[dtype])
        for r in range(p):
            fh = to_host(flat[r])
            back = ob.unflatten(fh, members, offset, numel)
            for j, t in enumerate(members):
                assert_bit_equal(to_host(outs[r][j]), back[t], f"tensor {t}")


# ---------------------------------------------------------- literal schedule
@pytest.mark.parametrize("p,n", [(1, 1000), (2, 17), (3, 1000), (4, 277421), (5, 4), (8, 65541), (13, 20011)])
def test_allreduce_steps_fp32_state_after_every_step(p, n):
    devs, hosts, _ = make_replicas(p, n, "f32", "normal", seed=400 + p)
    want, info = orc.allreduce(hosts, n, float(p), "f32", snapshots=True)
    with D.DDPRing(D.DDP_OP_ALLREDUCE, devs, None, n, D.DDP_FLOAT32, float(p)) as ring:
        assert ring.num_steps() == len(info["snapshots"]) == (1 if p == 1 else 2 * (p - 1))
        for s in range(ring.num_steps()):
            ring.step()
            ring.sync()
            for r in range(p):
                assert_bit_equal(to_host(devs[r]), info["snapshots"][s][r][:n], f"step {s} rank {r}")
        for r in range(p):
            assert ring.bytes_sent(r) == info["bytes_sent"][r]
        with pytest.raises(D.DDPError) as e:
            ring.step()
        assert e.value.status == D.DDP_ERR_STATE


@pytest.mark.parametrize("p,n", [(2, 1001), (4, 277421), (8, 65541)])
def test_allreduce_steps_bf16_partials_in_fp32_workspace(p, n):
    devs, hosts, _ = make_replicas(p, n, "bf16", "normal", seed=500 + p)
    want, info = orc.allreduce(hosts, n, float(p), "bf16", snapshots=True)
    cs = info["cs"]
    with D.DDPRing(D.DDP_OP_ALLREDUCE, devs, None, n, D.DDP_BFLOAT16, float(p)) as ring:
        ws_ptr, slot = ring.workspace()
        assert ws_ptr and slot == cs
        for s in range(ring.num_steps()):
            ring.step()
            ring.sync()
            snap = info["snapshots"][s]
            if s < p - 2:  # the partial rank d just received is in slot d of half s & 1
                host_ws = _read_f32(ws_ptr, 2 * p * cs)
                for d in range(p):
                    c = (d - 1 - s) % p
                    lo, hi = c * cs, min(n, (c + 1) * cs)
                    base = ((s & 1) * p + d) * cs
                    assert_bit_equal(host_ws[base:base + max(0, hi - lo)], snap[d][lo:hi], f"step {s} slot {d}")
            else:  # finished chunks are in the buffers, the others still hold the inputs
                done = s - (p - 2)
                for r in range(p):
                    got = bf16_to_f32(to_host(devs[r]))
                    finished = {(r + 1 - j) % p for j in range(done + 1)}
                    for c in range(p):
                        lo, hi = c * cs, min(n, (c + 1) * cs)
                        ref = snap[r][lo:hi] if c in finished else bf16_to_f32(hosts[r][lo:hi])
                        assert_bit_equal(got[lo:hi], ref, f"step {s} rank {r} chunk {c}")
        for r in range(p):
            assert ring.bytes_sent(r) == info["bytes_sent"][r]
    for r in range(p):
        assert_bit_equal(to_host(devs[r]), want[r])


def _read_f32(ptr, count):
    """Copy `count` fp32 values at a raw device pointer to the host."""
    class Raw:
        __cuda_array_interface__ = {"shape": (count,), "typestr": "<f4", "data": (ptr, False), "version": 2}
    return torch.as_tensor(Raw(), device="cuda").cpu().numpy().copy()


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("own", ["rank", "ring"])
@pytest.mark.parametrize("p", [1, 2, 4, 7])
def test_reduce_scatter_and_allgather_handles(p, own, dtype):
    n = 1001 * p + (0 if own == "rank" else 2)
    devs, hosts, _ = make_replicas(p, n, dtype, "uniform", seed=600 + p)
    cs = orc.chunk_size(n, p)
    tdt = torch.float32 if dtype == "f32" else torch.bfloat16
    outs = [torch.zeros(cs, dtype=tdt, device="cuda") for _ in range(p)]
    code = D.DDP_OWN_RANK if own == "rank" else D.DDP_OWN_RING
    want, info = orc.reduce_scatter(hosts, n, 2.0, dtype, own)
    with D.DDPRing(D.DDP_OP_REDUCE_SCATTER, devs, outs, n, DT[dtype], 2.0, code) as ring:
        assert ring.num_steps() == max(1, p - 1)
        while ring.steps_done() < ring.num_steps():
            ring.step()
        ring.sync()
        for r in range(p):
            assert ring.bytes_sent(r) == info["bytes_sent"][r]
    for r in range(p):
        assert_bit_equal(to_host(outs[r])[:len(want[r])], want[r], f"rank {r}")
    if own == "rank" or n % p == 0:
        m = cs
        gathered = [torch.zeros(p * m, dtype=tdt, device="cuda") for _ in range(p)]
        gwant, ginfo = orc.allgather([to_host(o) for o in outs], dtype, own, snapshots=True)
        with D.DDPRing(D.DDP_OP_ALLGATHER, outs, gathered, m, DT[dtype], 1.0, code) as ring:
            for s in range(ring.num_steps()):
                ring.step()
                ring.sync()
                if p > 1:
                    for r in range(p):
                        g = to_host(gathered[r])
                        snap = ginfo["snapshots"][s][r]
                        filled = snap != 0
                        assert_bit_equal(g[filled], snap[filled], f"all-gather step {s} rank {r}")
        for r in range(p):
            assert_bit_equal(to_host(gathered[r]), gwant[r])


@pytest.mark.parametrize("p,root", [(2, 0), (5, 2), (8, 7), (9, 0)])
def test_broadcast_handle_tree_steps(p, root):
    nbytes = 4099
    host = [np.full(nbytes, r, dtype=np.uint8) for r in range(p)]
    devs = [torch.from_numpy(h).cuda() for h in host]
    want, steps, snaps = orc.broadcast_tree(host, root, snapshots=True)
    with D.DDPRing(D.DDP_OP_BROADCAST, devs, None, nbytes, root=root) as ring:
        assert ring.num_steps() == steps
        for s in range(steps):
            ring.step()
            ring.sync()
            for r in range(p):
                assert np.array_equal(devs[r].cpu().numpy(), snaps[s][r]), (s, r)
        sent = [ring.bytes_sent(r) for r in range(p)]
    assert sum(sent) == (p - 1) * nbytes


# ------------------------------------------------------------- whole syncs
SYNCS = [(D.DDP_ALGO_FUSED, D.DDP_SYNC_IN_PLACE), (D.DDP_ALGO_FUSED_TMA, D.DDP_SYNC_IN_PLACE),
         (D.DDP_ALGO_FUSED, D.DDP_SYNC_FLATTEN), (D.DDP_ALGO_FUSED_TMA, D.DDP_SYNC_FLATTEN),
         (D.DDP_ALGO_RING_STEPS, D.DDP_SYNC_FLATTEN)]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("algo,mode", SYNCS)
def test_tiny_ddp_sync_full_parity(algo, mode, dtype):
    """Ten odd-sized tensors, p = 4: every element of every gradient after one sync."""
    cfg = dict(W.CONFIGS["tiny"], dtype=dtype)
    p = cfg["p"]
    grads, _ = W.make_grads(cfg)
    red = Reducer(grads, cfg["first_cap"], cfg["cap"])
    if dtype == "f32":
        assert red.buckets == [[9, 8], [7, 6, 5, 4, 3, 2, 1, 0]]
    red.sync_gradients(W.divisor(cfg), algo, mode)
    torch.cuda.synchronize()
    check_whole_set(cfg, red, grads)
    assert D.ddp_device_error() == 0


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("algo,mode", SYNCS)
def test_tiny_ddp_sync_replicas_misaligned_differently(algo, mode, dtype):
    """The tiny set with each tensor moved 0-2 elements off its allocation's
    start, by an amount that differs between replicas: the in-place sync's
    tiles, whose replicas then differ mod 16 bytes, take the scalar path."""
    cfg = dict(W.CONFIGS["tiny"], dtype=dtype)
    p = cfg["p"]
    src, _ = W.make_grads(cfg)
    keep, grads = [], []
    for r in range(p):
        row = []
        for t, g in enumerate(src[r]):
            base = torch.empty(g.numel() + 3, dtype=g.dtype, device="cuda")
            sh = (t + r) % 3
            v = base[sh:sh + g.numel()]
            v.copy_(g.view(-1))
            keep.append(base)
            row.append(v.view(g.shape))
        grads.append(row)
    red = Reducer(grads, cfg["first_cap"], cfg["cap"])
    red.sync_gradients(W.divisor(cfg), algo, mode)
    torch.cuda.synchronize()
    check_whole_set(cfg, red, grads)
    assert D.ddp_device_error() == 0


@pytest.mark.parametrize("skew", [False, True])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("p", [1, 2, 3, 4, 8, 16, 17, 64])
def test_bucket_allreduce_in_place_matches_flatten_path_oracle(p, dtype, skew):
    """One bucket of odd tensors (some spanning several chunks, some inside one,
    a zero-size one, misaligned offsets) reduced straight on the gradients.
    With skew, a tensor's start differs between replicas mod 16 bytes, so its
    tiles take the scalar path."""
    rng = np.random.default_rng(p)
    sizes = [int(x) for x in rng.integers(0, 3000, size=12)] + [0, 1, 5, 40000]
    order = list(range(len(sizes)))[::-1]
    offset = {}
    pos = 0
    for t in order:
        offset[t] = pos
        pos += sizes[t]
    n = pos
    tdt = torch.float32 if dtype == "f32" else torch.bfloat16
    grads, hosts = [], []
    import synth
    for r in range(p):
        row, hrow = [], []
        for t, sz in enumerate(sizes):
            base = torch.empty(sz + 3, dtype=tdt, device="cuda")
            sh = (t + r) % 3 if skew else t % 3  # misaligned starts, the same on every replica unless skewed
            v = base[sh:sh + sz]
            if sz:
                synth.fill_(v, "normal", 77, r * 100 + t)
            row.append(v)
            hrow.append(synth.values_np("normal", 77, r * 100 + t, np.arange(sz), 1.0, dtype))
        grads.append(row)
        hosts.append(hrow)
    members = order
    D.ddp_bucket_allreduce([[grads[r][t] for t in members] for r in range(p)], [sizes[t] for t in members],
                           [offset[t] for t in members], tdt, float(p))
    torch.cuda.synchronize()
    off_list = [offset.get(t, 0) for t in range(len(sizes))]
    ins = []
    for r in range(p):
        wide = [bf16_to_f32(h) if dtype == "bf16" else h for h in hosts[r]]
        flat = ob.flatten(wide, members, off_list, n)
        if dtype == "bf16":
            from oracle.bf16 import f32_to_bf16
            flat = f32_to_bf16(flat)
        ins.append(flat)
    want, _ = orc.allreduce(ins, n, float(p), dtype)
    for r in range(p):
        back = ob.unflatten(want[r], members, off_list, sizes)
        for t in members:
            assert_bit_equal(to_host(grads[r][t]), back[t], f"tensor {t} replica {r}")
    assert D.ddp_device_error() == 0


@pytest.mark.parametrize("algo", [D.DDP_ALGO_FUSED, D.DDP_ALGO_FUSED_TMA])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("p", [2, 3, 16, 17, 64, 256])
def test_in_place_sync_every_replica_count_branch(p, dtype, algo):
    """The whole-Reducer in-place sync (one launch over the device-resident
    piece table) at replica counts that take each of its compiled forms: p = 2
    and 16 unrolled (register or shared-memory staged), 3, 17, 64 and 256 (the
    largest the library takes) the generic register loop (p = 4 and 8 run in
    the tests above). The tiny set's ten tensors on p replicas, every element
    against the oracle's flatten + ring + unflatten on the oracle's own plan."""
    cfg = dict(W.CONFIGS["tiny"], dtype=dtype, p=p)
    grads, _ = W.make_grads(cfg, p=p)
    red = Reducer(grads, cfg["first_cap"], cfg["cap"])
    red.sync_gradients(W.divisor(cfg), algo, D.DDP_SYNC_IN_PLACE)
    torch.cuda.synchronize()
    check_whole_set(cfg, red, grads)
    assert D.ddp_device_error() == 0


def test_default_in_place_form_per_dtype_and_replica_count():
    """ddp_reducer_staged reports the form DDP_ALGO_FUSED takes in place:
    staged for fp32 at p = 4 and 8 and for bf16 at p = 2 and 4, registers
    elsewhere (the header's table)."""
    want = {("f32", 4), ("f32", 8), ("bf16", 2), ("bf16", 4)}
    for dtype in ("f32", "bf16"):
        for p in (1, 2, 3, 4, 8, 16, 17):
            cfg = dict(W.CONFIGS["tiny"], dtype=dtype, p=p)
            grads, _ = W.make_grads_from_host(cfg, p=p)
            red = Reducer(grads, cfg["first_cap"], cfg["cap"])
            assert red.staged() == ((dtype, p) in want), (dtype, p)
            red.destroy()


@pytest.mark.parametrize("algo,mode", [(D.DDP_ALGO_FUSED, D.DDP_SYNC_IN_PLACE),
                                       (D.DDP_ALGO_FUSED_TMA, D.DDP_SYNC_IN_PLACE),
                                       (D.DDP_ALGO_FUSED, D.DDP_SYNC_FLATTEN)])
@pytest.mark.parametrize("name", ["resnet50", "gpt2_small"])
def test_model_sized_sync_sampled_parity(name, algo, mode):
    """Full-size fp32 gradient sets in the bench's launch configuration."""
    cfg = W.CONFIGS[name]
    grads, _ = W.make_grads(cfg)
    red = Reducer(grads, cfg["first_cap"], cfg["cap"])
    red.sync_gradients(W.divisor(cfg), algo, mode)
    torch.cuda.synchronize()
    check_sync_sampled(cfg, red, grads, np.random.default_rng(5))
    # every replica ends identical (the data-parallel invariant), on whole tensors
    for t in range(len(grads[0])):
        for r in range(1, cfg["p"]):
            assert torch.equal(grads[r][t].view(torch.int32), grads[0][t].view(torch.int32))
    assert D.ddp_device_error() == 0


@pytest.mark.parametrize("one_launch,algo", [(False, D.DDP_ALGO_FUSED), (False, D.DDP_ALGO_FUSED_TMA),
                                             (True, None)])
def test_llama_bf16_sync_and_buffer_broadcast_sampled_parity(one_launch, algo):
    """1.2B bf16 gradients on 8 replicas (about 39 GB with the buckets), and the
    per-forward broadcast of 64 fp32 buffers from replica 0: as two calls (the
    coalesced broadcast, then the in-place sync, register or staged form) and
    as the one-launch step the bench's configs field times. Buffers against
    the oracle's coalesced broadcast of the host-generated bytes."""
    cfg = W.CONFIGS["llama_1b"]
    bufs = W.buffer_set(cfg)
    host = W.buffer_set_host(cfg)
    want_bufs, _ = orc.broadcast_coalesced(host, 0)
    grads, _ = W.make_grads(cfg)
    red = Reducer(grads, cfg["first_cap"], cfg["cap"])
    assert len(red.buckets) == 66
    if one_launch:
        red.set_buffers(bufs, 0)
        red.step(W.divisor(cfg))
    else:
        broadcast_buffers(bufs, 0)
        red.sync_gradients(W.divisor(cfg), algo)
    torch.cuda.synchronize()
    for r in range(cfg["p"]):
        for j, b in enumerate(bufs[r]):
            assert np.array_equal(b.cpu().numpy().view(np.uint8), want_bufs[r][j]), (r, j)
    check_sync_sampled(cfg, red, grads, np.random.default_rng(6), per_bucket=300)
    assert D.ddp_device_error() == 0


@pytest.mark.parametrize("name", ["tiny", "resnet50"])
def test_sync_reads_what_the_kernel_before_it_wrote(name):
    """The whole-Reducer sync is launched as a programmatic dependent of the
    kernel before it, and the coalesced broadcast lets its dependent start
    early. Here that broadcast writes the gradients themselves (replica 0's
    copied to every replica) and the sync follows on the same stream with no
    host synchronisation: the sync must reduce the broadcast values, i.e. p
    copies of replica 0's gradients summed in ring order and divided by D."""
    cfg = W.CONFIGS[name]
    p = cfg["p"]
    grads, _ = W.make_grads(cfg)
    red = Reducer(grads, cfg["first_cap"], cfg["cap"])
    numel = W.numels(cfg)
    starts = W.tensor_starts(cfg)
    s = torch.cuda.current_stream()
    nbytes = [t.numel() * t.element_size() for t in grads[0]]
    for rep in range(3):
        broadcast_buffers(grads, 0, 0, D.DDP_ALGO_FUSED, s)
        red.sync_gradients(W.divisor(cfg), D.DDP_ALGO_FUSED, D.DDP_SYNC_IN_PLACE, 1.0, s)
        if rep == 0:
            torch.cuda.synchronize()
            buckets, offset, bnumel = oracle_plan(cfg, red)
            rng = np.random.default_rng(11)
            for b, members in enumerate(buckets):
                t = members[int(rng.integers(0, len(members)))]
                idx = np.unique(np.concatenate([np.arange(min(64, numel[t])),
                                                rng.integers(0, numel[t], size=min(512, numel[t]))]))
                x0 = W.host_values(cfg, 0, starts[t] + idx)
                # every replica holds replica 0's values: the oracle's ring over p copies of them
                want, _ = orc.allreduce([x0] * p, bnumel[b], W.divisor(cfg), cfg["dtype"], idx=offset[t] + idx)
                for r in range(p):
                    assert_bit_equal(to_host(grads[r][t])[idx], want[r], f"tensor {t} replica {r}")
    torch.cuda.synchronize()
    for t in range(len(numel)):
        for r in range(1, p):
            assert torch.equal(grads[r][t].view(torch.int32), grads[0][t].view(torch.int32))
    assert D.ddp_device_error() == 0


@pytest.mark.parametrize("name", ["tiny", "resnet50"])
def test_ready_firing_reads_what_the_kernel_before_it_wrote(name):
    """Readiness-driven firing launches each bucket as a programmatic dependent
    of the kernel before it: the coalesced broadcast that writes the gradients,
    then the previous bucket. Every bucket must reduce the broadcast values."""
    cfg = W.CONFIGS[name]
    p = cfg["p"]
    grads, _ = W.make_grads(cfg)
    red = Reducer(grads, cfg["first_cap"], cfg["cap"])
    numel = W.numels(cfg)
    starts = W.tensor_starts(cfg)
    s = torch.cuda.current_stream()
    Dv = W.divisor(cfg)
    for rep in range(3):
        broadcast_buffers(grads, 0, 0, D.DDP_ALGO_FUSED, s)
        red.prepare()
        fired = sum(red.mark_ready(t, Dv, None, s) for t in range(len(numel) - 1, -1, -1))
        assert fired == len(red.buckets)
        if rep == 0:
            torch.cuda.synchronize()
            buckets, offset, bnumel = oracle_plan(cfg, red)
            rng = np.random.default_rng(12)
            for b, members in enumerate(buckets):
                for t in members:
                    idx = np.unique(np.concatenate([np.arange(min(64, numel[t])),
                                                    rng.integers(0, numel[t], size=min(256, numel[t]))]))
                    x0 = W.host_values(cfg, 0, starts[t] + idx)
                    want, _ = orc.allreduce([x0] * p, bnumel[b], Dv, cfg["dtype"], idx=offset[t] + idx)
                    for r in range(p):
                        assert_bit_equal(to_host(grads[r][t])[idx], want[r], f"tensor {t} replica {r}")
    torch.cuda.synchronize()
    for t in range(len(numel)):
        for r in range(1, p):
            assert torch.equal(grads[r][t].view(torch.int32), grads[0][t].view(torch.int32))
    assert D.ddp_device_error() == 0
