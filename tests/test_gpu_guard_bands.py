"""Guard bands and small exhaustive sizes (GPU).

Every replica and output buffer sits inside an allocation with 4 KiB margins
on both sides, filled with a sentinel pattern. Each collective runs on every
element count n in [0, 70] and rank count p in [1, 9] (n < p included), then
the margins must be untouched and the result equal to the oracle's bit for
bit. This is the overrun check the pool's closed sanitizer would otherwise
give: chunk edges, padding and trim."""
import numpy as np
import pytest

import ring_all_reduce_ddp_gb300 as D
import synth
from oracle import ring as orc
from oracle import trees as ot

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

GUARD = 4096  # bytes each side
SENTINEL = 0xA5
PS = [1, 2, 3, 4, 5, 7, 8, 9]
NS = list(range(0, 71))


class Guarded:
    """n elements of dtype in the middle of a sentinel-filled allocation."""

    def __init__(self, n, dtype, r=0, seed=0, kind="normal", fill=True, shift=0):
        """shift: elements between the margin and the tensor, so that the
        tensor's start can sit off a 16-byte boundary."""
        self.esz = 4 if dtype == "f32" else 2
        self.tdt = torch.float32 if dtype == "f32" else torch.bfloat16
        self.g = GUARD // self.esz + shift
        self.raw = torch.full((2 * GUARD + (max(n, 1) + shift) * self.esz,), SENTINEL, dtype=torch.uint8,
                              device="cuda")
        self.t = self.raw.view(self.tdt)[self.g:self.g + n]
        self.n = n
        if fill and n:
            synth.fill_(self.t, kind, seed, r)

    def margins_intact(self):
        raw = self.raw.cpu().numpy()
        lo = self.g * self.esz
        end = lo + self.n * self.esz
        return bool((raw[:lo] == SENTINEL).all() and (raw[end:] == SENTINEL).all())


def _host(g, dtype):
    t = g.t.detach().cpu()
    return t.view(torch.int16).numpy().view(np.uint16) if dtype == "bf16" else t.numpy()


def _replicas(p, n, dtype, seed):
    gs = [Guarded(n, dtype, r, seed) for r in range(p)]
    return gs, [_host(g, dtype) for g in gs]


def _eq(a, b):
    return np.array_equal(np.asarray(a).view(np.uint8), np.asarray(b).view(np.uint8))


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("algo", [D.DDP_ALGO_FUSED, D.DDP_ALGO_FUSED_TMA, D.DDP_ALGO_RING_STEPS])
def test_allreduce_small_sizes_stay_inside(algo, dtype):
    dt = D.DDP_FLOAT32 if dtype == "f32" else D.DDP_BFLOAT16
    for p in PS:
        for n in NS:
            gs, hosts = _replicas(p, n, dtype, 300 + n)
            D.ddp_allreduce([g.t for g in gs], n, dt, float(p), algo)
            want, _ = orc.allreduce(hosts, n, float(p), dtype)
            for r, g in enumerate(gs):
                assert g.margins_intact(), (p, n, r)
                assert _eq(_host(g, dtype), want[r]), (p, n, r)


@pytest.mark.parametrize("algo", [D.DDP_ALGO_FUSED, D.DDP_ALGO_RING_STEPS])
@pytest.mark.parametrize("own", [D.DDP_OWN_RANK, D.DDP_OWN_RING])
def test_reduce_scatter_small_sizes_stay_inside(own, algo):
    for p in PS:
        for n in NS:
            if own == D.DDP_OWN_RANK and n % p:
                continue
            cs = -(-n // p) if n else 0
            m = n // p if own == D.DDP_OWN_RANK else cs
            gs, hosts = _replicas(p, n, "f32", 400 + n)
            outs = [Guarded(m, "f32", fill=False) for _ in range(p)]
            before = [o.raw.clone() for o in outs]
            D.ddp_reduce_scatter([g.t for g in gs], [o.t for o in outs], n, D.DDP_FLOAT32, 2.0, own, algo)
            want, _ = orc.reduce_scatter(hosts, n, 2.0, ownership="rank" if own == D.DDP_OWN_RANK else "ring")
            for r in range(p):
                assert outs[r].margins_intact(), (p, n, r)
                got = _host(outs[r], "f32")
                k = len(want[r])  # ring ownership writes only the chunk's real elements
                assert _eq(got[:k], want[r]), (p, n, r)
                if k < m:  # trimmed padding: untouched
                    assert torch.equal(outs[r].raw[GUARD + 4 * k:GUARD + 4 * m], before[r][GUARD + 4 * k:GUARD + 4 * m])
                assert gs[r].margins_intact() and _eq(_host(gs[r], "f32"), hosts[r]), (p, n, r)


@pytest.mark.parametrize("algo", [D.DDP_ALGO_FUSED, D.DDP_ALGO_FUSED_TMA, D.DDP_ALGO_RING_STEPS])
def test_allgather_and_broadcast_small_sizes_stay_inside(algo):
    for p in PS:
        for m in range(0, 12):
            gs, hosts = _replicas(p, m, "f32", 500 + m)
            outs = [Guarded(p * m, "f32", fill=False) for _ in range(p)]
            D.ddp_allgather([g.t for g in gs], [o.t for o in outs], m, D.DDP_FLOAT32, D.DDP_OWN_RANK, algo)
            want, _ = orc.allgather(hosts)
            for r in range(p):
                assert outs[r].margins_intact(), (p, m, r)
                assert _eq(_host(outs[r], "f32"), want[r]), (p, m, r)
        for nb in list(range(0, 40)) + [4095, 4097]:
            root = (nb * 7) % p
            raws = []
            for r in range(p):
                raw = torch.full((2 * GUARD + max(nb, 1),), SENTINEL, dtype=torch.uint8, device="cuda")
                if nb:
                    raw[GUARD:GUARD + nb] = (torch.arange(nb, device="cuda") * 7 + 31 * r + 1) % 251
                raws.append(raw)
            want = raws[root][GUARD:GUARD + nb].clone()
            D.ddp_broadcast([x[GUARD:GUARD + nb] for x in raws], nb, root, algo)
            for r in range(p):
                h = raws[r].cpu().numpy()
                assert (h[:GUARD] == SENTINEL).all() and (h[GUARD + nb:GUARD + nb + GUARD] == SENTINEL).all(), (p, nb, r)
                assert torch.equal(raws[r][GUARD:GUARD + nb], want), (p, nb, r)


@pytest.mark.parametrize("name", ["rd", "rab", "tree"])
def test_tree_allreduces_small_sizes_stay_inside(name):
    algo, ref = {"rd": (D.DDP_ALGO_RECURSIVE_DOUBLING, ot.recursive_doubling),
                 "rab": (D.DDP_ALGO_RABENSEIFNER, ot.rabenseifner),
                 "tree": (D.DDP_ALGO_TREE, ot.tree)}[name]
    for p in PS:
        if name != "tree" and p & (p - 1):
            continue
        for n in NS:
            for dtype, dt in (("f32", D.DDP_FLOAT32), ("bf16", D.DDP_BFLOAT16)):
                gs, hosts = _replicas(p, n, dtype, 700 + n)
                D.ddp_allreduce([g.t for g in gs], n, dt, float(p), algo)
                want, _ = ref(hosts, n, float(p), dtype)
                for r, g in enumerate(gs):
                    assert g.margins_intact(), (p, n, r, dtype)
                    assert _eq(_host(g, dtype), want[r]), (p, n, r, dtype)


def test_in_place_bucket_small_tensors_stay_inside():
    """Buckets of 1..6 tiny tensors (0..9 elements each): every tensor in its
    own guarded allocation; margins intact and the flatten-path bits."""
    from oracle import buckets as ob
    rng = np.random.default_rng(9)
    for p in PS:
        for case in range(12):
            k = int(rng.integers(1, 7))
            sizes = [int(x) for x in rng.integers(0, 10, size=k)]
            n = sum(sizes)
            offs = [int(x) for x in np.cumsum([0] + sizes[:-1])]
            gs = [[Guarded(sz, "f32", r * 10 + j, 800 + case) for j, sz in enumerate(sizes)] for r in range(p)]
            hosts = [[_host(g, "f32") for g in row] for row in gs]
            D.ddp_bucket_allreduce([[g.t for g in row] for row in gs], sizes, offs, D.DDP_FLOAT32, float(p))
            members = list(range(k))
            ins = [ob.flatten(hosts[r], members, offs, n) for r in range(p)]
            want, _ = orc.allreduce(ins, n, float(p))
            for r in range(p):
                back = ob.unflatten(want[r], members, offs, sizes)
                for j in range(k):
                    assert gs[r][j].margins_intact(), (p, case, r, j)
                    assert _eq(_host(gs[r][j], "f32"), back[j]), (p, case, r, j)


@pytest.mark.parametrize("form", ["register", "staged", "step"])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_reducer_table_forms_stay_inside(dtype, form):
    """The Reducer's one-launch piece-table kernel, register form
    (DDP_ALGO_FUSED_LDST), staged form (DDP_ALGO_FUSED_TMA) and the default
    one-launch step with attached buffers, at p = 2, 3, 4, 8 and 16: tensors
    of 0..1,299 elements (up to three 2 KB tiles), each in its own guarded
    allocation, starting 0-3 elements off a 16-byte boundary by the same
    amount on every replica (the staged form's bulk copies) or, in every
    other case, by an amount that differs between replicas (the scalar path).
    Small caps give several buckets. Margins intact, gradients equal to the
    oracle's flatten + ring + unflatten on the oracle's own plan, buffers
    equal to the root's bytes."""
    from oracle import buckets as ob
    from oracle.bf16 import bf16_to_f32, f32_to_bf16
    from ring_all_reduce_ddp_gb300.reducer import Reducer
    esz = 4 if dtype == "f32" else 2
    rng = np.random.default_rng(13 if dtype == "f32" else 14)
    algo = {"register": D.DDP_ALGO_FUSED_LDST, "staged": D.DDP_ALGO_FUSED_TMA, "step": None}[form]
    for p in (2, 3, 4, 8, 16):
        for case in range(4):
            k = int(rng.integers(1, 9))
            sizes = [int(x) for x in rng.integers(0, 1300, size=k)]
            skew = case % 2 == 1
            shift = [[(3 * t + (r if skew else 0)) % 4 for t in range(k)] for r in range(p)]
            gs = [[Guarded(sz, dtype, r * 10 + t, 1300 + case, shift=shift[r][t]) for t, sz in enumerate(sizes)]
                  for r in range(p)]
            hosts = [[_host(g, dtype) for g in row] for row in gs]
            first, cap = 1024, 4096
            red = Reducer([[g.t for g in row] for row in gs], first, cap)
            plan = ob.assign_buckets(sizes, esz, first, cap, "reversed")
            _, offset, bnumel = ob.bucket_layout(sizes, plan)
            assert red.buckets == plan
            bufs = None
            if form == "step":
                bsizes = [int(x) for x in rng.integers(0, 700, size=3)]
                bufs = [[Guarded(sz, "f32", r * 10 + j, 1400 + case, kind="uniform", shift=(j + r) % 4)
                         for j, sz in enumerate(bsizes)] for r in range(p)]
                want_b = [_host(g, "f32") for g in bufs[p - 1]]
                red.set_buffers([[g.t for g in row] for row in bufs], p - 1)
                red.step(float(p))
            else:
                red.sync_gradients(float(p), algo, D.DDP_SYNC_IN_PLACE)
            torch.cuda.synchronize()
            for b, members in enumerate(plan):
                wide = [[bf16_to_f32(h) if dtype == "bf16" else h for h in hosts[r]] for r in range(p)]
                ins = [ob.flatten(wide[r], members, offset, bnumel[b]) for r in range(p)]
                if dtype == "bf16":
                    ins = [f32_to_bf16(x) for x in ins]
                want, _ = orc.allreduce(ins, bnumel[b], float(p), dtype)
                for r in range(p):
                    back = ob.unflatten(want[r], members, offset, sizes)
                    for t in members:
                        assert gs[r][t].margins_intact(), (p, case, r, t)
                        assert _eq(_host(gs[r][t], dtype), back[t]), (p, case, r, t)
            if bufs is not None:
                for r in range(p):
                    for j, g in enumerate(bufs[r]):
                        assert g.margins_intact(), (p, case, r, j)
                        assert _eq(_host(g, "f32"), want_b[j]), (p, case, r, j)
            red.destroy()
            assert D.ddp_device_error() == 0


def test_persistent_ring_small_sizes_stay_inside():
    for p in PS:
        for n in NS:
            gs, hosts = _replicas(p, n, "f32", 900 + n)
            D.ddp_allreduce_persistent([g.t for g in gs], n, D.DDP_FLOAT32, float(p), 50_000_000)
            want, _ = orc.allreduce(hosts, n, float(p))
            for r, g in enumerate(gs):
                assert g.margins_intact(), (p, n, r)
                assert _eq(_host(g, "f32"), want[r]), (p, n, r)
    assert D.ddp_device_error() == 0
