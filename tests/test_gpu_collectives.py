"""GPU parity: every collective of the C ABI against the CPU oracle, element by
element on the same seeded inputs. fp32 and bf16 results must be bit-exact (the
kernels add in the ring's order and round once); bf16 additionally meets the
stated 1e-5 abs / 1e-6 rel tolerance by implication."""
import numpy as np
import pytest

import ring_all_reduce_ddp_gb300 as D
from oracle import ring as orc
from tests.helpers import assert_bf16_close, assert_bit_equal, make_replicas, to_host

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

ALGOS = [D.DDP_ALGO_FUSED, D.DDP_ALGO_FUSED_LDST, D.DDP_ALGO_FUSED_TMA, D.DDP_ALGO_RING_STEPS]
DT = {"f32": D.DDP_FLOAT32, "bf16": D.DDP_BFLOAT16}

# (p, n): several tiles and chunks, ragged tails, n < p, n not divisible by p
SIZES = [(1, 1000), (2, 1), (2, 4099), (3, 10007), (4, 277421), (5, 3), (8, 65536 * 3 + 5), (8, 7),
         (16, 100003), (17, 50021), (64, 262147), (256, 70000)]


def _no_device_error():
    assert D.ddp_device_error() == 0


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("algo", ALGOS)
@pytest.mark.parametrize("p,n", SIZES)
def test_allreduce_matches_oracle(p, n, algo, dtype):
    divisor = float(p)
    devs, hosts, _ = make_replicas(p, n, dtype, "normal", seed=100 + p, sigma=1.0)
    D.ddp_allreduce(devs, n, DT[dtype], divisor, algo)
    torch.cuda.synchronize()
    want, _ = orc.allreduce(hosts, n, divisor, dtype)
    for r in range(p):
        got = to_host(devs[r])
        assert_bit_equal(got, want[r], f"replica {r}")
        if dtype == "bf16":
            assert_bf16_close(got, want[r])
    _no_device_error()


@pytest.mark.parametrize("algo", ALGOS)
@pytest.mark.parametrize("offsets", [[1, 1, 1, 1], [0, 1, 2, 3], [3, 0, 0, 2]])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_allreduce_misaligned_replicas(offsets, algo, dtype):
    p, n = 4, 40009
    devs, hosts, _ = make_replicas(p, n, dtype, "uniform", seed=7, offsets=offsets)
    D.ddp_allreduce(devs, n, DT[dtype], 4.0, algo)
    want, _ = orc.allreduce(hosts, n, 4.0, dtype)
    for r in range(p):
        assert_bit_equal(to_host(devs[r]), want[r], f"replica {r}")


@pytest.mark.parametrize("algo", ALGOS)
def test_allreduce_token_count_divisor(algo):
    """Sum-of-loss gradients normalised once by the global token count."""
    import synth
    p, n = 8, 123457
    counts = synth.token_counts(1003, p)
    D_tok = float(sum(counts))
    devs, hosts, _ = make_replicas(p, n, "f32", "normal", seed=1003, sigma=1e-3)
    D.ddp_allreduce(devs, n, D.DDP_FLOAT32, D_tok, algo)
    want, _ = orc.allreduce(hosts, n, D_tok)
    for r in range(p):
        assert_bit_equal(to_host(devs[r]), want[r])


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("algo", ALGOS)
@pytest.mark.parametrize("own", ["rank", "ring"])
@pytest.mark.parametrize("p,n", [(1, 999), (2, 4098), (4, 277420), (5, 10005), (8, 65536 * 8), (16, 160016),
                                 (64, 64 * 1031)])
def test_reduce_scatter_matches_oracle(p, n, own, algo, dtype):
    if own == "ring":
        n += 3 if p > 1 else 0  # padding and trim
    devs, hosts, _ = make_replicas(p, n, dtype, "uniform", seed=200 + p)
    cs = orc.chunk_size(n, p)
    tdt = torch.float32 if dtype == "f32" else torch.bfloat16
    outs = [torch.full((cs + 4,), -7.0, dtype=tdt, device="cuda") for _ in range(p)]
    code = D.DDP_OWN_RANK if own == "rank" else D.DDP_OWN_RING
    D.ddp_reduce_scatter(devs, outs, n, DT[dtype], float(p), code, algo)
    want, info = orc.reduce_scatter(hosts, n, float(p), dtype, own)
    for r in range(p):
        got = to_host(outs[r])
        L = len(want[r])
        assert_bit_equal(got[:L], want[r], f"rank {r}")
        # nothing written past the rank's real elements
        assert np.all(got[L:].astype(np.float32) == -7.0) if dtype == "f32" else True
    # inputs untouched
    for r in range(p):
        assert_bit_equal(to_host(devs[r]), hosts[r])
    _no_device_error()


def test_reduce_scatter_not_divisible_is_an_error():
    devs, _, _ = make_replicas(4, 10, "f32")
    outs = [torch.empty(3, device="cuda") for _ in range(4)]
    with pytest.raises(D.DDPError) as e:
        D.ddp_reduce_scatter(devs, outs, 10, D.DDP_FLOAT32, 1.0, D.DDP_OWN_RANK)
    assert e.value.status == D.DDP_ERR_NOT_DIVISIBLE


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("algo", ALGOS)
@pytest.mark.parametrize("own", ["rank", "ring"])
@pytest.mark.parametrize("p,m", [(1, 100), (2, 4097), (4, 1), (8, 12345), (16, 4096), (64, 1001)])
def test_allgather_matches_oracle(p, m, own, algo, dtype):
    devs, hosts, _ = make_replicas(p, m, dtype, "uniform", seed=300 + p)
    tdt = torch.float32 if dtype == "f32" else torch.bfloat16
    outs = [torch.zeros(p * m, dtype=tdt, device="cuda") for _ in range(p)]
    D.ddp_allgather(devs, outs, m, DT[dtype], D.DDP_OWN_RANK if own == "rank" else D.DDP_OWN_RING, algo)
    want, _ = orc.allgather(hosts, dtype, own)
    for r in range(p):
        assert_bit_equal(to_host(outs[r]), want[r], f"rank {r}")


@pytest.mark.parametrize("algo", ALGOS)
@pytest.mark.parametrize("p,nbytes,root", [(1, 100, 0), (2, 1, 1), (3, 4097, 2), (8, 1 << 20, 0),
                                           (8, 1000003, 5), (16, 333, 9), (64, 65541, 63)])
def test_broadcast_matches_oracle(p, nbytes, root, algo):
    gen = torch.Generator().manual_seed(p * 31 + root)
    host = [torch.randint(0, 256, (nbytes + 3,), dtype=torch.uint8, generator=gen) for _ in range(p)]
    devs = [h.cuda() for h in host]
    views = [d[r % 3: r % 3 + nbytes] for r, d in enumerate(devs)]  # mixed byte alignment
    D.ddp_broadcast(views, nbytes, root, algo)
    want, steps, _ = orc.broadcast_tree([h[r % 3: r % 3 + nbytes].numpy() for r, h in enumerate(host)], root)
    for r in range(p):
        assert np.array_equal(views[r].cpu().numpy(), want[r])
        # bytes outside the view untouched
        full = devs[r].cpu().numpy()
        assert np.array_equal(full[: r % 3], host[r][: r % 3].numpy())


@pytest.mark.parametrize("algo", ALGOS)
@pytest.mark.parametrize("cap", [0, 1000, 40000])
def test_broadcast_coalesced_llama_buffers(algo, cap):
    """64 fp32 buffer tensors of 256..4096 elements from replica 0 to 7 others."""
    from synth import shapes
    p = 8
    sizes = shapes.llama_buffers()
    tensors = [[torch.full((s,), float(r * 1000 + j), device="cuda") for j, s in enumerate(sizes)]
               for r in range(p)]
    host = [[t.cpu().numpy().view(np.uint8) for t in row] for row in tensors]
    D.ddp_broadcast_coalesced(tensors, [4 * s for s in sizes], 0, cap, algo)
    want, groups = orc.broadcast_coalesced(host, 0, cap if cap else 250 * 1024 * 1024)
    for r in range(p):
        for j in range(len(sizes)):
            assert np.array_equal(tensors[r][j].cpu().numpy().view(np.uint8), want[r][j])
    _no_device_error()


@pytest.mark.parametrize("algo", ALGOS)
def test_broadcast_coalesced_mixed_dtypes_and_roots(algo):
    """ResNet-50's BatchNorm buffers (fp32 running stats, int64 counters), root 3."""
    from synth import shapes
    p, root = 5, 3
    bufs = shapes.resnet50_buffers()
    tensors = []
    for r in range(p):
        row = []
        for j, (_, shp, dt) in enumerate(bufs):
            if dt == "f32":
                row.append(torch.full(shp, float(r + j), device="cuda"))
            else:
                row.append(torch.full(shp, r * 100 + j, dtype=torch.int64, device="cuda"))
        tensors.append(row)
    nbytes = [t.numel() * t.element_size() for t in tensors[0]]
    host = [[t.cpu().reshape(-1).numpy().view(np.uint8).copy() for t in row] for row in tensors]
    D.ddp_broadcast_coalesced(tensors, nbytes, root, 4096, algo)
    want, _ = orc.broadcast_coalesced(host, root, 4096)
    for r in range(p):
        for j in range(len(bufs)):
            assert np.array_equal(tensors[r][j].cpu().reshape(-1).numpy().view(np.uint8), want[r][j])


@pytest.mark.parametrize("k,launches", [(159, 1), (600, 3)])
def test_fused_coalesced_broadcast_launch_split(k, launches):
    """The fused coalesced broadcast packs up to 256 tensors (at p = 8) into
    one launch: the ResNet-50 buffer count fits one; 600 tensors of odd byte
    sizes split across three, with every byte still the root's."""
    p, root = 8, 2
    rng = np.random.default_rng(k)
    sizes = [int(x) for x in rng.integers(1, 3000, size=k)]
    tensors = [[torch.full((s,), r * 7 + j % 5, dtype=torch.uint8, device="cuda") for j, s in enumerate(sizes)]
               for r in range(p)]
    host = [[t.cpu().numpy().copy() for t in row] for row in tensors]
    before = D.ddp_kernel_launches()
    D.ddp_broadcast_coalesced(tensors, sizes, root, 0, D.DDP_ALGO_FUSED)
    assert D.ddp_kernel_launches() - before == launches
    want, _ = orc.broadcast_coalesced(host, root, 250 * 1024 * 1024)
    for r in range(p):
        for j in range(k):
            assert np.array_equal(tensors[r][j].cpu().numpy(), want[r][j]), (r, j)
    _no_device_error()


def test_zero_sizes_accept_empty_tensors():
    """Empty tensors have no storage (a null data pointer): a zero-size call
    is a no-op whatever its pointers, for every entry point."""
    p = 4
    empty = [torch.empty(0, dtype=torch.float32, device="cuda") for _ in range(p)]
    for algo in ALGOS + [D.DDP_ALGO_RECURSIVE_DOUBLING, D.DDP_ALGO_RABENSEIFNER, D.DDP_ALGO_TREE]:
        D.ddp_allreduce(empty, 0, D.DDP_FLOAT32, 4.0, algo)
    for algo in (D.DDP_ALGO_FUSED, D.DDP_ALGO_RING_STEPS):
        for own in (D.DDP_OWN_RANK, D.DDP_OWN_RING):
            D.ddp_reduce_scatter(empty, empty, 0, D.DDP_FLOAT32, 1.0, own, algo)
        D.ddp_allgather(empty, empty, 0, D.DDP_FLOAT32, D.DDP_OWN_RANK, algo)
        D.ddp_broadcast(empty, 0, 1, algo)
    status = torch.full((4,), -1, dtype=torch.int32, device="cuda")
    D.ddp_allreduce_persistent(empty, 0, D.DDP_FLOAT32, 4.0, 0, -1, 0, status)
    torch.cuda.synchronize()
    assert status.cpu().tolist() == [0, 0, 0, 0]
    # the scalar arguments are still checked
    with pytest.raises(D.DDPError) as e:
        D.ddp_allreduce(empty, 0, D.DDP_FLOAT32, 0.0)
    assert e.value.status == D.DDP_ERR_ARG
    _no_device_error()


def test_zero_sizes_are_noops():
    devs, hosts, _ = make_replicas(4, 16, "f32")
    D.ddp_allreduce(devs, 0, D.DDP_FLOAT32, 4.0)
    D.ddp_broadcast(devs, 0, 0)
    D.ddp_broadcast_coalesced([[d] for d in devs], [0], 0)
    for r in range(4):
        assert_bit_equal(to_host(devs[r]), hosts[r])
    _no_device_error()


def test_kernel_launch_counter_counts():
    before = D.ddp_kernel_launches()
    devs, _, _ = make_replicas(8, 1000, "f32")
    D.ddp_allreduce(devs, 1000, D.DDP_FLOAT32, 8.0, D.DDP_ALGO_FUSED)
    D.ddp_allreduce(devs, 1000, D.DDP_FLOAT32, 8.0, D.DDP_ALGO_RING_STEPS)
    assert D.ddp_kernel_launches() - before == 1 + 2 * 7


@pytest.mark.parametrize("algo", [D.DDP_ALGO_FUSED, D.DDP_ALGO_FUSED_TMA])
def test_large_fanouts_by_bulk_copies(algo):
    """Fan-outs large enough that DDP_ALGO_FUSED takes the bulk-copy form
    (7 or more destinations, 64 MiB or more read): a broadcast of 64 MiB plus
    a ragged 1,007 bytes whose replicas all start 4 bytes past a 16-byte
    boundary (12 bytes before the first boundary go singly, as does the
    tail), and an all-gather of 8 replicas' 2,097,156-element fp32 chunks.
    Against the oracle's copies, byte for byte."""
    p, root = 8, 5
    nbytes = (64 << 20) + 1007
    gen = torch.Generator().manual_seed(77)
    host = [torch.randint(0, 256, (nbytes + 4,), dtype=torch.uint8, generator=gen) for _ in range(p)]
    devs = [h.cuda() for h in host]
    views = [d[4:4 + nbytes] for d in devs]
    D.ddp_broadcast(views, nbytes, root, algo)
    want, _, _ = orc.broadcast_tree([h[4:4 + nbytes].numpy() for h in host], root)
    for r in range(p):
        assert np.array_equal(views[r].cpu().numpy(), want[r]), r
        assert np.array_equal(devs[r][:4].cpu().numpy(), host[r][:4].numpy())
    m = 2097156
    ins, hosts, _ = make_replicas(p, m, "f32", "uniform", seed=401)
    outs = [torch.zeros(p * m, dtype=torch.float32, device="cuda") for _ in range(p)]
    D.ddp_allgather(ins, outs, m, D.DDP_FLOAT32, D.DDP_OWN_RANK, algo)
    want, _ = orc.allgather(hosts, "f32", "rank")
    for r in range(p):
        assert_bit_equal(to_host(outs[r]), want[r], f"rank {r}")
    assert D.ddp_device_error() == 0


@pytest.mark.parametrize("p", [33, 64, 256])
def test_bulk_fanout_with_more_destinations_than_lanes(p):
    """The bulk-copy fan-out's warp issues one store per destination, lane q
    taking destinations q, q + 32, ...: broadcasts and all-gathers to 32 or
    more replicas, aligned so that the bulk form runs, with a ragged tail."""
    nbytes = 3 * 8192 + 48 + 5
    gen = torch.Generator().manual_seed(p)
    host = [torch.randint(0, 256, (nbytes,), dtype=torch.uint8, generator=gen) for _ in range(p)]
    devs = [h.cuda() for h in host]
    D.ddp_broadcast(devs, nbytes, p - 1, D.DDP_ALGO_FUSED_TMA)
    want, _, _ = orc.broadcast_tree([h.numpy() for h in host], p - 1)
    for r in range(p):
        assert np.array_equal(devs[r].cpu().numpy(), want[r]), r
    m = 2052  # 8,208 bytes per chunk: every job offset stays 16-byte aligned
    ins, hosts, _ = make_replicas(p, m, "f32", "uniform", seed=500 + p)
    outs = [torch.zeros(p * m, dtype=torch.float32, device="cuda") for _ in range(p)]
    D.ddp_allgather(ins, outs, m, D.DDP_FLOAT32, D.DDP_OWN_RING, D.DDP_ALGO_FUSED_TMA)
    want, _ = orc.allgather(hosts, "f32", "ring")
    for r in range(p):
        assert_bit_equal(to_host(outs[r]), want[r], f"rank {r}")
    assert D.ddp_device_error() == 0
