"""GPU parity of the variants beyond the default path: the per-hop bf16 ring
(partials rounded to bf16 at every hop, as a bf16 wire format carries them),
in its literal and fused forms, against the oracle's per-hop simulation."""
import numpy as np
import pytest

import ring_all_reduce_ddp_gb300 as D
from oracle import ring as orc
from oracle.bf16 import bf16_to_f32, f32_to_bf16
from tests.helpers import assert_bit_equal, make_replicas, to_host

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

ALGOS = [D.DDP_ALGO_FUSED, D.DDP_ALGO_FUSED_LDST, D.DDP_ALGO_FUSED_TMA, D.DDP_ALGO_RING_STEPS]


@pytest.mark.parametrize("algo", ALGOS)
@pytest.mark.parametrize("p,n", [(1, 100), (2, 4099), (3, 10007), (8, 65536 * 3 + 5), (16, 100003), (17, 5001),
                                 (64, 262147)])
def test_per_hop_bf16_matches_oracle(p, n, algo):
    devs, hosts, _ = make_replicas(p, n, "bf16", "normal", seed=700 + p)
    D.ddp_allreduce_ex(devs, n, D.DDP_BFLOAT16, float(p), algo, D.DDP_FLAG_ROUND_EACH_HOP)
    want, _ = orc.allreduce(hosts, n, float(p), "bf16", hop_round=True)
    for r in range(p):
        assert_bit_equal(to_host(devs[r]), want[r], f"replica {r}")
    assert D.ddp_device_error() == 0


@pytest.mark.parametrize("algo", ALGOS)
def test_per_hop_worked_example(algo):
    """256 on each chunk's origin rank, 1 elsewhere, p = 8: per hop 256, accumulated 264."""
    p, n = 8, 8 * 1000
    cs = n // p
    hop, acc = [], []
    for r in range(p):
        v = np.ones(n, dtype=np.float32)
        v[r * cs:(r + 1) * cs] = 256.0
        b = torch.from_numpy(f32_to_bf16(v).view(np.int16)).view(torch.bfloat16).cuda()
        hop.append(b)
        acc.append(b.clone())
    D.ddp_allreduce_ex(hop, n, D.DDP_BFLOAT16, 1.0, algo, D.DDP_FLAG_ROUND_EACH_HOP)
    D.ddp_allreduce(acc, n, D.DDP_BFLOAT16, 1.0, algo)
    assert np.all(bf16_to_f32(to_host(hop[0])) == 256.0)
    assert np.all(bf16_to_f32(to_host(acc[0])) == 264.0)


def test_per_hop_error_grows_with_p_on_the_gpu():
    """Mean |error| against the exact sum: rounding every hop versus once."""
    n = 1 << 18
    ratio = {}
    for p in (2, 8, 32):
        a, hosts, _ = make_replicas(p, n, "bf16", "normal", seed=800 + p)
        b = [t.clone() for t in a]
        D.ddp_allreduce_ex(a, n, D.DDP_BFLOAT16, 1.0, D.DDP_ALGO_FUSED, 0)
        D.ddp_allreduce_ex(b, n, D.DDP_BFLOAT16, 1.0, D.DDP_ALGO_FUSED, D.DDP_FLAG_ROUND_EACH_HOP)
        exact = np.sum(np.stack([bf16_to_f32(h) for h in hosts]).astype(np.float64), axis=0)
        e_once = np.mean(np.abs(bf16_to_f32(to_host(a[0])) - exact))
        e_hop = np.mean(np.abs(bf16_to_f32(to_host(b[0])) - exact))
        ratio[p] = e_hop / e_once
    assert ratio[2] >= 1.0 and ratio[8] > 1.5 and ratio[32] > ratio[8]


def test_per_hop_flag_needs_bf16():
    devs, _, _ = make_replicas(2, 100, "f32")
    with pytest.raises(D.DDPError) as e:
        D.ddp_allreduce_ex(devs, 100, D.DDP_FLOAT32, 1.0, D.DDP_ALGO_FUSED, D.DDP_FLAG_ROUND_EACH_HOP)
    assert e.value.status == D.DDP_ERR_DTYPE
    with pytest.raises(D.DDPError) as e:
        D.ddp_allreduce_ex(devs, 100, D.DDP_FLOAT32, 1.0, D.DDP_ALGO_FUSED, 8)
    assert e.value.status == D.DDP_ERR_ARG


# ---------------------------------------------------------- tree-shaped all-reduces
from oracle import trees as ot  # noqa: E402

TREE = {"rd": (D.DDP_ALGO_RECURSIVE_DOUBLING, ot.recursive_doubling),
        "rab": (D.DDP_ALGO_RABENSEIFNER, ot.rabenseifner),
        "tree": (D.DDP_ALGO_TREE, ot.tree)}


@pytest.mark.parametrize("name", ["rd", "rab"])
@pytest.mark.parametrize("p,n", [(1, 100), (2, 1), (2, 4099), (4, 3), (4, 277421), (8, 65536 * 3 + 5), (16, 100003),
                                 (64, 262147)])
def test_power_of_two_trees_match_oracle(name, p, n):
    algo, ref = TREE[name]
    devs, hosts, _ = make_replicas(p, n, "f32", "normal", seed=1100 + p)
    before = D.ddp_kernel_launches()
    D.ddp_allreduce(devs, n, D.DDP_FLOAT32, float(p), algo)
    launched = D.ddp_kernel_launches() - before
    want, info = ref(hosts, n, float(p))
    for r in range(p):
        assert_bit_equal(to_host(devs[r]), want[r], f"replica {r}")
    if p > 1:
        assert launched == info["steps"]  # log2 p, or 2 log2 p for Rabenseifner


@pytest.mark.parametrize("p,n", [(1, 10), (2, 4099), (3, 10007), (5, 3), (6, 65541), (8, 123457), (13, 50021),
                                 (16, 100003)])
def test_tree_matches_oracle(p, n):
    algo, ref = TREE["tree"]
    devs, hosts, _ = make_replicas(p, n, "f32", "uniform", seed=1200 + p)
    D.ddp_allreduce(devs, n, D.DDP_FLOAT32, float(p), algo)
    want, _ = ref(hosts, n, float(p))
    for r in range(p):
        assert_bit_equal(to_host(devs[r]), want[r], f"replica {r}")


def test_tree_algos_reject_what_they_cannot_do():
    devs, _, _ = make_replicas(6, 100, "f32")
    for algo in (D.DDP_ALGO_RECURSIVE_DOUBLING, D.DDP_ALGO_RABENSEIFNER):
        with pytest.raises(D.DDPError) as e:
            D.ddp_allreduce(devs, 100, D.DDP_FLOAT32, 1.0, algo)
        assert e.value.status == D.DDP_ERR_ARG
    devs, _, _ = make_replicas(6, 100, "bf16")
    for algo in (D.DDP_ALGO_RECURSIVE_DOUBLING, D.DDP_ALGO_RABENSEIFNER):
        with pytest.raises(D.DDPError) as e:
            D.ddp_allreduce(devs, 100, D.DDP_BFLOAT16, 1.0, algo)
        assert e.value.status == D.DDP_ERR_ARG


@pytest.mark.parametrize("name", ["rd", "rab", "tree"])
@pytest.mark.parametrize("p,n", [(1, 77), (2, 4099), (4, 3), (8, 65536 * 3 + 5), (16, 100003)])
def test_trees_in_bf16_round_once(name, p, n):
    """bf16 replicas: fp32 partials through the whole schedule, one rounding
    of each finished value; the bits equal the oracle's."""
    algo, ref = TREE[name]
    devs, hosts, _ = make_replicas(p, n, "bf16", "normal", seed=1300 + p)
    before = D.ddp_kernel_launches()
    D.ddp_allreduce(devs, n, D.DDP_BFLOAT16, float(p), algo)
    launched = D.ddp_kernel_launches() - before
    want, info = ref(hosts, n, float(p), "bf16")
    for r in range(p):
        assert_bit_equal(to_host(devs[r]), want[r], f"replica {r}")
    if p > 1:
        assert launched == info["steps"] + 2  # widen, the schedule's steps, narrow
    assert D.ddp_device_error() == 0


def test_tree_bf16_on_unaligned_replicas():
    """Replicas at odd element offsets take the element-by-element widen and
    narrow; the result is the same and nothing outside the replicas changes."""
    p, n = 4, 5003
    algo, ref = TREE["tree"]
    offs = [1, 3, 0, 5]
    devs, hosts, bases = make_replicas(p, n, "bf16", "uniform", seed=1400, offsets=offs)
    before = [to_host(b).copy() for b in bases]
    D.ddp_allreduce(devs, n, D.DDP_BFLOAT16, 3.0, algo)
    want, _ = ref(hosts, n, 3.0, "bf16")
    for r in range(p):
        assert_bit_equal(to_host(devs[r]), want[r], f"replica {r}")
        after = to_host(bases[r])
        assert np.array_equal(after[:offs[r]], before[r][:offs[r]])
        assert np.array_equal(after[offs[r] + n:], before[r][offs[r] + n:])
