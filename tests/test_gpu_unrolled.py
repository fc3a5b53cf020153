"""GPU parity of the fused register kernel's unrolled form: at p = 2 and 4 each
thread takes four or two vectors once a chunk is large enough that the grid
still holds 4 blocks per SM (152 SMs: 608 blocks). The sizes here sit past that
point, with ragged tails, so the unrolled loop and its bounds run; one size per
p sits just below it. Everything is bit-exact against the oracle."""
import numpy as np
import pytest

import ring_all_reduce_ddp_gb300 as D
from oracle import ring as orc
from tests.helpers import assert_bit_equal, make_replicas, to_host

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

DT = {"f32": D.DDP_FLOAT32, "bf16": D.DDP_BFLOAT16}
VEC = {"f32": 4, "bf16": 8}  # elements per 16-byte vector
UNROLL = {2: 4, 4: 2}


def unrolled(p, n, dtype, sms=152):
    """Whether the launch rule picks the unrolled form for this call."""
    cs = -(-n // p)
    vectors = cs // VEC[dtype] + 1
    per_block = 256 * UNROLL[p]
    return -(-vectors // per_block) * p >= 4 * sms


# (p, n, dtype): past the threshold with ragged tails, and one just below it
CASES = [(2, 3_000_017, "f32"), (2, 5_000_011, "bf16"), (4, 1_300_003, "f32"), (4, 2_600_009, "bf16"),
         (2, 2_400_001, "f32"), (4, 1_200_001, "f32")]


def test_cases_straddle_the_threshold():
    assert [unrolled(p, n, dt) for p, n, dt in CASES] == [True, True, True, True, False, False]


@pytest.mark.parametrize("p,n,dtype", CASES)
@pytest.mark.parametrize("algo", [D.DDP_ALGO_FUSED, D.DDP_ALGO_FUSED_LDST])
def test_allreduce(p, n, dtype, algo):
    devs, hosts, _ = make_replicas(p, n, dtype, "normal", seed=900 + p)
    D.ddp_allreduce(devs, n, DT[dtype], float(p), algo)
    want, _ = orc.allreduce(hosts, n, float(p), dtype)
    for r in range(p):
        assert_bit_equal(to_host(devs[r]), want[r], f"replica {r}")
    assert D.ddp_device_error() == 0


@pytest.mark.parametrize("p,n", [(p, n) for p, n, dt in CASES[:4] if dt == "bf16"])
def test_allreduce_per_hop_bf16(p, n):
    devs, hosts, _ = make_replicas(p, n, "bf16", "normal", seed=910 + p)
    D.ddp_allreduce_ex(devs, n, D.DDP_BFLOAT16, float(p), D.DDP_ALGO_FUSED, D.DDP_FLAG_ROUND_EACH_HOP)
    want, _ = orc.allreduce(hosts, n, float(p), "bf16", hop_round=True)
    for r in range(p):
        assert_bit_equal(to_host(devs[r]), want[r], f"replica {r}")


@pytest.mark.parametrize("offsets", [[1, 1, 1, 1], [0, 1, 2, 3]])
@pytest.mark.parametrize("p", [2, 4])
def test_allreduce_misaligned(p, offsets):
    n = 3_000_017 if p == 2 else 1_300_003
    devs, hosts, _ = make_replicas(p, n, "f32", "uniform", seed=920 + p, offsets=offsets[:p])
    D.ddp_allreduce(devs, n, D.DDP_FLOAT32, float(p))
    want, _ = orc.allreduce(hosts, n, float(p), "f32")
    for r in range(p):
        assert_bit_equal(to_host(devs[r]), want[r], f"replica {r}")


@pytest.mark.parametrize("own", ["rank", "ring"])
@pytest.mark.parametrize("p,n,dtype", [(2, 3_000_018, "f32"), (4, 1_300_004, "f32"), (4, 2_600_012, "bf16")])
def test_reduce_scatter(p, n, dtype, own):
    if own == "ring":
        n += 3  # padding and trim
    assert unrolled(p, n, dtype)
    devs, hosts, _ = make_replicas(p, n, dtype, "uniform", seed=930 + p)
    cs = orc.chunk_size(n, p)
    tdt = torch.float32 if dtype == "f32" else torch.bfloat16
    outs = [torch.full((cs + 4,), -7.0, dtype=tdt, device="cuda") for _ in range(p)]
    code = D.DDP_OWN_RANK if own == "rank" else D.DDP_OWN_RING
    D.ddp_reduce_scatter(devs, outs, n, DT[dtype], float(p), code, D.DDP_ALGO_FUSED)
    want, _ = orc.reduce_scatter(hosts, n, float(p), dtype, own)
    for r in range(p):
        got = to_host(outs[r])
        L = len(want[r])
        assert_bit_equal(got[:L], want[r], f"rank {r}")
        if dtype == "f32":
            assert np.all(got[L:] == -7.0), f"rank {r} written past its elements"
    for r in range(p):
        assert_bit_equal(to_host(devs[r]), hosts[r])
