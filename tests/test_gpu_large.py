"""Maximum sizes: one replica buffer of more than 2^31 elements (8.6 GB of fp32
or 4.3 GB of bf16 per replica), so every 32-bit index would overflow. The
fused, in-place and literal paths are checked on sampled elements (both sides of the chunk
boundary, the ends, and random indices) against the oracle's ring restricted to
those elements, from inputs regenerated on the host."""
import numpy as np
import pytest

import ring_all_reduce_ddp_gb300 as D
import synth
from oracle import ring as orc
from tests.helpers import assert_bit_equal, to_host

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

N = (1 << 31) + 1027
P = 2


@pytest.fixture(scope="module")
def big():
    free, _ = torch.cuda.mem_get_info()
    if free < 3 * P * N * 4:
        pytest.skip("not enough device memory for the > 2^31-element case")
    bufs = [torch.empty(N, dtype=torch.float32, device="cuda") for _ in range(P)]
    return bufs


def _fill(bufs):
    for r, b in enumerate(bufs):
        synth.fill_(b, "uniform", 4242, r)


def _sample():
    cs = orc.chunk_size(N, P)
    rng = np.random.default_rng(0)
    idx = set(range(8)) | set(range(N - 8, N)) | {cs - 2, cs - 1, cs, cs + 1, (1 << 31) - 1, 1 << 31, (1 << 31) + 1}
    idx |= set(int(x) for x in rng.integers(0, N, size=4000))
    return np.array(sorted(i for i in idx if 0 <= i < N), dtype=np.int64)


def _check(bufs, divisor):
    idx = _sample()
    ins = [synth.values_np("uniform", 4242, r, idx) for r in range(P)]
    want, _ = orc.allreduce(ins, N, divisor, idx=idx)
    t_idx = torch.from_numpy(idx).cuda()
    for r in range(P):
        assert_bit_equal(to_host(bufs[r][t_idx]), want[r], f"replica {r}")


@pytest.mark.parametrize("algo", [D.DDP_ALGO_FUSED, D.DDP_ALGO_RING_STEPS])
def test_allreduce_past_2_to_the_31_elements(big, algo):
    _fill(big)
    D.ddp_allreduce(big, N, D.DDP_FLOAT32, 2.0, algo)
    torch.cuda.synchronize()
    _check(big, 2.0)
    assert D.ddp_device_error() == 0


def test_in_place_bucket_past_2_to_the_31_elements(big):
    _fill(big)
    D.ddp_bucket_allreduce([[b] for b in big], [N], [0], D.DDP_FLOAT32, 2.0)
    torch.cuda.synchronize()
    _check(big, 2.0)


@pytest.fixture(scope="module")
def big_bf16():
    free, _ = torch.cuda.mem_get_info()
    if free < 3 * P * N * 2:
        pytest.skip("not enough device memory for the > 2^31-element bf16 case")
    return [torch.empty(N, dtype=torch.bfloat16, device="cuda") for _ in range(P)]


def _check_bf16(bufs, divisor):
    idx = _sample()
    ins = [synth.values_np("uniform", 4343, r, idx, 1.0, "bf16") for r in range(P)]
    want, _ = orc.allreduce(ins, N, divisor, "bf16", idx=idx)
    t_idx = torch.from_numpy(idx).cuda()
    for r in range(P):
        assert_bit_equal(to_host(bufs[r][t_idx]), want[r], f"replica {r}")


@pytest.mark.parametrize("path", ["fused", "in_place_bucket"])
def test_bf16_past_2_to_the_31_elements(big_bf16, path):
    """bf16 replicas of 2^31 + 1027 elements: the flat fused kernel and the
    in-place bucket kernel (64 KB tiles) on sampled elements."""
    for r, b in enumerate(big_bf16):
        synth.fill_(b, "uniform", 4343, r)
    if path == "fused":
        D.ddp_allreduce(big_bf16, N, D.DDP_BFLOAT16, 2.0, D.DDP_ALGO_FUSED)
    else:
        D.ddp_bucket_allreduce([[b] for b in big_bf16], [N], [0], D.DDP_BFLOAT16, 2.0)
    torch.cuda.synchronize()
    _check_bf16(big_bf16, 2.0)
    assert D.ddp_device_error() == 0
