"""The reduce-scatter that allocates nothing, checked against the ordinary one.

Some callers cannot allocate device memory while a call runs. One example is a
framework whose caching allocator already holds the whole device; another is a
training step that must not risk an allocation failing, or synchronising,
halfway through. For those callers ddp_reduce_scatter_noalloc keeps the ring's
fp32 partials in a fixed 8 MiB array inside the library instead of a temporary.

Its results must equal ddp_reduce_scatter's, which runs the same literal ring,
bit for bit: the tolerance every parity test here uses for fp32 and bf16. The
check runs on two calls in a row, because the second call finds the first
call's leftovers in the shared array. Calls past the array's size must be
refused with a clear error.
"""
import pytest

import ring_all_reduce_ddp_gb300 as D
from tests.helpers import assert_bit_equal, make_replicas, to_host

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

DT = {"f32": D.DDP_FLOAT32, "bf16": D.DDP_BFLOAT16}
LIMIT_ELEMS = 1 << 20  # p * ceil(n/p) that fills the 8 MiB array exactly


@pytest.fixture(scope="module", autouse=True)
def _library():
    from ring_all_reduce_ddp_gb300 import build
    build.build_library()


def _outs(p, n, dtype):
    cs = -(-n // p)
    tdt = torch.float32 if dtype == "f32" else torch.bfloat16
    return [torch.full((cs,), -3.0, dtype=tdt, device="cuda") for _ in range(p)]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("own", ["rank", "ring"])
@pytest.mark.parametrize("p,n", [(1, 1000), (2, 4098), (4, 277420), (8, LIMIT_ELEMS), (64, 64 * 1031)])
def test_noalloc_equals_reduce_scatter_on_two_calls(p, n, own, dtype):
    if own == "ring" and p > 1:
        n -= 5  # padding and trim; still within the limit
    code = D.DDP_OWN_RANK if own == "rank" else D.DDP_OWN_RING
    for call in range(2):
        ins, _, _ = make_replicas(p, n, dtype, "normal", seed=9000 + 10 * p + call)
        want = _outs(p, n, dtype)
        got = _outs(p, n, dtype)
        D.ddp_reduce_scatter(ins, want, n, DT[dtype], float(p), code, D.DDP_ALGO_RING_STEPS)
        D.ddp_reduce_scatter_noalloc(ins, got, n, DT[dtype], float(p), code)
        torch.cuda.synchronize()
        for r in range(p):
            assert_bit_equal(to_host(got[r]), to_host(want[r]), f"call {call} rank {r}")
    assert D.ddp_device_error() == 0


def test_noalloc_refuses_sizes_past_its_array():
    p = 8
    n = LIMIT_ELEMS + p  # one more element per chunk than the array holds
    ins, _, _ = make_replicas(p, n, "f32", "uniform", seed=9100)
    outs = _outs(p, n, "f32")
    with pytest.raises(D.DDPError) as e:
        D.ddp_reduce_scatter_noalloc(ins, outs, n, D.DDP_FLOAT32, 1.0, D.DDP_OWN_RANK)
    assert e.value.status == D.DDP_ERR_ARG
    assert "scratch" in str(e.value) and "8388608" in str(e.value)
    # nothing was enqueued: the outputs are untouched
    assert all(bool(torch.all(o == -3.0)) for o in outs)
