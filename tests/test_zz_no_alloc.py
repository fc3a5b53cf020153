"""The reduce-scatter that allocates nothing, checked against the ordinary one.

Some callers cannot allocate device memory while a call runs. One example is a
framework whose caching allocator already holds the whole device; another is a
training step that must not risk an allocation failing, or synchronising,
halfway through. For those callers ddp_reduce_scatter_noalloc keeps the ring's
fp32 partials in a fixed 8 MiB array inside the library instead of a temporary.

Its results must equal ddp_reduce_scatter's, which runs the same literal ring,
and the oracle's reduce-scatter, bit for bit: the tolerance every parity test
here uses for fp32 and bf16. The check runs on two calls in a row, because the
second call finds the first call's leftovers in the shared array. Calls past
the array's size must be refused with a clear error, and a call must take no
memory from the device's stream-ordered pool (which the ordinary call's
temporary comes from) and leave the device's free memory as it was.
"""
import ctypes
import glob
import os

import numpy as np
import pytest

import ring_all_reduce_ddp_gb300 as D
from oracle import ring as orc
from tests.helpers import assert_bit_equal, make_replicas, to_host

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

DT = {"f32": D.DDP_FLOAT32, "bf16": D.DDP_BFLOAT16}
LIMIT_ELEMS = 1 << 20  # p * ceil(n/p) that fills the 8 MiB array exactly


@pytest.fixture(scope="module", autouse=True)
def _library():
    from ring_all_reduce_ddp_gb300 import build
    build.build_library()


def _cudart():
    """The CUDA runtime as a shared library (torch has one loaded already)."""
    cands = ["libcudart.so.13", "libcudart.so"]
    tdir = os.path.dirname(torch.__file__)
    cands += sorted(glob.glob(os.path.join(tdir, "lib", "libcudart.so*")))
    cands += sorted(glob.glob(os.path.join(tdir, "..", "nvidia", "*", "lib", "libcudart.so*")))
    cands += sorted(glob.glob("/usr/local/cuda/lib64/libcudart.so*"))
    for c in cands:
        try:
            return ctypes.CDLL(c)
        except OSError:
            continue
    pytest.fail("no CUDA runtime library to read the memory pool with")


POOL_USED_HIGH = 8  # cudaMemPoolAttrUsedMemHigh


class _Pool:
    """High-water mark of the memory in use from the current device's
    stream-ordered pool (where cudaMallocAsync takes its memory)."""

    def __init__(self):
        self.rt = _cudart()
        self.pool = ctypes.c_void_p()
        assert self.rt.cudaDeviceGetMemPool(ctypes.byref(self.pool), torch.cuda.current_device()) == 0

    def reset(self):
        zero = ctypes.c_uint64(0)
        assert self.rt.cudaMemPoolSetAttribute(self.pool, POOL_USED_HIGH, ctypes.byref(zero)) == 0

    def used_high(self):
        v = ctypes.c_uint64()
        assert self.rt.cudaMemPoolGetAttribute(self.pool, POOL_USED_HIGH, ctypes.byref(v)) == 0
        return v.value


_MINUS3 = {"f32": np.float32(-3.0), "bf16": np.uint16(0xC040)}  # what _outs fills with


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
        ins, hosts, _ = make_replicas(p, n, dtype, "normal", seed=9000 + 10 * p + call)
        want = _outs(p, n, dtype)
        got = _outs(p, n, dtype)
        D.ddp_reduce_scatter(ins, want, n, DT[dtype], float(p), code, D.DDP_ALGO_RING_STEPS)
        D.ddp_reduce_scatter_noalloc(ins, got, n, DT[dtype], float(p), code)
        torch.cuda.synchronize()
        oracle, _ = orc.reduce_scatter(hosts, n, float(p), dtype, own)
        for r in range(p):
            g = to_host(got[r])
            assert_bit_equal(g, to_host(want[r]), f"call {call} rank {r} against ddp_reduce_scatter")
            m = len(oracle[r])
            assert_bit_equal(g[:m], oracle[r], f"call {call} rank {r} against the oracle")
            assert np.all(g[m:] == _MINUS3[dtype]), f"call {call} rank {r}: trimmed padding was written"
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


def test_noalloc_takes_no_device_memory():
    """At the largest size it accepts, the call takes nothing from the stream-
    ordered pool and leaves the device's free memory unchanged, while the
    ordinary literal reduce-scatter of the same size takes its 8 MiB temporary
    from that pool (which shows the probe sees an allocation)."""
    p, n = 8, LIMIT_ELEMS
    ins, hosts, _ = make_replicas(p, n, "f32", "uniform", seed=9200)
    outs = _outs(p, n, "f32")
    pool = _Pool()
    D.ddp_reduce_scatter_noalloc(ins, outs, n, D.DDP_FLOAT32, 1.0, D.DDP_OWN_RANK)  # first call: set-up
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    pool.reset()
    for _ in range(2):
        D.ddp_reduce_scatter_noalloc(ins, outs, n, D.DDP_FLOAT32, 1.0, D.DDP_OWN_RANK)
    torch.cuda.synchronize()
    assert pool.used_high() == 0
    assert torch.cuda.mem_get_info()[0] == free0
    want, _ = orc.reduce_scatter(hosts, n, 1.0, "f32", "rank")
    for r in range(p):
        assert_bit_equal(to_host(outs[r]), want[r], f"rank {r}")
    pool.reset()
    D.ddp_reduce_scatter(ins, outs, n, D.DDP_FLOAT32, 1.0, D.DDP_OWN_RANK, D.DDP_ALGO_RING_STEPS)
    torch.cuda.synchronize()
    assert pool.used_high() >= 2 * p * (n // p) * 4


def test_noalloc_empty_call_ignores_pointers():
    """n == 0 is a no-op that returns OK whatever the pointers, as for
    ddp_reduce_scatter."""
    for fn in (lambda: D.ddp_reduce_scatter_noalloc([0] * 4, [0] * 4, 0, D.DDP_FLOAT32, 4.0, D.DDP_OWN_RANK),
               lambda: D.ddp_reduce_scatter([0] * 4, [0] * 4, 0, D.DDP_FLOAT32, 4.0, D.DDP_OWN_RANK,
                                            D.DDP_ALGO_RING_STEPS)):
        fn()
    torch.cuda.synchronize()
