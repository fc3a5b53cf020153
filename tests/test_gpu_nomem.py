"""Allocation failures on the device. Every call that takes device memory for
a temporary or a handle returns DDP_ERR_NOMEM before any of its kernels is
enqueued, leaves no CUDA error pending, and leaks nothing. The device is
filled with one blocker tensor until less memory is left than the call needs;
no kernel runs while it is held. After the blocker is released the same call
succeeds."""
import contextlib

import numpy as np
import pytest

import ring_all_reduce_ddp_gb300 as D
from oracle import ring as orc
from tests.helpers import assert_bit_equal, make_replicas, to_host

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

MiB = 1 << 20
LEAVE = 64 * MiB


@contextlib.contextmanager
def squeezed(need):
    """Hold all but about LEAVE bytes of free device memory; yields what is left,
    which the caller's temporary of `need` bytes does not fit in."""
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    free, _ = torch.cuda.mem_get_info()
    size = free - LEAVE
    blocker = None
    while blocker is None and size > 0:
        try:
            blocker = torch.empty(size, dtype=torch.uint8, device="cuda")
        except torch.cuda.OutOfMemoryError:
            size -= 256 * MiB
    try:
        left = torch.cuda.mem_get_info()[0]
        assert left < need, f"could not squeeze: {left} bytes left, the call needs {need}"
        yield left
    finally:
        del blocker
        torch.cuda.synchronize()
        torch.cuda.empty_cache()


def expect_nomem(fn, what):
    with pytest.raises(D.DDPError) as ei:
        fn()
    assert ei.value.status == D.DDP_ERR_NOMEM, str(ei.value)
    assert what in str(ei.value), str(ei.value)


def context_is_clean():
    """No CUDA error pending, and a small all-reduce gives the oracle's bits."""
    torch.cuda.synchronize()
    devs, hosts, _ = make_replicas(3, 1000, "f32", "normal", seed=91)
    D.ddp_allreduce(devs, 1000, D.DDP_FLOAT32, 3.0)
    want, _ = orc.allreduce(hosts, 1000, 3.0, "f32")
    for r in range(3):
        assert_bit_equal(to_host(devs[r]), want[r], f"replica {r}")
    assert D.ddp_device_error() == 0


def unchanged(devs, hosts):
    for r, (d, h) in enumerate(zip(devs, hosts)):
        assert_bit_equal(to_host(d), h, f"replica {r} was written by a call that failed")


@pytest.mark.parametrize("algo,what", [(D.DDP_ALGO_TREE, "tree workspace"),
                                       (D.DDP_ALGO_RING_STEPS, "workspace allocation")])
def test_bf16_allreduce_workspace(algo, what):
    p, n = 2, 1 << 27  # 256 MiB of bf16 per replica; fp32 workspace 1 GiB
    devs, hosts, _ = make_replicas(p, n, "bf16", "normal", seed=92)
    with squeezed(4 * n * p):
        expect_nomem(lambda: D.ddp_allreduce(devs, n, D.DDP_BFLOAT16, 2.0, algo), what)
        torch.cuda.synchronize()
    unchanged(devs, hosts)
    D.ddp_allreduce(devs, n, D.DDP_BFLOAT16, 2.0, algo)
    torch.cuda.synchronize()
    context_is_clean()


def test_bf16_persistent_workspace():
    p, n = 2, 1 << 27
    devs, hosts, _ = make_replicas(p, n, "bf16", "normal", seed=93)
    with squeezed(4 * n * p):
        expect_nomem(lambda: D.ddp_allreduce_persistent(devs, n, D.DDP_BFLOAT16, 2.0), "persistent ring workspace")
        torch.cuda.synchronize()
    unchanged(devs, hosts)
    D.ddp_allreduce_persistent(devs, n, D.DDP_BFLOAT16, 2.0)
    torch.cuda.synchronize()
    context_is_clean()


def test_literal_reduce_scatter_workspace():
    p, n = 2, 1 << 27  # 512 MiB of fp32 per replica; partials 2 p ceil(n/p) floats = 1 GiB
    ins, hosts, _ = make_replicas(p, n, "f32", "normal", seed=94)
    outs = [torch.zeros(n // p, dtype=torch.float32, device="cuda") for _ in range(p)]
    with squeezed(8 * n):
        expect_nomem(lambda: D.ddp_reduce_scatter(ins, outs, n, D.DDP_FLOAT32, 2.0, D.DDP_OWN_RING,
                                                  D.DDP_ALGO_RING_STEPS), "workspace allocation")
        torch.cuda.synchronize()
    unchanged(ins, hosts)
    assert all(int(torch.count_nonzero(o)) == 0 for o in outs)
    context_is_clean()


def test_ring_handle_workspace():
    p, n = 2, 1 << 27
    ins, hosts, _ = make_replicas(p, n, "f32", "normal", seed=95)
    outs = [torch.zeros(n // p, dtype=torch.float32, device="cuda") for _ in range(p)]
    with squeezed(8 * n) as left:
        expect_nomem(lambda: D.DDPRing(D.DDP_OP_REDUCE_SCATTER, ins, outs, n, D.DDP_FLOAT32, 2.0),
                     "handle workspace allocation")
        assert torch.cuda.mem_get_info()[0] >= left - 2 * MiB  # nothing kept by the failed create
    with D.DDPRing(D.DDP_OP_REDUCE_SCATTER, ins, outs, n, D.DDP_FLOAT32, 2.0) as ring:
        for _ in range(ring.num_steps()):
            ring.step()
        ring.sync()
    context_is_clean()


def test_literal_coalesced_broadcast_workspace():
    p, k, each = 2, 2, 200 * MiB  # the default 250 MiB cap puts each tensor in its own group
    rows = [[torch.full((each // 4,), float(r + 1), device="cuda") for _ in range(k)] for r in range(p)]
    with squeezed(p * each):
        expect_nomem(lambda: D.ddp_broadcast_coalesced(rows, [each] * k, root=1, algo=D.DDP_ALGO_RING_STEPS),
                     "broadcast workspace allocation")
        torch.cuda.synchronize()
    assert all(bool(torch.all(t == 1.0)) for t in rows[0])
    D.ddp_broadcast_coalesced(rows, [each] * k, root=1, algo=D.DDP_ALGO_RING_STEPS)
    assert all(bool(torch.all(t == 2.0)) for t in rows[0])
    context_is_clean()


def test_reducer_create_buckets():
    p = 2
    grads = [[torch.full((1 << 26,), float(r + 1), device="cuda") for _ in range(2)] for r in range(p)]
    with squeezed(p * 2 * (1 << 28)) as left:
        expect_nomem(lambda: D.DDPReducer(grads, 1 << 20, 1 << 30), "reducer buckets")
        assert torch.cuda.mem_get_info()[0] >= left - 2 * MiB  # the arenas it did get are released
    red = D.DDPReducer(grads, 1 << 20, 1 << 30)
    red.sync(2.0, mode=D.DDP_SYNC_FLATTEN)
    torch.cuda.synchronize()
    assert all(bool(torch.all(g == 1.5)) for row in grads for g in row)
    red.destroy()
    context_is_clean()


def test_reducer_rebuild_that_fails_leaves_a_bucketless_handle():
    """A rebuild along a walk whose largest bucket is bigger needs a bigger
    bf16 workspace than the one it released. Registration order C, B, A of
    64, 64, 128 MiB with a first cap just above 128 MiB: the reversed walk
    A, B, C buckets {A, B} and {C} (largest 192 MiB, workspace 768 MiB); the
    walk C, B, A buckets {C, B, A} (256 MiB, workspace 1 GiB)."""
    p = 2
    sizes = [1 << 25, 1 << 25, 1 << 26]  # bf16 elements of C, B, A
    grads = [[torch.full((m,), float(r + 1), dtype=torch.bfloat16, device="cuda") for m in sizes] for r in range(p)]
    red = D.DDPReducer(grads, (1 << 27) + 2, 1)
    assert red.num_buckets() == 2
    with squeezed(1 << 30):
        with pytest.raises(D.DDPError) as ei:
            red.rebuild([0, 1, 2])
        assert ei.value.status == D.DDP_ERR_NOMEM, str(ei.value)
        assert "reducer workspace" in str(ei.value) and "no buckets" in str(ei.value)
    assert red.num_buckets() == 0
    for call in (lambda: red.sync(2.0), lambda: red.sync(2.0, mode=D.DDP_SYNC_FLATTEN), red.prepare,
                 lambda: red.mark_ready(0, 2.0)):
        with pytest.raises(D.DDPError) as ei:
            call()
        assert ei.value.status == D.DDP_ERR_STATE, str(ei.value)
    assert all(bool(torch.all(g == float(r + 1))) for r, row in enumerate(grads) for g in row)
    red.rebuild([0, 1, 2])
    assert red.num_buckets() == 1
    red.sync(2.0)
    torch.cuda.synchronize()
    assert all(bool(torch.all(g == 1.5)) for row in grads for g in row)
    red.destroy()
    context_is_clean()
