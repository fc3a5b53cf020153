"""Calls from several host threads at once: handle-free calls and calls on
different handles run concurrently (ctypes releases the GIL for the length of
a foreign call); the error text is per thread."""
import threading

import numpy as np
import pytest

import ring_all_reduce_ddp_gb300 as D
from oracle import buckets as ob


def _run_threads(fns):
    errors = []

    def wrap(fn):
        try:
            fn()
        except BaseException as e:  # reported to the main thread below
            errors.append(e)

    ts = [threading.Thread(target=wrap, args=(f,)) for f in fns]
    for t in ts:
        t.start()
    for t in ts:
        t.join()
    if errors:
        raise errors[0]


def test_bucket_assignment_from_many_threads_matches_the_oracle():
    rng = np.random.default_rng(5)
    cases = []
    for _ in range(8):
        k = int(rng.integers(1, 300))
        numel = [int(x) for x in rng.integers(0, 100000, size=k)]
        cases.append((numel, ob.assign_buckets(numel, 4, 1 << 16, 1 << 20)))

    def worker(numel, want):
        def run():
            for _ in range(200):
                got = D.ddp_bucket_assign(numel, 4, 1 << 16, 1 << 20)["buckets"]
                assert got == want
        return run

    _run_threads([worker(n, w) for n, w in cases])


def test_error_text_is_per_thread():
    barrier = threading.Barrier(2)
    seen = {}

    def bad_divisor():
        barrier.wait()
        for _ in range(500):
            with pytest.raises(D.DDPError) as e:
                D.ddp_allreduce([0, 0], 0, D.DDP_FLOAT32, 0.0, stream=0)
            assert "divisor" in str(e.value)
        seen["a"] = str(e.value)

    def bad_p():
        barrier.wait()
        for _ in range(500):
            with pytest.raises(D.DDPError) as e:
                D.ddp_allreduce([0] * 300, 0, D.DDP_FLOAT32, 2.0, stream=0)
            assert "p must be" in str(e.value)
        seen["b"] = str(e.value)

    _run_threads([bad_divisor, bad_p])
    assert "divisor" in seen["a"] and "p must be" in seen["b"]


@pytest.mark.gpu
def test_two_reducers_synced_from_two_threads_at_once():
    """Each thread owns a Reducer and a stream; both sync repeatedly at the
    same time. The bits equal the oracle's and a sync of the same inputs run
    alone."""
    torch = pytest.importorskip("torch")
    from ring_all_reduce_ddp_gb300.reducer import Reducer
    from synth import workloads as W
    cfg = W.CONFIGS["tiny"]
    ref, _ = W.make_grads(cfg)
    Reducer(ref, cfg["first_cap"], cfg["cap"]).sync_gradients(W.divisor(cfg))
    torch.cuda.synchronize()
    sets = [W.make_grads(cfg)[0] for _ in range(2)]
    reds = [Reducer(g, cfg["first_cap"], cfg["cap"]) for g in sets]
    streams = [torch.cuda.Stream() for _ in range(2)]

    def worker(i):
        def run():
            torch.cuda.set_device(0)
            with torch.cuda.stream(streams[i]):
                reds[i].sync_gradients(W.divisor(cfg), D.DDP_ALGO_FUSED, D.DDP_SYNC_IN_PLACE, 1.0, streams[i])
                for _ in range(50):  # the mean of equal replicas is the same mean
                    reds[i].sync_gradients(W.divisor(cfg), D.DDP_ALGO_FUSED, D.DDP_SYNC_IN_PLACE, 1.0, streams[i])
            streams[i].synchronize()
        return run

    _run_threads([worker(0), worker(1)])
    for g in sets:  # many concurrent syncs: every replica ends identical
        for t in range(len(g[0])):
            for r in range(1, cfg["p"]):
                assert torch.equal(g[r][t].view(torch.int32), g[0][t].view(torch.int32))
    # one concurrent sync per thread on fresh inputs: the bits of a sync run alone
    fresh = [W.make_grads(cfg)[0] for _ in range(2)]
    reds2 = [Reducer(g, cfg["first_cap"], cfg["cap"]) for g in fresh]

    def once(i):
        def run():
            torch.cuda.set_device(0)
            reds2[i].sync_gradients(W.divisor(cfg), D.DDP_ALGO_FUSED, D.DDP_SYNC_IN_PLACE, 1.0, streams[i])
            streams[i].synchronize()
        return run

    _run_threads([once(0), once(1)])
    from tests.oracle_sync import check_whole_set
    for g, red in zip(fresh, reds2):  # every element against the oracle
        check_whole_set(cfg, red, g)
    for g in fresh:
        for r in range(cfg["p"]):
            for t in range(len(g[r])):
                assert torch.equal(g[r][t].view(torch.int32), ref[r][t].view(torch.int32))
    assert D.ddp_device_error() == 0
