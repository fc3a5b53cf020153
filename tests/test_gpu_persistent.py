"""The persistent literal ring: one cooperative kernel in which every simulated
rank's blocks wait, boundedly, for their left neighbour's previous step.

Parity: the same bits as the oracle's literal ring. Failure detection: the
host injects "rank f never posts step t"; the successor's wait must run out
within its limit, the kernel must record where it gave up and end, the
library's device error word must report it, and the context must stay usable.
Nothing here faults, traps or hangs the GPU: every wait has a 50 ms limit."""
import time

import numpy as np
import pytest

import ring_all_reduce_ddp_gb300 as D
from oracle import ring as orc
from tests.helpers import assert_bit_equal, make_replicas, to_host

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

LIMIT_NS = 50_000_000  # 50 ms per wait


@pytest.mark.parametrize("p,n", [(1, 1000), (2, 1), (2, 4099), (3, 10007), (4, 277421), (8, 65536 * 3 + 5),
                                 (8, 7), (16, 100003), (64, 262147)])
def test_persistent_ring_matches_oracle(p, n):
    devs, hosts, _ = make_replicas(p, n, "f32", "normal", seed=900 + p)
    status = torch.full((4,), -1, dtype=torch.int32, device="cuda")
    D.ddp_allreduce_persistent(devs, n, D.DDP_FLOAT32, float(p), LIMIT_NS, -1, 0, status)
    torch.cuda.synchronize()
    want, _ = orc.allreduce(hosts, n, float(p))
    for r in range(p):
        assert_bit_equal(to_host(devs[r]), want[r], f"replica {r}")
    assert status.cpu().tolist() == [0, 0, 0, 0]
    assert D.ddp_device_error() == 0


@pytest.mark.parametrize("p,fault_rank,fault_step", [(2, 0, 0), (3, 1, 2), (4, 2, 0), (8, 5, 3), (8, 0, 13),
                                                     (16, 7, 20)])
def test_injected_fault_is_detected_and_the_context_survives(p, fault_rank, fault_step):
    n = 40000 * p + 3
    devs, hosts, _ = make_replicas(p, n, "f32", "uniform", seed=950 + p)
    status = torch.zeros(4, dtype=torch.int32, device="cuda")
    t0 = time.perf_counter()
    D.ddp_allreduce_persistent(devs, n, D.DDP_FLOAT32, 1.0, LIMIT_NS, fault_rank, fault_step, status)
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    code, rank, step, gave_up = status.cpu().tolist()
    assert code == D.DDP_ERR_TIMEOUT
    # the first wait to run out is a successor of the stopped rank, waiting for
    # the step the stoppage withheld from it: rank f+j at step fault_step+j (or
    # the final check, step 2(p-1))
    j = (rank - fault_rank) % p
    assert j >= 1
    assert step == min(fault_step + j, 2 * (p - 1))
    assert gave_up >= 1
    assert elapsed < 50 * LIMIT_NS / 1e9 + 5.0
    assert D.ddp_device_error() == 2  # read and cleared
    assert D.ddp_device_error() == 0
    # the context is still usable: a normal all-reduce on fresh data is exact
    devs2, hosts2, _ = make_replicas(p, 1001, "f32", "normal", seed=960 + p)
    D.ddp_allreduce(devs2, 1001, D.DDP_FLOAT32, float(p))
    want, _ = orc.allreduce(hosts2, 1001, float(p))
    for r in range(p):
        assert_bit_equal(to_host(devs2[r]), want[r])


@pytest.mark.parametrize("p,n", [(1, 999), (2, 4099), (4, 277421), (8, 65536 * 3 + 5), (16, 100003)])
def test_persistent_ring_in_bf16_rounds_once(p, n):
    """bf16 replicas: the ring runs on fp32 partials in a workspace and each
    finished value is rounded once, so the bits equal the literal ring's."""
    devs, hosts, _ = make_replicas(p, n, "bf16", "normal", seed=970 + p)
    status = torch.full((4,), -1, dtype=torch.int32, device="cuda")
    before = D.ddp_kernel_launches()
    D.ddp_allreduce_persistent(devs, n, D.DDP_BFLOAT16, float(p), LIMIT_NS, -1, 0, status)
    launched = D.ddp_kernel_launches() - before
    torch.cuda.synchronize()
    want, _ = orc.allreduce(hosts, n, float(p), "bf16")
    for r in range(p):
        assert_bit_equal(to_host(devs[r]), want[r], f"replica {r}")
    assert status.cpu().tolist() == [0, 0, 0, 0]
    assert launched == (3 if p > 1 else 1)  # widen, the ring, narrow
    assert D.ddp_device_error() == 0


def test_bf16_persistent_ring_reports_an_injected_fault():
    p, n = 4, 40000 * 4 + 3
    devs, _, _ = make_replicas(p, n, "bf16", "uniform", seed=980)
    status = torch.zeros(4, dtype=torch.int32, device="cuda")
    D.ddp_allreduce_persistent(devs, n, D.DDP_BFLOAT16, 1.0, LIMIT_NS, 1, 2, status)
    torch.cuda.synchronize()
    code, rank, step, gave_up = status.cpu().tolist()
    assert code == D.DDP_ERR_TIMEOUT and gave_up >= 1
    j = (rank - 1) % p
    assert j >= 1 and step == min(2 + j, 2 * (p - 1))
    assert D.ddp_device_error() == 2
    assert D.ddp_device_error() == 0


def test_persistent_ring_rejects_bad_arguments():
    devs, _, _ = make_replicas(4, 100, "f32")
    with pytest.raises(D.DDPError) as e:
        D.ddp_allreduce_persistent(devs, 100, D.DDP_FLOAT32, 1.0, 0, 4, 0)
    assert e.value.status == D.DDP_ERR_ARG
    with pytest.raises(D.DDPError) as e:
        D.ddp_allreduce_persistent(devs, 100, D.DDP_FLOAT32, 1.0, 0, 1, 6)  # only steps 0..5 exist
    assert e.value.status == D.DDP_ERR_ARG
