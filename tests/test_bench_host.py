"""Host-side logic of bench.py (CPU only): clock-sample parsing and the
timed-window filter, on synthetic nvidia-smi lines."""
import datetime

import bench


def _line(ts, sm, reasons=("Not Active",) * 4):
    return ", ".join([ts.strftime("%Y/%m/%d %H:%M:%S.%f")[:-3], str(sm), "2070", "900.00", "0x0"] + list(reasons))


def test_clock_samples_are_filtered_to_the_timed_window():
    t0 = datetime.datetime(2026, 12, 2, 8, 0, 0)
    s = bench.ClockSampler(0)
    s.lines = [_line(t0 + datetime.timedelta(seconds=i * 0.1), 1400 if i < 5 else 2070) for i in range(20)]
    s.lines.append(_line(t0 + datetime.timedelta(seconds=1.2), 1900,
                         ("Not Active", "Not Active", "Not Active", "Active")))
    w = ((t0 + datetime.timedelta(seconds=0.6)).timestamp(), (t0 + datetime.timedelta(seconds=1.5)).timestamp())
    rows = s._parse(w)
    assert len(rows) == 11 and all(r[0] >= 1900 for r in rows)
    assert set().union(*[r[2] for r in rows]) == {"sw_power_cap"}
    assert len(s._parse(None)) == 21


def test_peak_and_workload_text():
    peak, kind = bench.peak_hbm()
    assert peak > 1000 and kind in ("measured", "fallback")
    assert "ResNet-50" in bench.WORKLOAD_TEXT["resnet50"]


def test_literal_traffic_counts_match_the_schedule():
    """The sweep's load-and-store byte counts for the literal schedules, counted
    here access by access over the steps (chunks from the oracle's plan)."""
    from oracle.ring import chunk_bounds
    for p in range(2, 10):
        n = 1024 * p  # the sweep's sizes divide by every p it uses
        M = 4 * n
        chunks = chunk_bounds(n, p)
        # all-reduce: every reduce-scatter step, each rank loads its chunk and the
        # received one and stores the sum; every all-gather step, each rank
        # loads one chunk and stores it at its neighbour
        rs = sum(3 * 4 * (hi - lo) for _ in range(p - 1) for lo, hi in chunks)
        ag = sum(2 * 4 * (hi - lo) for _ in range(p - 1) for lo, hi in chunks)
        assert bench.literal_traffic_bytes("allreduce", "ring_steps", p, M) == rs + ag
        assert bench.literal_traffic_bytes("reduce_scatter_rank", "ring_steps", p, M) == rs
        # all-gather of n / p elements per rank: a placement copy, then p - 1 steps
        m = n // p
        assert bench.literal_traffic_bytes("allgather", "ring_steps", p, M) == 2 * 4 * m * p * p
        # doubling tree: every rank but the root receives one copy of M bytes
        copies = 0
        span = 1
        while span < p:
            copies += sum(1 for v in range(span) if v + span < p)
            span *= 2
        assert copies == p - 1
        assert bench.literal_traffic_bytes("broadcast", "ring_steps", p, M) == 2 * copies * M
    assert bench.literal_traffic_bytes("allreduce", "fused", 8, 1 << 20) is None
    assert bench.literal_traffic_bytes("allreduce", "rd", 8, 1 << 20) is None
