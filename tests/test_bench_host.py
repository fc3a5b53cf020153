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
