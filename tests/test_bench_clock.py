"""bench.py's in-kernel clock: per-launch medians for long launches, a pooled clock for
short ones, whose global-timer intervals are coarse (host logic, no GPU)."""
from __future__ import annotations

import torch

import bench


def _trace(spans_ns, mhz, step_ns=0):
    """Clock-trace words for launches of the given lengths at `mhz`, with the global
    timer read in steps of `step_ns` (0: exact)."""
    rows, t, c = [], 1_000_000, 5_000_000
    for i, dn in enumerate(spans_ns):
        t0, t1 = t, t + dn
        q0 = t0 - (t0 % step_ns) if step_ns else t0
        q1 = t1 - (t1 % step_ns) if step_ns else t1
        c0, c1 = c, c + int(round(dn * mhz / 1e3))
        rows.append([q0, c0, q1, c1])
        t, c = t1 + 3_137 + 17 * i, c1 + 1_000
    return torch.tensor(rows, dtype=torch.int64)


def test_long_launches_report_the_median():
    kc = bench.kernel_clock_mhz(_trace([150_000] * 50, 1_400.0, step_ns=1_000))
    out = bench.merge_clocks(None, kc)
    assert abs(out["sm_mhz"] - 1_400.0) < 15.0
    assert "median of 50" in out["sm_mhz_source"]


def test_short_launches_report_the_pooled_clock():
    spans = [6_600 + 37 * (i % 11) for i in range(400)]
    kc = bench.kernel_clock_mhz(_trace(spans, 1_950.0, step_ns=1_000))
    per = kc["per_launch"]
    assert max(per) > 2_070.0                 # single intervals read above the maximum clock
    out = bench.merge_clocks(None, kc)
    assert abs(out["sm_mhz"] - 1_950.0) < 20.0, out["sm_mhz"]
    assert "pooled over 400" in out["sm_mhz_source"]
    assert out["kernel_mhz_max"] == max(per) and out["kernel_mhz_min"] == min(per)


def test_no_trace_leaves_the_smi_record():
    smi = {"sm_mhz": 1_700.0, "sm_max_mhz": 2_070.0, "reasons": [], "samples": 5, "samples_under_load": 5,
           "power_w_max": 900.0}
    out = bench.merge_clocks(smi, None)
    assert out["sm_mhz"] == 1_700.0 and "nvidia-smi" in out["sm_mhz_source"]
    empty = bench.kernel_clock_mhz(torch.zeros(3, 4, dtype=torch.int64))
    assert empty == {"per_launch": [], "pooled": None, "median_ns": None}
    assert bench.merge_clocks(None, empty)["sm_mhz"] is None


def test_launches_too_short_give_no_in_kernel_clock():
    spans = [2_600 + 37 * (i % 11) for i in range(400)]
    kc = bench.kernel_clock_mhz(_trace(spans, 1_950.0, step_ns=1_000))
    smi = {"sm_mhz": None, "sm_max_mhz": 2_070.0, "reasons": [], "samples": 3, "samples_under_load": 0,
           "power_w_max": 150.0}
    out = bench.merge_clocks(smi, kc)
    assert out["sm_mhz"] is None and "not used" in out["sm_mhz_source"]


def test_pooled_clock_above_the_maximum_is_dropped():
    spans = [9_000] * 100
    kc = bench.kernel_clock_mhz(_trace(spans, 2_600.0))       # a clock no GB300 SM reaches
    smi = {"sm_mhz": 1_800.0, "sm_max_mhz": 2_070.0, "reasons": [], "samples": 5, "samples_under_load": 5,
           "power_w_max": 900.0}
    out = bench.merge_clocks(smi, kc)
    assert out["sm_mhz"] == 1_800.0 and "not used" in out["sm_mhz_source"]
