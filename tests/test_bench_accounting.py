"""The bench's host-side work accounting (the FLOP count behind every TFLOP/s it prints)
against the oracle: N, K, N_pairs = sum_t (pos_t + 1) and N_flat = sum_t g_t for every
workload, computed by bench.py with plain loops over parent pointers and by the oracle's plan
from the root-to-leaf paths."""
import os
import sys

import pytest

import oracle
from workloads import CONFIGS, make_workload

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
import bench  # noqa: E402


@pytest.mark.parametrize("name", sorted(CONFIGS))
def test_host_stats_match_the_oracle(name):
    wl = make_workload(name)
    got = bench.host_stats(wl.parent, wl.node_len)
    ref = oracle.tree_stats(oracle.plan(wl.parent, wl.node_len))
    assert got["N"] == ref["n_tree"]
    assert got["K"] == ref["n_paths"]
    assert got["n_pairs"] == ref["n_pairs"]
    assert got["n_flat"] == ref["n_flat"]


def _clock_line(t, sm_mhz, power_cap="Not Active"):
    import datetime
    ts = datetime.datetime.fromtimestamp(t).strftime("%Y/%m/%d %H:%M:%S.%f")[:-3]
    return f"{ts}, {sm_mhz}, 2070, 900.00, 0x0000000000000000, Not Active, Not Active, Not Active, {power_cap}\n"


def test_clock_summary_keeps_the_timed_region(tmp_path):
    """Samples before and after the timed region (an idle GPU at low clocks) are left out; a
    throttle reason seen inside it is reported."""
    import time
    cs = bench.ClockSampler(0)
    cs.path = str(tmp_path / "clocks.csv")
    t0 = time.time()
    with open(cs.path, "w") as f:
        f.write(_clock_line(t0 - 0.3, 600) + _clock_line(t0 + 0.01, 2070) +
                _clock_line(t0 + 0.03, 2040, "Active") + _clock_line(t0 + 0.5, 900))
    cs.t0, cs.t1 = t0, t0 + 0.05
    s = cs.summary()
    assert s["samples"] == 2
    assert s["sm_mhz"] == 2055.0
    assert s["reasons"] == ["sw_power_cap"]


def test_clock_summary_short_region_takes_the_nearest_sample(tmp_path):
    import time
    cs = bench.ClockSampler(0)
    cs.path = str(tmp_path / "clocks.csv")
    t0 = time.time()
    with open(cs.path, "w") as f:
        f.write(_clock_line(t0 - 0.3, 600) + _clock_line(t0 + 0.05, 2070) + _clock_line(t0 + 0.4, 900))
    cs.t0, cs.t1 = t0, t0 + 0.002
    s = cs.summary()
    assert s["samples"] == 1 and s["sm_mhz"] == 2070.0 and s["reasons"] == []
