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
