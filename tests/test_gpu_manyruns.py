"""Parity on the tree shapes that take the kernels' less common branches ("Tree Training 技术详解",
section 4.2 mask M_ij and section 4.3 node DFS intervals):

* tiles holding more than TREE_MAX_RUNS (16) runs of one node: agent turns of a few tokens,
  one-token nodes, chains through zero-length nodes.  The forward and the backward then test
  the ancestor interval once per key (or query) instead of once per run;
* trees of more than 1024 tiles, whose longest row or column lists exceed what the kernels
  stage in shared memory (read from global memory past that), and whose plan orders and
  offsets are computed over more than one block's worth of tiles.

Forward and backward are compared with the fp64 oracle at the target tolerances (O, LSE
max-abs 2e-2; dQ, dK, dV 5e-2 of max|reference|)."""
import sys

import numpy as np
import pytest
import torch

import oracle
import tree_masked_attention_plan_gb300 as tam
from workloads import make_tensors, random_tree
from workloads.trees import Workload

from _gateway import gateway_tree
from _gpu import GRAD_TOL, O_TOL, compare_bwd, compare_fwd, f64, oracle_ref, rel_err, run_gpu

pytestmark = pytest.mark.gpu

# the oracle enumerates paths and preorder recursively: a chain of 1100 nodes recurses that deep
sys.setrecursionlimit(max(sys.getrecursionlimit(), 20000))


def _wl(parent, node_len, Hq, Hkv, d):
    return Workload(name="t", parent=np.asarray(parent, np.int32), node_len=np.asarray(node_len, np.int32),
                    Hq=Hq, Hkv=Hkv, d=d)


def _chain(lens):
    return np.array([-1] + list(range(len(lens) - 1))), np.asarray(lens)


def _many_run_trees():
    rng = np.random.default_rng(5)
    return [
        ("chain_300x3", _chain([3] * 300)),
        ("star_400_leaves", (np.array([-1] + [0] * 400), np.r_[20, rng.integers(0, 7, size=400)])),
        ("one_and_zero_chain", _chain([1, 0] * 300)),
        ("random_tiny_nodes", random_tree(21, 300, max_len=6)),
    ]


SHAPES = [(2, 2, 64), (4, 1, 64), (2, 2, 128), (4, 1, 128)]


@pytest.mark.parametrize("Hq,Hkv,d", SHAPES, ids=[f"h{a}_{b}_d{c}" for a, b, c in SHAPES])
@pytest.mark.parametrize("name,tree", _many_run_trees(), ids=[t[0] for t in _many_run_trees()])
def test_tiles_with_many_node_runs(name, tree, Hq, Hkv, d):
    wl = _wl(*tree, Hq, Hkv, d)
    t = make_tensors(wl)
    g = run_gpu(wl.parent, wl.node_len, t)
    nruns = g["plan"].arrays()["tile_nruns"].cpu().numpy()
    assert nruns.max() > tam.MAX_RUNS, "the tree must exercise the per-key mask branch"
    ref = oracle_ref(wl.parent, wl.node_len, t, heads=range(Hq))
    eo, el = compare_fwd(g, ref, range(Hq), wl.n_tokens)
    e = compare_bwd(g, ref, range(Hq), Hq, Hkv)
    print(f"{name}: N={wl.n_tokens} max runs {nruns.max()} O {eo:.2e} LSE {el:.2e} grads {e}")
    assert eo <= O_TOL and el <= O_TOL
    assert max(e.values()) <= GRAD_TOL


def test_gateway_child_of_tiny_nodes():
    """A partition below a gateway whose subtrees are nodes of 0-4 tokens (more than 16 runs per
    tile in the child partitions) matches the whole-tree oracle."""
    from test_gpu_gateway import _tensors, run_partitioned
    dev = torch.device("cuda", 0)
    parent, lens, cut = gateway_tree(6, [90, 61], branch_len=20, n_extra=400, max_len=4)
    N = int(np.sum(lens))
    t = _tensors(N, 4, 1, 128, seed=17)
    P, got = run_partitioned(parent, lens, cut, t, dev)
    runs = max(int(tam.tree_plan(c.parent, c.node_len, device=dev, pos_offset=P["A"]).arrays()["tile_nruns"].max())
               for c in P["children"])
    assert runs > tam.MAX_RUNS
    ref = oracle.attention_nodes(parent, lens, t["q"], t["k"], t["v"], t["u"], heads=list(range(4)), theta=10000.0)
    eo = np.abs(f64(got["o"]) - ref["o"]).max()
    el = np.abs(f64(got["lse"]) - ref["lse"]).max()
    errs = {x: rel_err(f64(got[x]), ref[x]) for x in ("dq", "dk", "dv")}
    print(f"gateway tiny nodes: N={N} A={P['A']} max child runs {runs} O {eo:.2e} LSE {el:.2e} grads {errs}")
    assert eo <= O_TOL and el <= O_TOL
    assert max(errs.values()) <= GRAD_TOL


def test_star_of_1100_leaves():
    """1101 tiles: the root's key tile has a column of 1101 query tiles (more than the 1024 staged
    in shared memory), and the plan's offsets and orders span 1101 tiles.  Whole-tree parity."""
    parent = np.array([-1] + [0] * 1100)
    lens = np.full(1101, 128)
    wl = _wl(parent, lens, 2, 1, 64)
    t = make_tensors(wl)
    g = run_gpu(wl.parent, wl.node_len, t)
    a = g["plan"].arrays()
    col_len = np.diff(a["col_ptr"].cpu().numpy())
    assert g["plan"].n_tiles == 1101 and col_len.max() > 1024
    ref = oracle_ref(wl.parent, wl.node_len, t, heads=[0, 1])
    eo, el = compare_fwd(g, ref, [0, 1], wl.n_tokens)
    e = compare_bwd(g, ref, [0, 1], 2, 1)
    print(f"star 1100: T={g['plan'].n_tiles} longest column {col_len.max()} O {eo:.2e} LSE {el:.2e} grads {e}")
    assert eo <= O_TOL and el <= O_TOL
    assert max(e.values()) <= GRAD_TOL


def test_chain_of_1100_tiles():
    """One path of 140,800 tokens: the last query tiles' rows hold 1100 key tiles (more than the
    1024 staged in shared memory).  The oracle evaluates the last two nodes' queries (the longest
    rows): their O, LSE and dQ are exact there."""
    parent, lens = _chain([128] * 1100)
    wl = _wl(parent, lens, 2, 1, 64)
    t = make_tensors(wl)
    g = run_gpu(wl.parent, wl.node_len, t)
    row_len = np.diff(g["plan"].arrays()["row_ptr"].cpu().numpy())
    assert row_len.max() > 1024
    last = [1098, 1099]
    ref = oracle.attention_nodes(wl.parent, wl.node_len, t["q"], t["k"], t["v"], t["u"], heads=[0, 1],
                                 theta=10000.0, nodes=set(last))
    rows = np.arange(1098 * 128, 1100 * 128)
    o, lse, dq = f64(g["o"]), f64(g["lse"]), f64(g["dq"])
    eo = np.abs(o[rows] - ref["o"][rows]).max()
    el = np.abs(lse[:, rows] - ref["lse"][:, rows]).max()
    eq = rel_err(dq[rows], ref["dq"][rows])
    print(f"chain 1100: longest row {row_len.max()} O {eo:.2e} LSE {el:.2e} dq {eq:.2e}")
    assert eo <= O_TOL and el <= O_TOL and eq <= GRAD_TOL
