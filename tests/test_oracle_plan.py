"""Pins for the oracle's plan against the pages' worked example, closed forms and brute force.

Every check here computes its expected value some other way than the oracle does: by hand
from the pages (golden fixture), from the explainer's closed forms, by walking parent
pointers instead of enumerating paths, or pair by pair.
"""
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
from workloads import (CONFIGS, caterpillar_tree, make_workload, random_tree, tiny_tree)


# ----------------------------------------------------------------------------------------
# brute-force helpers that walk parent pointers (independent of the oracle's recursion)
def _ancestors_or_self(parent, v):
    out = [v]
    while parent[v] != -1:
        v = parent[v]
        out.append(v)
    return out


def _is_anc_or_self(parent, a, b):
    """a is b or an ancestor of b."""
    return a in _ancestors_or_self(parent, b)


def _leaf_walk_counts(parent):
    """Number of leaves below each node: from every leaf, walk to the root adding one."""
    n = len(parent)
    has_child = np.zeros(n, dtype=bool)
    for p in parent:
        if p >= 0:
            has_child[p] = True
    cnt = np.zeros(n, dtype=np.int64)
    for leaf in np.nonzero(~has_child)[0]:
        for v in _ancestors_or_self(parent, leaf):
            cnt[v] += 1
    return cnt, int((~has_child).sum())


def _random_trees():
    out = []
    for s in range(12):
        out.append(random_tree(s, n_nodes=3 + s * 3, max_len=9, zero_prob=0.2 if s % 3 == 0 else 0.0,
                               n_roots=1 + (s % 4 == 1) * 2))
    out.append(tiny_tree())
    out.append(caterpillar_tree(p=5, T=6, delta=3, a=2))
    return out


# ----------------------------------------------------------------------------------------
def test_tiny_example_golden(golden_dir):
    gd = json.load(open(os.path.join(golden_dir, "tiny_tree.json")))
    p = oracle.plan(gd["parent"], gd["node_len"])
    assert p["order"].tolist() == gd["dfs_order"]
    assert p["tok_start"][p["order"]].tolist() == gd["tok_start_in_dfs_order"]
    assert p["dfs_in"].tolist() == gd["dfs_in_by_id"]
    assert p["dfs_out"].tolist() == gd["dfs_out_by_id"]
    assert p["n_paths"] == gd["n_paths"]
    for v, (lo, hi) in enumerate(gd["pos_range_by_id"]):
        s = p["tok_start"][v]
        assert p["pos"][s:s + gd["node_len"][v]].tolist() == list(range(lo, hi + 1))
        assert np.all(p["g"][s:s + gd["node_len"][v]] == gd["g_by_id"][v])
        assert np.all(p["w"][s:s + gd["node_len"][v]] == np.float32(float(Fraction(gd["w_by_id"][v]))))
    st = oracle.tree_stats(p)
    assert st["n_flat"] == gd["n_flat"] and st["n_tree"] == gd["n_unique"]
    assert st["n_pairs"] == gd["n_pairs"]
    N = gd["n_unique"]
    assert N * (N + 1) // 2 == gd["n_pairs_dense_causal"]
    assert p["n_tiles"] == gd["n_tiles"] and p["tile_class"].tolist() == gd["tile_class"]


def test_tiny_sibling_leak_pairs_hidden():
    """Under plain causal masking n2 would read n1, n3, n4 (section 4.1): the tree mask hides them."""
    parent, node_len = tiny_tree()
    p = oracle.plan(parent, node_len)
    n2 = np.arange(p["tok_start"][2], p["tok_start"][2] + node_len[2])
    hidden = 0
    for i in n2:
        for j in range(i + 1):
            if not _is_anc_or_self(parent, p["tok_node"][j], p["tok_node"][i]):
                hidden += 1
                assert p["tok_node"][j] in (1, 3, 4)
    assert hidden == 8 * (8 + 12 + 12)
    # the tile's visible pair count is the section 13 N_pairs
    assert p["tile_pairs"].sum() == 1424


@pytest.mark.parametrize("p_,T,delta", [(256, 40, 64), (7, 13, 5), (0, 43, 10)])
def test_caterpillar_closed_forms_zero_length_leaves(p_, T, delta):
    """Section 2: T time steps, prefix p, Delta new tokens per step:
    N_flat = Tp + Delta T (T+1)/2 and N_unique = p + T Delta (each step = a zero-length leaf)."""
    parent, lens = caterpillar_tree(p=p_, T=T, delta=delta, a=0)
    plan = oracle.plan(parent, lens)
    st = oracle.tree_stats(plan)
    assert plan["n_paths"] == T
    assert st["n_flat"] == T * p_ + delta * T * (T + 1) // 2
    assert st["n_tree"] == p_ + T * delta
    R = Fraction(st["n_flat"], st["n_tree"])
    assert R == Fraction(T * p_ + Fraction(delta * T * (T + 1), 2), p_ + T * delta)
    if p_ == 0:
        # short prefix: R = (T+1)/2; T = 43 gives the 22x of section 1, POR = 1 - 1/22 (section 10)
        assert R == Fraction(T + 1, 2) == 22
        assert math.isclose(st["por"], 1 - 1 / 22) and round(st["por"] * 100, 2) == 95.45
        assert math.isclose(st["s_upper"], 1 / (1 - st["por"]))


def test_caterpillar_with_action_leaves():
    """The caterpillar workload (a = 16-token action leaves): N_flat = T(p+a) + Delta T(T+1)/2,
    N_unique = p + T(Delta + a) (derived from section 2 with a per-step leaf)."""
    p_, T, delta, a = 256, 40, 64, 16
    plan = oracle.plan(*caterpillar_tree(p_, T, delta, a))
    st = oracle.tree_stats(plan)
    assert st["n_flat"] == T * (p_ + a) + delta * T * (T + 1) // 2 == 63360
    assert st["n_tree"] == p_ + T * (delta + a) == 3456
    assert plan["n_full"] == 51 and plan["n_partial"] == 327


@pytest.mark.parametrize("name", list(CONFIGS))
def test_identity_sum_over_paths(name):
    """Section 6.2: sum_k sum_{t in p_k} l_t = sum_t g_t l_t, with random integer l (exact)."""
    wl = make_workload(name)
    plan = oracle.plan(wl.parent, wl.node_len)
    rng = np.random.default_rng(7)
    ell = rng.integers(-1000, 1000, size=plan["n_tokens"]).astype(np.int64)
    lhs = 0
    for path in plan["paths"]:
        for v in path:
            s = plan["tok_start"][v]
            lhs += int(ell[s:s + wl.node_len[v]].sum())
    assert lhs == int((plan["g"] * ell).sum())
    # and g_t matches a leaf count taken by walking parent pointers
    cnt, K = _leaf_walk_counts(wl.parent)
    assert K == plan["n_paths"]
    assert np.array_equal(plan["g"], cnt[plan["tok_node"]])


@pytest.mark.parametrize("tree", _random_trees())
def test_plan_against_parent_walks(tree):
    parent, node_len = tree
    p = oracle.plan(parent, node_len)
    n, N = len(parent), p["n_tokens"]
    # section 5: pos = sum of ancestor lengths + offset, by walking parents
    for v in range(n):
        off = sum(int(node_len[a]) for a in _ancestors_or_self(parent, v)[1:])
        assert p["depth_off"][v] == off
        s = p["tok_start"][v]
        assert p["pos"][s:s + node_len[v]].tolist() == list(range(off, off + node_len[v]))
    # DFS intervals: u in subtree(v) (parent walk)  <=>  dfs_in(v) <= dfs_in(u) <= dfs_out(v)
    for v in range(n):
        for u in range(n):
            walk = _is_anc_or_self(parent, v, u)
            assert walk == (p["dfs_in"][v] <= p["dfs_in"][u] <= p["dfs_out"][v])
    # preorder: every parent before its children, siblings in ascending id, subtrees contiguous
    where = {v: i for i, v in enumerate(p["order"])}
    for u in range(n):
        if parent[u] >= 0:
            assert where[parent[u]] < where[u]
        for w_ in range(u + 1, n):
            if parent[w_] == parent[u]:                 # siblings (or roots) in ascending id
                assert where[u] < where[w_]
    # token layout (X_DFS): node segments back to back in preorder
    ts = p["tok_start"][p["order"]]
    assert ts[0] == 0 and np.array_equal(ts[1:], ts[:-1] + np.asarray(node_len)[p["order"]][:-1])
    cnt, K = _leaf_walk_counts(parent)
    assert np.array_equal(p["leaves"], cnt) and K == p["n_paths"]
    assert np.array_equal(p["w"], (p["g"] / K).astype(np.float32))


@pytest.mark.parametrize("tree", _random_trees())
def test_mask_forms_agree(tree):
    """Section 4.2 mask (ancestor walk) == interval form on dfs_in/dfs_out == j <= i <= hi[j]
    == 'some root-to-leaf path holds both'."""
    parent, node_len = tree
    p = oracle.plan(parent, node_len)
    N = p["n_tokens"]
    member = np.zeros((N, p["n_paths"]), dtype=bool)
    for k, path in enumerate(p["paths"]):
        for v in path:
            member[p["tok_start"][v]:p["tok_start"][v] + node_len[v], k] = True
    for i in range(N):
        ni = p["tok_node"][i]
        anc = set(_ancestors_or_self(parent, ni))
        for j in range(N):
            nj = p["tok_node"][j]
            m_walk = j <= i and nj in anc
            m_int = j <= i and p["dfs_in"][nj] <= p["dfs_in"][ni] <= p["dfs_out"][nj]
            m_hi = j <= i <= p["hi"][j]
            m_path = j <= i and bool(np.any(member[i] & member[j]))
            assert m_walk == m_int == m_hi == m_path


@pytest.mark.parametrize("tile", [4, 8, 16])
@pytest.mark.parametrize("seed", range(6))
def test_tile_classes_pairwise(tile, seed):
    parent, node_len = random_tree(100 + seed, n_nodes=4 + 4 * seed, max_len=11,
                                   zero_prob=0.15, n_roots=1 + seed % 2)
    p = oracle.plan(parent, node_len, tile=tile)
    N, T = p["n_tokens"], p["n_tiles"]
    cnt = np.zeros((T, T), dtype=np.int64)
    for i in range(N):
        anc = set(_ancestors_or_self(parent, p["tok_node"][i]))
        for j in range(i + 1):
            if p["tok_node"][j] in anc:
                cnt[i // tile, j // tile] += 1
    assert np.array_equal(cnt, p["tile_pairs"])
    cls = p["tile_class"].reshape(T, T)
    for q in range(T):
        for k in range(T):
            expect = 0 if cnt[q, k] == 0 else (2 if cnt[q, k] == tile * tile else 1)
            assert cls[q, k] == expect
            if q == k:
                assert cls[q, k] == 1          # a diagonal tile is never all-visible
    # CSR lists ascending, counts and heaviest-first orders consistent
    rp, ri, cp, ci = p["row_ptr"], p["row_idx"], p["col_ptr"], p["col_idx"]
    for q in range(T):
        assert ri[rp[q]:rp[q + 1]].tolist() == [k for k in range(T) if cls[q, k]]
    for k in range(T):
        assert ci[cp[k]:cp[k + 1]].tolist() == [q for q in range(T) if cls[q, k]]
    rc = np.diff(rp)[p["row_order"]]
    assert sorted(p["row_order"].tolist()) == list(range(T)) and np.all(np.diff(rc) <= 0)
    # columns: by descending last non-empty query tile, then descending count, then index
    last = [max(q for q in range(T) if cls[q, k]) for k in range(T)]
    key = [(-last[k], -(cp[k + 1] - cp[k]), k) for k in p["col_order"]]
    assert sorted(p["col_order"].tolist()) == list(range(T)) and key == sorted(key)
    assert p["nnz"] == int((cls != 0).sum()) == p["n_full"] + p["n_partial"]


@pytest.mark.parametrize("tile", [8, 16])
@pytest.mark.parametrize("seed", range(5))
def test_tile_runs_rebuild_the_mask(tile, seed):
    """The per-tile node runs partition each key tile into maximal stretches of one node, carry
    that node's Euler interval, and the interval test over runs (plus j <= i) reproduces the
    mask found by walking parents, for every query row against every key tile."""
    parent, node_len = random_tree(300 + seed, n_nodes=5 + 6 * seed, max_len=9,
                                   zero_prob=0.2, n_roots=1 + seed % 3)
    p = oracle.plan(parent, node_len, tile=tile)
    N, T = p["n_tokens"], p["n_tiles"]
    for kt in range(T):
        runs = p["tile_runs"][kt]
        assert p["tile_nruns"][kt] == len(runs)
        assert runs[0][0] == 0 and runs[-1][1] == tile
        for (a, b, din, dout), nxt in zip(runs, runs[1:] + [None]):
            assert a < b and (nxt is None or (nxt[0] == b and nxt[2] != din))
            for j in range(kt * tile + a, kt * tile + b):
                if j < N:
                    v = p["tok_node"][j]
                    assert (din, dout) == (p["dfs_in"][v], p["dfs_out"][v])
                else:                                  # padding keys: an empty interval
                    assert (din, dout) == (-1, -2)
        for i in range(N):
            anc = set(_ancestors_or_self(parent, p["tok_node"][i]))
            qin = p["dfs_in"][p["tok_node"][i]]
            for (a, b, din, dout) in runs:
                for j in range(kt * tile + a, kt * tile + b):
                    by_runs = j <= i and din <= qin <= dout
                    by_walk = j < N and j <= i and p["tok_node"][j] in anc
                    assert by_runs == by_walk, (i, j)


def test_weight_double_rounding_equals_fp32_division():
    """w = float32(g/K) computed in fp64 equals IEEE fp32 division g/K (53 >= 2*24 + 2)."""
    g = np.arange(1, 700, dtype=np.int64)
    for K in range(1, 700):
        gg = g[g <= K]
        a = (gg.astype(np.float64) / K).astype(np.float32)
        b = gg.astype(np.float32) / np.float32(K)
        assert np.array_equal(a, b)


@pytest.mark.parametrize("parent,lens", [
    ([0], [3]),                       # self parent
    ([-1, 5], [1, 1]),                # parent out of range
    ([1, 0], [1, 1]),                 # cycle, no root
    ([-1, 2, 1], [1, 1, 1]),          # cycle below a root
    ([-1, 0], [1, -1]),               # negative length
    ([-1, 0], [0, 0]),                # no tokens
    ([], []),                         # empty
])
def test_validate_rejects(parent, lens):
    with pytest.raises(oracle.TreeError):
        oracle.validate_tree(parent, lens)


def test_forest_is_block_diagonal():
    """A forest of single-node chains: each token sees exactly the earlier tokens of its own
    sequence, positions restart at 0 (agent-RL tutorial section 14.1), g = 1, w = 1/K."""
    wl = make_workload("forest")
    p = oracle.plan(wl.parent, wl.node_len)
    assert p["n_paths"] == len(wl.parent)
    assert np.all(p["g"] == 1)
    starts = np.repeat(p["tok_start"], wl.node_len)
    assert np.array_equal(p["pos"], np.arange(p["n_tokens"]) - starts)
    assert oracle.tree_stats(p)["n_pairs"] == int(sum(L * (L + 1) // 2 for L in wl.node_len))


def test_rollout_generator_shape():
    wl = make_workload("rollout32k")
    assert wl.n_tokens <= 32768 and wl.n_tokens > 32768 - 16
    assert np.all(wl.parent[1:] < np.arange(1, len(wl.parent)))
    cnt, K = _leaf_walk_counts(wl.parent)
    depth = [len(_ancestors_or_self(wl.parent, v)) - 1 for v in range(len(wl.parent))]
    assert max(depth) <= 5 and K >= 2
