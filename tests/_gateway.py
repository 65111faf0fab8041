"""Test-side bookkeeping for tree partitions ("Tree Training 技术详解", section 8.2): cut a tree
below one node, describe the parent partition, the child partitions (subtrees of the cut node's
children) and the gateway (the tokens on the path from the root to the cut node, root first),
and map every partition token back to its index in the whole tree's packed order.

Nothing here computes attention; it only renumbers nodes and tokens.  Node ids keep their
relative order inside each partition, so a partition's depth-first order (children by ascending
id) is the whole tree's order restricted to it.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

import oracle


@dataclass
class Part:
    parent: np.ndarray        # partition tree, ids 0..n-1
    node_len: np.ndarray
    nodes: np.ndarray         # whole-tree id of each partition node
    tokens: np.ndarray        # whole-tree packed index of each partition token (partition order)
    pos_offset: int           # 0 for the parent partition, the gateway length for children


def _subtree(parent, v):
    kids = {}
    for c, p in enumerate(parent):
        kids.setdefault(int(p), []).append(c)
    out, stack = [], [v]
    while stack:
        x = stack.pop()
        out.append(x)
        stack.extend(kids.get(x, []))
    return sorted(out)


def _make_part(parent, node_len, full_plan, nodes, pos_offset):
    nodes = np.array(sorted(nodes), dtype=np.int64)
    remap = {int(v): i for i, v in enumerate(nodes)}
    par = np.array([remap.get(int(parent[v]), -1) for v in nodes], dtype=np.int64)
    lens = np.asarray(node_len, dtype=np.int64)[nodes]
    sub = oracle.plan(par, lens)
    tokens = np.empty(sub["n_tokens"], dtype=np.int64)
    for i, v in enumerate(nodes):
        s_sub, s_full, n = sub["tok_start"][i], full_plan["tok_start"][v], lens[i]
        tokens[s_sub:s_sub + n] = np.arange(s_full, s_full + n)
    return Part(parent=par, node_len=lens, nodes=nodes, tokens=tokens, pos_offset=pos_offset)


def partition(parent, node_len, cut):
    """Parent partition (everything but the subtrees of cut's children), one child partition per
    child of cut, the gateway tokens (whole-tree indices, path order) and, for each gateway row,
    its index inside the parent partition."""
    parent = np.asarray(parent, dtype=np.int64)
    full = oracle.plan(parent, node_len)
    path = [cut]
    while parent[path[-1]] >= 0:
        path.append(int(parent[path[-1]]))
    path = path[::-1]                                 # root ... cut
    gw_tokens = np.concatenate([np.arange(full["tok_start"][v], full["tok_start"][v] + node_len[v])
                                for v in path]).astype(np.int64)
    A = len(gw_tokens)
    kids = [c for c in range(len(parent)) if parent[c] == cut]
    child_sets = [_subtree(parent, c) for c in kids]
    in_child = set(x for cs in child_sets for x in cs)
    par_nodes = [v for v in range(len(parent)) if v not in in_child]
    ppart = _make_part(parent, node_len, full, par_nodes, 0)
    children = [_make_part(parent, node_len, full, cs, A) for cs in child_sets]
    where = {int(t): i for i, t in enumerate(ppart.tokens)}
    gw_rows = np.array([where[int(t)] for t in gw_tokens], dtype=np.int64)
    return dict(full=full, parent=ppart, children=children, gw_tokens=gw_tokens, gw_rows=gw_rows, A=A)


def gateway_tree(seed: int, gw_lens, branch_len: int, n_extra: int, max_len: int):
    """A tree with a chosen root-to-cut path: nodes 0..len(gw_lens)-1 form the path (lengths
    gw_lens), the cut node (last of them) gets two random subtrees below it, and the root gets
    one more random branch beside the path.  Returns (parent, node_len, cut)."""
    rng = np.random.default_rng(seed)
    parent = [-1] + list(range(len(gw_lens) - 1))
    lens = list(gw_lens)
    cut = len(gw_lens) - 1
    parent.append(0)                                  # a side branch of the root
    lens.append(branch_len)
    side = len(parent) - 1
    heads = []
    for _ in range(2):                                # two children of the cut node
        parent.append(cut)
        lens.append(int(rng.integers(1, max_len + 1)))
        heads.append(len(parent) - 1)
    for i in range(n_extra):                          # random growth below the children / side
        attach = int(rng.choice(heads + [side] + list(range(len(gw_lens) + 1, len(parent)))))
        parent.append(attach)
        lens.append(int(rng.integers(0 if i % 5 == 4 else 1, max_len + 1)))
    return np.array(parent, dtype=np.int64), np.array(lens, dtype=np.int64), cut
