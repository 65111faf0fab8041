"""Host-side bookkeeping for running a tree as partitions ("Tree Training 技术详解", section 8.2).

A tree too large for one pass is cut below a node `cut`: the parent partition keeps every node
except the subtrees of cut's children, and each child of cut roots one child partition.  The
child partitions read the K/V of the path root..cut (the gateway) from the parent partition
instead of recomputing it, and their gradients w.r.t. the gateway are relayed back to it.

This module only renumbers nodes and tokens; the packed token starts come from the library's
own host plan pass (tree_plan_nodes), and the attention itself runs in the library.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np


@dataclass
class Partition:
    parent: np.ndarray        # partition tree, node ids 0..n-1 (relative order of the whole tree's ids)
    node_len: np.ndarray
    nodes: np.ndarray         # whole-tree id of each partition node
    tokens: np.ndarray        # whole-tree packed index of each partition token, in partition order
    pos_offset: int           # first position of the partition's root(s): 0, or the gateway length


def packed_starts(parent, node_len):
    """First packed token of every node, from the library's host plan pass (depth-first
    preorder, roots and children by ascending id)."""
    from . import tree_plan_nodes
    return tree_plan_nodes(parent, node_len)["tok_start"]


def _subtree(kids, v):
    out, stack = [], [v]
    while stack:
        x = stack.pop()
        out.append(x)
        stack.extend(kids[x])
    return out


def _part(parent, node_len, starts, nodes, pos_offset):
    nodes = np.array(sorted(nodes), dtype=np.int64)
    remap = {int(v): i for i, v in enumerate(nodes)}
    par = np.array([remap.get(int(parent[v]), -1) for v in nodes], dtype=np.int64)
    lens = node_len[nodes]
    sub = packed_starts(par, lens)
    tokens = np.empty(int(lens.sum()), dtype=np.int64)
    for i, v in enumerate(nodes):
        tokens[sub[i]:sub[i] + lens[i]] = np.arange(starts[v], starts[v] + lens[i])
    return Partition(parent=par, node_len=lens, nodes=nodes, tokens=tokens, pos_offset=pos_offset)


def partition_tree(parent, node_len, cut: int) -> dict:
    """Cut below node `cut` (which must have children).  Returns dict(parent=Partition,
    children=[Partition], gw_tokens=whole-tree tokens of the path root..cut in path order,
    gw_rows=their indices inside the parent partition, A=gateway length)."""
    parent = np.asarray(parent, dtype=np.int64)
    node_len = np.asarray(node_len, dtype=np.int64)
    kids = [[] for _ in range(len(parent))]
    for v, p in enumerate(parent):
        if p >= 0:
            kids[p].append(v)
    if not kids[cut]:
        raise ValueError(f"node {cut} has no children to cut off")
    starts = packed_starts(parent, node_len)
    path = [cut]
    while parent[path[-1]] >= 0:
        path.append(int(parent[path[-1]]))
    path.reverse()
    gw_tokens = np.concatenate([np.arange(starts[v], starts[v] + node_len[v]) for v in path]).astype(np.int64)
    A = int(len(gw_tokens))
    if A == 0:
        raise ValueError("the path to the cut node holds no tokens")
    child_sets = [_subtree(kids, c) for c in kids[cut]]
    below = set(x for cs in child_sets for x in cs)
    ppart = _part(parent, node_len, starts, [v for v in range(len(parent)) if v not in below], 0)
    children = [_part(parent, node_len, starts, cs, A) for cs in child_sets if node_len[cs].sum() > 0]
    where = np.empty(int(node_len.sum()), dtype=np.int64)
    where[ppart.tokens] = np.arange(len(ppart.tokens))
    return dict(parent=ppart, children=children, gw_tokens=gw_tokens, gw_rows=where[gw_tokens], A=A, cut=int(cut))


def context_tree(part: Partition, ctx_len: int):
    """A child partition's tree with one more root in front (node 0, holding `ctx_len` tokens):
    the partition's nodes follow as ids 1.., their root now a child of node 0, so depth-first
    packing puts the context tokens first and the partition's tokens after them in partition
    order.  Layers that carry context along root paths (section 9) run on this tree:
    * causal convolution with K taps: node 0 holds the gateway path's last min(K-1, A) tokens
      (their rows gathered from the parent partition), its upstream gradient rows are zero, and
      the gradient its rows receive is the child's contribution to those gateway tokens;
    * recurrent-state routing: node 0 (ctx_len >= 1) carries the state the gateway path ends
      with, which every node of the partition that has no token-holding ancestor inside it
      starts from; the routing backward's gradient for node 0 goes to that gateway node."""
    if ctx_len < 0:
        raise ValueError("ctx_len must be >= 0")
    parent = np.concatenate([[-1], np.where(part.parent < 0, 0, part.parent + 1)]).astype(np.int64)
    node_len = np.concatenate([[ctx_len], part.node_len]).astype(np.int64)
    return parent, node_len


def gateway_state_node(P: dict, parent, node_len) -> int:
    """Index, inside the parent partition of partition_tree's result P, of the node whose final
    recurrent state the child partitions start from: the cut node if it holds tokens, else its
    nearest ancestor that does (-1 if none: the children start from zeros)."""
    parent = np.asarray(parent, dtype=np.int64)
    node_len = np.asarray(node_len, dtype=np.int64)
    ppart = P["parent"]
    where = {int(v): i for i, v in enumerate(ppart.nodes)}
    v = int(P["cut"])
    while v >= 0 and node_len[v] == 0:
        v = int(parent[v])
    return where[v] if v >= 0 else -1


def largest_cut(parent, node_len):
    """A cut that moves the most tokens into child partitions: the node with children whose
    children's subtrees hold the most tokens (ties: smallest id)."""
    parent = np.asarray(parent, dtype=np.int64)
    node_len = np.asarray(node_len, dtype=np.int64)
    size = node_len.astype(np.int64).copy()
    for v in sorted(range(len(parent)), key=lambda x: -_depth(parent, x)):
        if parent[v] >= 0:
            size[parent[v]] += size[v]
    below = {}
    for v, p in enumerate(parent):
        if p >= 0:
            below[p] = below.get(p, 0) + size[v]
    return max(sorted(below), key=lambda v: below[v])


def _depth(parent, v):
    d = 0
    while parent[v] >= 0:
        v = parent[v]
        d += 1
    return d
