"""Oracle plan: the prefix tree, its root-to-leaf paths, and every per-node / per-token /
per-tile quantity the plan produces (TEST INFRASTRUCTURE ONLY).

Written from "Tree Training 技术详解" (tingdeliu.github.io):
  * section 3.1  - each node holds a token segment; a root-to-leaf path is one sample;
  * section 3.2  - baseline expansion X_base repeats ancestors per path; DFS serialization
                   X_DFS emits each node once, children after their parent (Fig. 2 gives the
                   order n0,n1,n3,n4,n2,n5 for n0->{n1,n2}, n1->{n3,n4}, n2->{n5});
  * section 4.2  - visibility M_ij = 0 iff j <= i and node(j) is node(i) or an ancestor;
  * section 4.3  - node DFS intervals, parent, depth, and a block table of ancestor blocks;
  * section 5    - pos(t) = sum of ancestor segment lengths + offset inside the node;
  * section 6.2  - g_t = number of root-to-leaf paths through t, weight g_t / K;
  * section 12   - per-node depth_token_offset and path_count, concatenated in DFS order;
  * section 13   - N_pairs = sum_t D(t) visible pairs;
  * section 10   - POR = 1 - N_tree / N_flat, S_upper = 1 / (1 - POR).

Quantities are derived from the enumerated paths (membership), not from interval
arithmetic, so that they check the interval-based CUDA plan independently.
Readings where the pages are silent: children are visited in ascending node id, roots in
ascending id; positions start at 0; a node may hold 0 tokens (a zero-length leaf still
ends a path); a forest's K counts the leaves of all roots.
"""
from __future__ import annotations

import sys

import numpy as np

TILE = 128
INT32_MAX = 2 ** 31 - 1


class TreeError(ValueError):
    pass


def validate_tree(parent, node_len):
    """Reject parents out of range, self-parents, cycles, no root, negative lengths and a token
    total outside [1, 2^31 - 1]."""
    parent = np.asarray(parent, dtype=np.int64)
    node_len = np.asarray(node_len, dtype=np.int64)
    n = len(parent)
    if n == 0 or len(node_len) != n:
        raise TreeError("empty tree or length mismatch")
    if np.any(node_len < 0):
        raise TreeError("negative node length")
    for i, p in enumerate(parent):
        if p < -1 or p >= n or p == i:
            raise TreeError(f"node {i}: parent {p} out of range")
    if not np.any(parent == -1):
        raise TreeError("no root")
    for i in range(n):                      # walk to a root in at most n steps
        v, steps = i, 0
        while parent[v] != -1:
            v = parent[v]
            steps += 1
            if steps > n:
                raise TreeError(f"cycle through node {i}")
    total = int(node_len.sum())
    if total < 1 or total > INT32_MAX:
        raise TreeError(f"token total {total} outside [1, 2^31-1]")
    return parent, node_len


def _children(parent):
    ch = [[] for _ in range(len(parent))]
    for c, p in enumerate(parent):
        if p >= 0:
            ch[p].append(c)
    return [sorted(x) for x in ch]


def root_to_leaf_paths(parent, node_len=None):
    """Every root-to-leaf path as a list of node ids, by recursion over children in ascending id
    (roots in ascending id).  These are the K samples of the baseline expansion X_base."""
    parent = np.asarray(parent, dtype=np.int64)
    ch = _children(parent)
    out = []

    def rec(v, prefix):
        prefix = prefix + [v]
        if not ch[v]:
            out.append(prefix)
        for c in ch[v]:
            rec(c, prefix)

    old = sys.getrecursionlimit()
    sys.setrecursionlimit(max(old, 4 * len(parent) + 100))
    try:
        for r in [i for i in range(len(parent)) if parent[i] == -1]:
            rec(r, [])
    finally:
        sys.setrecursionlimit(old)
    return out


def _preorder(parent):
    """Recursive DFS: preorder list and, per node, (enter index, index of last node in subtree)."""
    ch = _children(parent)
    order, enter, last = [], {}, {}

    def rec(v):
        enter[v] = len(order)
        order.append(v)
        for c in ch[v]:
            rec(c)
        last[v] = len(order) - 1

    old = sys.getrecursionlimit()
    sys.setrecursionlimit(max(old, 4 * len(parent) + 100))
    try:
        for r in [i for i in range(len(parent)) if parent[i] == -1]:
            rec(r)
    finally:
        sys.setrecursionlimit(old)
    n = len(parent)
    return (np.array(order, dtype=np.int64), np.array([enter[i] for i in range(n)], dtype=np.int64),
            np.array([last[i] for i in range(n)], dtype=np.int64))


def plan(parent, node_len, tile: int = TILE):
    """The whole plan as a dict of NumPy arrays (int64 / float32), independent of the CUDA plan.

    Per node (indexed by node id): order (DFS preorder of ids), dfs_in, dfs_out (inclusive),
    tok_start (first packed token), depth_off (sum of ancestor lengths), leaves (paths through
    the node).  Per packed token: tok_node, pos, g, w = float32(g / K), tok_in, tok_out, hi
    (last packed token of node(t)'s subtree).  Scalars: n_nodes, n_tokens, n_tiles, n_paths.
    Tile table: tile_class [T*T] u8 (0 empty, 1 partial, 2 full), row/col CSR, LPT orders.
    """
    parent, node_len = validate_tree(parent, node_len)
    n = len(parent)
    order, dfs_in, dfs_out = _preorder(parent)
    paths = root_to_leaf_paths(parent)
    K = len(paths)

    tok_start = np.zeros(n, dtype=np.int64)
    acc = 0
    for v in order:                       # X_DFS: each node's segment once, in preorder
        tok_start[v] = acc
        acc += node_len[v]
    N = int(acc)

    tok_node = np.full(N, -1, dtype=np.int64)
    for v in range(n):
        tok_node[tok_start[v]:tok_start[v] + node_len[v]] = v

    # positions, path counts and depth offsets from the expanded paths (X_base)
    pos = np.full(N, -1, dtype=np.int64)
    g = np.zeros(N, dtype=np.int64)
    depth_off = np.full(n, -1, dtype=np.int64)
    leaves = np.zeros(n, dtype=np.int64)
    for p in paths:
        off = 0
        for v in p:
            if depth_off[v] == -1:
                depth_off[v] = off
            elif depth_off[v] != off:
                raise AssertionError("paths disagree on a node's depth offset")
            leaves[v] += 1
            toks = np.arange(tok_start[v], tok_start[v] + node_len[v])
            idx = np.arange(off, off + node_len[v])
            seen = pos[toks] >= 0
            if np.any(pos[toks][seen] != idx[seen]):
                raise AssertionError("paths disagree on a token position")
            pos[toks] = idx
            g[toks] += 1
            off += node_len[v]
    assert np.all(pos >= 0) and np.all(g >= 1)
    w = (g.astype(np.float64) / K).astype(np.float32)

    # subtree membership from the paths: u is in subtree(v) iff some path has v at or before u
    in_sub = np.zeros((n, n), dtype=bool)
    for p in paths:
        for a, v in enumerate(p):
            in_sub[v, p[a:]] = True
    sub_hi = np.full(n, -1, dtype=np.int64)
    for v in range(n):
        members = [u for u in np.nonzero(in_sub[v])[0] if node_len[u] > 0]
        if members:
            sub_hi[v] = max(tok_start[u] + node_len[u] - 1 for u in members)
    hi = sub_hi[tok_node]

    out = dict(order=order, dfs_in=dfs_in, dfs_out=dfs_out, tok_start=tok_start,
               depth_off=depth_off, leaves=leaves, tok_node=tok_node, pos=pos, g=g, w=w,
               tok_in=dfs_in[tok_node], tok_out=dfs_out[tok_node], hi=hi,
               n_nodes=n, n_tokens=N, n_paths=K, paths=paths)
    out.update(tile_classes(parent, node_len, tile=tile, _plan=out))
    return out


def tile_classes(parent, node_len, tile: int = TILE, _plan=None):
    """Visible-pair count of every tile (qt, kt) and its class, CSR lists and LPT orders.

    A token i sees key j iff j <= i and node(j) is node(i) or one of its ancestors, where the
    ancestors of a node are the nodes before it on a root-to-leaf path through it.  For each
    query node a and each visible key node b the rows of a see, per row i, the keys
    [start(b), min(end(b)-1, i)]; these run lengths are summed per tile.  Class: 0 when the
    tile holds no visible pair, 2 when all tile*tile pairs are visible (so a ragged tile or a
    diagonal tile is never 2), else 1.
    """
    p = _plan if _plan is not None else plan(parent, node_len, tile=tile)
    node_len = np.asarray(node_len, dtype=np.int64)
    N, n = p["n_tokens"], p["n_nodes"]
    T = (N + tile - 1) // tile
    anc = [set() for _ in range(n)]
    for path in p["paths"]:
        for a, v in enumerate(path):
            anc[v].update(path[:a])
    cnt = np.zeros((T, T), dtype=np.int64)
    for a in range(n):
        if node_len[a] == 0:
            continue
        s_a = p["tok_start"][a]
        rows = np.arange(s_a, s_a + node_len[a])
        qt = rows // tile
        for b in sorted(anc[a]) + [a]:
            if node_len[b] == 0:
                continue
            s_b, e_b = p["tok_start"][b], p["tok_start"][b] + node_len[b]
            last = np.minimum(e_b - 1, rows)              # j <= i and j inside b
            for kt in range(s_b // tile, (e_b - 1) // tile + 1):
                lo = max(s_b, kt * tile)
                c = np.clip(np.minimum(last, kt * tile + tile - 1) - lo + 1, 0, None)
                cnt[:, kt] += np.bincount(qt, weights=c, minlength=T).astype(np.int64)
    cls = np.where(cnt == 0, 0, np.where(cnt == tile * tile, 2, 1)).astype(np.uint8)
    row_ptr = np.zeros(T + 1, dtype=np.int64)
    col_ptr = np.zeros(T + 1, dtype=np.int64)
    row_idx, col_idx = [], []
    for q in range(T):
        ks = [k for k in range(T) if cls[q, k] != 0]
        row_idx += ks
        row_ptr[q + 1] = row_ptr[q] + len(ks)
    for k in range(T):
        qs = [q for q in range(T) if cls[q, k] != 0]
        col_idx += qs
        col_ptr[k + 1] = col_ptr[k] + len(qs)
    rcount = np.diff(row_ptr)
    ccount = np.diff(col_ptr)
    row_order = np.array(sorted(range(T), key=lambda q: (-rcount[q], q)), dtype=np.int64)
    last_q = [max((q for q in range(T) if cls[q, k] != 0), default=-1) for k in range(T)]
    col_order = np.array(sorted(range(T), key=lambda k: (-last_q[k], -ccount[k], k)), dtype=np.int64)
    # runs of consecutive packed tokens that belong to one node, per tile (padding = dfs_in -1)
    tok_in = np.full(T * tile, -1, dtype=np.int64)
    tok_out = np.full(T * tile, -2, dtype=np.int64)
    tok_in[:N] = p["dfs_in"][p["tok_node"]]
    tok_out[:N] = p["dfs_out"][p["tok_node"]]
    runs, nruns = [], []
    for t in range(T):
        seg = tok_in[t * tile:(t + 1) * tile]
        st = [c for c in range(tile) if c == 0 or seg[c] != seg[c - 1]]
        ends = st[1:] + [tile]
        runs.append([(a, b, int(seg[a]), int(tok_out[t * tile + a])) for a, b in zip(st, ends)])
        nruns.append(len(st))
    return dict(n_tiles=T, tile_pairs=cnt, tile_class=cls.reshape(-1), row_ptr=row_ptr, tile_runs=runs,
                tile_nruns=np.array(nruns, dtype=np.int64),
                row_idx=np.array(row_idx, dtype=np.int64), col_ptr=col_ptr,
                col_idx=np.array(col_idx, dtype=np.int64), row_order=row_order,
                col_order=col_order, nnz=int(row_ptr[-1]), n_full=int((cls == 2).sum()),
                n_partial=int((cls == 1).sum()))


def tree_stats(p):
    """Token and pair counts of a plan: N_tree, N_flat = sum_t g_t, N_pairs = sum_t (pos_t + 1),
    POR = 1 - N_tree / N_flat, S_upper = N_flat / N_tree (explainer sections 2, 10, 13)."""
    N = p["n_tokens"]
    n_flat = int(p["g"].sum())
    n_pairs = int((p["pos"] + 1).sum())
    return dict(n_tree=N, n_flat=n_flat, n_pairs=n_pairs, por=1.0 - N / n_flat,
                s_upper=n_flat / N, n_paths=p["n_paths"])
