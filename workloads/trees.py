"""Seeded synthetic prefix trees for the five benchmark workloads and for property tests.

A tree is two int32 arrays: ``parent[n]`` (-1 for a root) and ``node_len[n]`` (tokens held
by each node).  Node ids are assigned so that every parent id is smaller than its
children's ids.  Lengths follow the log-normal idiom of the agent-RL scaling tutorial
("规模扩展与效率", section 14.2): ``(median * exp(sigma * randn)).clamp(lo, hi).long()``.

Workload shapes (from the Tree Training explainer "Tree Training 技术详解", sections 2-3 and
11, and the packing section 14.1 of the agent-RL tutorial):

* ``tiny``        - the 6-node example tree n0->{n1,n2}, n1->{n3,n4}, n2->{n5} (Fig. 2),
                    lengths 16,8,8,12,12,8; 1 head, d = 64.
* ``caterpillar`` - a VLA episode: prefix p = 256, T = 40 trunk segments of 64 tokens,
                    each trunk node with a 16-token action leaf (section 2, section 11.1).
* ``rollout32k``  - an agentic rollout tree: 2048-token root, 2-4 children per node to
                    depth 5, node lengths log-normal(256, 0.8) clipped to [16, 4096],
                    trimmed to a 32768-token prefix subtree.
* ``forest``      - block-diagonal packing: sequences of log-normal length (median 1024,
                    p90 4096, max 8192) packed first-fit-decreasing into rows of 16384;
                    the first 8 rows concatenated as a forest of single-node chains.
* ``large128k``   - 8192-token root, full binary branching to depth 6 (64 leaves),
                    log-normal(1536, 0.8) lengths rescaled to 131072 tokens in total.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch


@dataclass
class Workload:
    name: str
    parent: np.ndarray          # int32 [n_nodes]
    node_len: np.ndarray        # int32 [n_nodes]
    Hq: int
    Hkv: int
    d: int
    theta: float = 10000.0
    uniform_grad: bool = False  # per-token loss gradient U_t = 1 (the tiny example)
    fp32_inputs: bool = False   # Q/K/V drawn in fp32 (then rounded to bf16 for the kernels)
    seeds: dict = field(default_factory=lambda: {"tree": 0, "q": 1, "k": 2, "v": 3, "u": 4})

    @property
    def n_tokens(self) -> int:
        return int(self.node_len.sum())


def _lognormal(gen: torch.Generator, n: int, median: float, sigma: float,
               lo: float | None, hi: float | None) -> torch.Tensor:
    x = median * torch.exp(sigma * torch.randn(n, generator=gen, dtype=torch.float64))
    if lo is not None or hi is not None:
        x = x.clamp(lo, hi)
    return x


def _as_tree(parent, node_len):
    return np.asarray(parent, dtype=np.int32), np.asarray(node_len, dtype=np.int32)


def tiny_tree():
    """The explainer's 6-node example (Fig. 2): n0->{n1,n2}, n1->{n3,n4}, n2->{n5}."""
    return _as_tree([-1, 0, 0, 1, 1, 2], [16, 8, 8, 12, 12, 8])


def caterpillar_tree(p: int = 256, T: int = 40, delta: int = 64, a: int = 16):
    """Trunk t (t = 1..T) is node 2t-1 with delta tokens; its action leaf is node 2t with a tokens."""
    parent, lens = [-1], [p]
    for t in range(1, T + 1):
        parent.append(0 if t == 1 else 2 * (t - 1) - 1)
        lens.append(delta)
        parent.append(2 * t - 1)
        lens.append(a)
    return _as_tree(parent, lens)


def _relabel_subset(parent, lens, keep):
    """Keep the nodes listed in `keep` (ascending old ids); renumber them 0..m-1 in that order."""
    new_id = {old: i for i, old in enumerate(keep)}
    par = [(-1 if parent[old] < 0 else new_id[parent[old]]) for old in keep]
    return _as_tree(par, [lens[old] for old in keep])


def rollout_tree(seed: int = 0, root_len: int = 2048, depth: int = 5, branch=(2, 4),
                 median: float = 256.0, sigma: float = 0.8, lo: int = 16, hi: int = 4096,
                 budget: int = 32768):
    """Breadth-first random tree to `depth`, then the prefix subtree that fits `budget` tokens.

    Draw order (torch CPU generator seeded with `seed`): one randint per internal node in
    id order for its child count, then one batch of log-normal lengths for nodes 1..n-1.
    The kept prefix visits nodes depth-first (children in ascending id) and keeps each
    node while the running total stays within the budget; the first node that does not
    fit is cut to the remainder when that is at least `lo` tokens, and generation stops.
    """
    gen = torch.Generator().manual_seed(seed)
    parent, lvl = [-1], [0]
    i = 0
    while i < len(parent):
        if lvl[i] < depth:
            nc = int(torch.randint(branch[0], branch[1] + 1, (1,), generator=gen))
            for _ in range(nc):
                parent.append(i)
                lvl.append(lvl[i] + 1)
        i += 1
    n = len(parent)
    raw = _lognormal(gen, n - 1, median, sigma, lo, hi).long().tolist()
    lens = [root_len] + raw
    children = [[] for _ in range(n)]
    for c in range(1, n):
        children[parent[c]].append(c)
    keep, total = [], 0
    stack = [0]
    while stack:
        v = stack.pop()
        if total + lens[v] <= budget:
            keep.append(v)
            total += lens[v]
            stack.extend(reversed(children[v]))
        else:
            rem = budget - total
            if rem >= lo:
                lens[v] = rem
                keep.append(v)
            break
    return _relabel_subset(parent, lens, sorted(keep))


def ffd_pack(lengths, row_tokens):
    """First-fit-decreasing bin packing: items are placed longest first (ties: lower index), each
    into the lowest-numbered row whose remaining room holds it, a new row opened when none does.
    Returns, per row, the item indices in placement order."""
    lengths = np.asarray(lengths, dtype=np.int64)
    too_long = np.flatnonzero(lengths > row_tokens)
    if too_long.size:
        raise ValueError(f"item {int(too_long[0])} ({int(lengths[too_long[0]])} tokens) does not fit a row of "
                         f"{row_tokens}")
    placement = np.lexsort((np.arange(lengths.size), -lengths))     # primary key: length, descending
    room = np.zeros(0, dtype=np.int64)                              # remaining capacity per open row
    row_of = np.empty(lengths.size, dtype=np.int64)
    for item in placement:
        fits = np.flatnonzero(room >= lengths[item])
        if fits.size == 0:
            room = np.append(room, row_tokens)
            target = room.size - 1
        else:
            target = int(fits[0])
        room[target] -= lengths[item]
        row_of[item] = target
    return [[int(i) for i in placement if row_of[i] == r] for r in range(room.size)]


def forest_tree(seed: int = 0, row_tokens: int = 16384, n_rows: int = 8, median: float = 1024.0,
                p90: float = 4096.0, lo: int = 1, hi: int = 8192, draw: int = 4096):
    """Sequences packed FFD into rows; rows 0..n_rows-1 concatenated as a forest of root-only chains."""
    sigma = math.log(p90 / median) / 1.2815515655446004   # z of the 90th percentile
    gen = torch.Generator().manual_seed(seed)
    pool = _lognormal(gen, draw, median, sigma, lo, hi).long().tolist()
    lengths, total = [], 0
    for L in pool:
        if total >= n_rows * row_tokens:
            break
        lengths.append(int(L))
        total += int(L)
    rows = ffd_pack(lengths, row_tokens)[:n_rows]
    lens = [lengths[i] for r in rows for i in r]
    return _as_tree([-1] * len(lens), lens)


def large_tree(seed: int = 0, root_len: int = 8192, depth: int = 6, median: float = 1536.0,
               sigma: float = 0.8, lo: int = 16, total: int = 131072):
    """Full binary tree (heap ids: children of i are 2i+1, 2i+2) with lengths rescaled to `total`."""
    n = 2 ** (depth + 1) - 1
    parent = [-1] + [(c - 1) // 2 for c in range(1, n)]
    gen = torch.Generator().manual_seed(seed)
    raw = _lognormal(gen, n - 1, median, sigma, None, None).numpy()
    s = (total - root_len) / raw.sum()
    lens = [root_len] + [max(lo, int(round(x * s))) for x in raw]
    resid = total - sum(lens)
    last = n - 1                      # the right-most leaf is visited last depth-first
    lens[last] += resid
    if lens[last] < lo:
        raise ValueError("rescaled lengths leave the last node below the minimum")
    return _as_tree(parent, lens)


def random_tree(seed: int, n_nodes: int, max_len: int = 12, zero_prob: float = 0.0,
                n_roots: int = 1, min_len: int = 0):
    """Random recursive tree for property tests: node i > 0 picks a parent uniformly among 0..i-1
    (the first `n_roots` nodes are roots); lengths uniform in [min_len, max_len], zeroed with
    probability `zero_prob`.  The total is kept positive."""
    rng = np.random.default_rng(seed)
    parent = [-1] * n_roots + [int(rng.integers(0, i)) for i in range(n_roots, n_nodes)]
    lens = rng.integers(min_len, max_len + 1, size=n_nodes)
    if zero_prob > 0:
        lens[rng.random(n_nodes) < zero_prob] = 0
    if lens.sum() == 0:
        lens[0] = 1
    return _as_tree(parent, lens)


CONFIGS = {
    "tiny": dict(tree=tiny_tree, Hq=1, Hkv=1, d=64, uniform_grad=True, fp32_inputs=True),
    "caterpillar": dict(tree=caterpillar_tree, Hq=32, Hkv=8, d=128),
    "rollout32k": dict(tree=rollout_tree, Hq=32, Hkv=8, d=128),
    "forest": dict(tree=forest_tree, Hq=32, Hkv=8, d=128),
    "large128k": dict(tree=large_tree, Hq=32, Hkv=8, d=128),
}


def make_workload(name: str) -> Workload:
    c = CONFIGS[name]
    parent, node_len = c["tree"]()
    return Workload(name=name, parent=parent, node_len=node_len, Hq=c["Hq"], Hkv=c["Hkv"], d=c["d"],
                    uniform_grad=c.get("uniform_grad", False), fp32_inputs=c.get("fp32_inputs", False))
