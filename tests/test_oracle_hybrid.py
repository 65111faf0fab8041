"""Pins of the hybrid-layer oracle ("Tree Training 技术详解", section 9) against things other
than itself:

* a chain is one sequence: the tree convolution equals torch's conv1d with left zero padding
  (forward, and its autograd gradients with the per-path loss);
* brute force: each token's k-th predecessor found by walking parent pointers (a different
  traversal from the path expansion) gives the same outputs, on trees with zero-length nodes
  and several roots;
* central finite differences of the tree loss for dx, dw, db;
* state routing composed with a toy linear recurrence: scanning each node from its routed
  initial state gives, token for token, the state of the sequential scan along every
  root-to-leaf path (section 9.1), and the routed backward is the transpose of the gather.
"""
import numpy as np
import pytest
import torch

import oracle
from workloads import random_tree


def _rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


def test_chain_equals_library_conv1d():
    lens = np.array([5, 7, 3, 9])
    parent = np.array([-1, 0, 1, 2])
    N, C, K = int(lens.sum()), 6, 4
    x, w, b, u = _rand((N, C), 1), _rand((K, C), 2), _rand(C, 3), _rand((N, C), 4)
    r = oracle.conv_paths(parent, lens, x, w, b, u)
    xt = torch.tensor(x.T[None], dtype=torch.float64, requires_grad=True)
    # torch correlates: out[i] = sum_j weight[j] * in[i + j - (K-1)] with K-1 zeros in front,
    # so weight[j] = w[K-1-j] (w[k] multiplies the input k steps back)
    wt = torch.tensor(w[::-1].T.copy()[:, None, :], dtype=torch.float64, requires_grad=True)
    bt = torch.tensor(b, dtype=torch.float64, requires_grad=True)
    y = torch.nn.functional.conv1d(torch.nn.functional.pad(xt, (K - 1, 0)), wt, bt, groups=C)
    assert np.abs(y[0].T.detach().numpy() - r["y"]).max() < 1e-12
    (y[0].T * torch.tensor(u)).sum().backward()          # one path: K_paths = 1
    assert np.abs(xt.grad[0].T.numpy() - r["dx"]).max() < 1e-12
    assert np.abs(wt.grad[:, 0].flip(-1).T.numpy() - r["dw"]).max() < 1e-12
    assert np.abs(bt.grad.numpy() - r["db"]).max() < 1e-12


def _prev_by_parent_walk(parent, lens, tok_start, tok_node, t, k):
    j = t
    for _ in range(k):
        v = tok_node[j]
        if j > tok_start[v]:
            j -= 1
            continue
        a = parent[v]
        while a >= 0 and lens[a] == 0:
            a = parent[a]
        if a < 0:
            return -1
        j = tok_start[a] + lens[a] - 1
    return j


@pytest.mark.parametrize("seed", range(6))
def test_brute_force_predecessors(seed):
    parent, lens = random_tree(40 + seed, n_nodes=6 + 3 * seed, max_len=5, zero_prob=0.25, n_roots=1 + seed % 3)
    p = oracle.plan(parent, lens)
    N, C, K = p["n_tokens"], 3, 1 + seed % 6
    x, w, b = _rand((N, C), seed), _rand((K, C), seed + 1), _rand(C, seed + 2)
    r = oracle.conv_paths(parent, lens, x, w, b)
    for t in range(N):
        expect = b.copy()
        for k in range(K):
            j = _prev_by_parent_walk(parent, lens, p["tok_start"], p["tok_node"], t, k)
            if j >= 0:
                expect += w[k] * x[j]
        assert np.abs(r["y"][t] - expect).max() < 1e-12, t


def test_finite_differences():
    parent, lens = random_tree(7, n_nodes=7, max_len=4, zero_prob=0.2)
    p = oracle.plan(parent, lens)
    N, C, K = p["n_tokens"], 2, 3
    x, w, b, u = _rand((N, C), 11), _rand((K, C), 12), _rand(C, 13), _rand((N, C), 14)
    g = p["g"].astype(np.float64) / p["n_paths"]

    def loss(x_, w_, b_):
        return float((oracle.conv_paths(parent, lens, x_, w_, b_)["y"] * u * g[:, None]).sum())

    r = oracle.conv_paths(parent, lens, x, w, b, u)
    eps = 1e-6
    for name, arr in (("dx", x), ("dw", w), ("db", b)):
        num = np.zeros_like(arr)
        for idx in np.ndindex(arr.shape):
            hi, lo = arr.copy(), arr.copy()
            hi[idx] += eps
            lo[idx] -= eps
            args_hi = [hi if a is arr else a for a in (x, w, b)]
            args_lo = [lo if a is arr else a for a in (x, w, b)]
            num[idx] = (loss(*args_hi) - loss(*args_lo)) / (2 * eps)
        assert np.abs(num - r[name]).max() < 1e-6 * max(1.0, np.abs(num).max()), name


@pytest.mark.parametrize("seed", range(4))
def test_routed_scan_equals_path_scan(seed):
    """h_t = a * h_{t-1} + x_t (per channel): per-node scans started from the routed final
    state of the token-holding parent reproduce the sequential scan along every path."""
    parent, lens = random_tree(60 + seed, n_nodes=8 + 2 * seed, max_len=4, zero_prob=0.3, n_roots=1 + seed % 2)
    p = oracle.plan(parent, lens)
    n, N, S = len(parent), p["n_tokens"], 4
    a = np.abs(_rand(S, seed)) * 0.5
    x = _rand((N, S), seed + 5)
    # node-by-node in preorder: scan each node from its routed initial state
    fin = np.zeros((n, S))
    h_tok = np.zeros((N, S))
    for v in p["order"]:
        init = oracle.route_states(parent, lens, fin)[v]
        h = init.copy()
        for t in range(p["tok_start"][v], p["tok_start"][v] + lens[v]):
            h = a * h + x[t]
            h_tok[t] = h
        fin[v] = h if lens[v] > 0 else init
    for path in p["paths"]:
        h = np.zeros(S)
        for v in path:
            for t in range(p["tok_start"][v], p["tok_start"][v] + lens[v]):
                h = a * h + x[t]
                assert np.abs(h - h_tok[t]).max() < 1e-12


@pytest.mark.parametrize("seed", range(3))
def test_route_backward_is_the_transpose(seed):
    parent, lens = random_tree(80 + seed, n_nodes=12, max_len=3, zero_prob=0.3, n_roots=2)
    n, S = len(parent), 4
    f, d = _rand((n, S), seed), _rand((n, S), seed + 9)
    lhs = (oracle.route_states(parent, lens, f) * d).sum()
    rhs = (f * oracle.route_states_bwd(parent, lens, d)).sum()
    assert abs(lhs - rhs) < 1e-12
