"""Oracle for the hybrid-layer primitives (TEST INFRASTRUCTURE ONLY), "Tree Training 技术详解"
section 9: what a causal convolution and a recurrent state see when a tree is trained as its
root-to-leaf paths.

* ``conv_paths``: the definition of the tree's causal depthwise convolution.  Every root-to-leaf
  path is an ordinary sequence; the convolution runs on it with zero padding before the root
  (section 9.2: a child's context is its parent's last tokens, not the sibling tokens next to
  it in the packed order); a token's output is the same on every path through it.  The
  gradients are those of the tree loss written as an average over paths,
  L = (1/K) sum_paths sum_{t in path} <U_t, y_t>, scatter-added over the paths (section 6.2).
* ``route_states`` / ``route_states_bwd``: section 9.1's h_c(0) = h_parent(c)(end), with the
  parent taken as the nearest ancestor holding tokens (a node without tokens passes its
  input state through), and the transpose of that gather for the backward.
"""
from __future__ import annotations

import numpy as np

from .tree import plan as _plan


def _path_tokens(p, node_len, path):
    return np.concatenate([np.arange(p["tok_start"][v], p["tok_start"][v] + node_len[v]) for v in path]
                          ).astype(np.int64)


def conv_paths(parent, node_len, x, w, bias=None, u=None, p=None):
    """x [N, C], w [K, C] (w[k] multiplies the input k steps back), bias [C]; u [N, C] the
    upstream gradient of the tree loss.  Returns dict y [N, C] and, with u, dx, dw, db (fp64)."""
    node_len = np.asarray(node_len, dtype=np.int64)
    p = p if p is not None else _plan(parent, node_len)
    x = np.asarray(x, dtype=np.float64)
    w = np.asarray(w, dtype=np.float64)
    N, C = x.shape
    K = w.shape[0]
    b = np.zeros(C) if bias is None else np.asarray(bias, dtype=np.float64)
    y = np.full((N, C), np.nan)
    grads = u is not None
    if grads:
        u = np.asarray(u, dtype=np.float64)
        dx, dw, db = np.zeros((N, C)), np.zeros((K, C)), np.zeros(C)
    n_paths = p["n_paths"]
    for path in p["paths"]:
        toks = _path_tokens(p, node_len, path)
        X = x[toks]
        L = len(toks)
        Y = np.tile(b, (L, 1))
        for k in range(min(K, L)):                   # taps reaching before the root see zeros
            Y[k:] += w[k] * X[:L - k]
        seen = ~np.isnan(y[toks])
        assert np.allclose(y[toks][seen], Y[seen], rtol=0, atol=1e-9), "output differs between paths"
        y[toks] = Y
        if grads:
            G = u[toks] / n_paths                      # dL/dY on this path
            dX = np.zeros_like(X)
            for k in range(min(K, L)):
                dX[:L - k] += w[k] * G[k:]
                dw[k] += (X[:L - k] * G[k:]).sum(axis=0)
            db += G.sum(axis=0)
            np.add.at(dx, toks, dX)
    out = dict(y=y)
    if grads:
        out.update(dx=dx, dw=dw, db=db)
    return out


def _token_ancestor(parent, node_len, v):
    a = parent[v]
    while a >= 0 and node_len[a] == 0:
        a = parent[a]
    return a


def route_states(parent, node_len, final_states):
    """init[v] = final[a], a the nearest ancestor of v that holds tokens; zeros if none."""
    parent = np.asarray(parent, dtype=np.int64)
    node_len = np.asarray(node_len, dtype=np.int64)
    fin = np.asarray(final_states, dtype=np.float64)
    init = np.zeros_like(fin)
    for v in range(len(parent)):
        a = _token_ancestor(parent, node_len, v)
        if a >= 0:
            init[v] = fin[a]
    return init


def route_states_bwd(parent, node_len, d_init):
    """The transpose: d_final[a] = sum of d_init over the nodes whose state comes from a."""
    parent = np.asarray(parent, dtype=np.int64)
    node_len = np.asarray(node_len, dtype=np.int64)
    d_init = np.asarray(d_init, dtype=np.float64)
    d_fin = np.zeros_like(d_init)
    for v in range(len(parent)):
        a = _token_ancestor(parent, node_len, v)
        if a >= 0:
            d_fin[a] += d_init[v]
    return d_fin
