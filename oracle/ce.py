"""Oracle for the tree's weighted next-token cross-entropy (TEST INFRASTRUCTURE ONLY),
"Tree Training 技术详解" sections 6.2, 6.3 and 12 (the loss construction).

Definition (section 6.2: the tree loss is the average over root-to-leaf paths of each path's
own loss).  Every path is an ordinary token sequence; on it, the logits of each token predict
the label of the next token (the packed-sequence shift of section 12), and positions whose
label is the ignore index carry no loss (section 6.3):

    L = (1/K) sum_paths sum_{consecutive (t, u) on the path, label_u != ignore}
            [ logsumexp(z_t) - z_t[label_u] ],        z_t = W h_t  (logits row of token t).

A pair (t, u) lies on exactly g_u paths, so this equals sum_u (g_u/K) * CE(z_{prev(u)}, label_u)
with prev(u) the token before u on its root path - which in packed order is u-1 inside a node
and the parent's last token for a node's first token (a node's last token is thus paired with
the first token of every child).  The first token of a root predicts nothing.

Gradients: dz_t = (1/K) sum over its pairs (softmax(z_t) - onehot(label_u)),
dh = dz W, dW = dz^T h (h [N, D], W [V, D]).
"""
from __future__ import annotations

import numpy as np

from .tree import plan as _plan


def _path_tokens(p, node_len, path):
    return np.concatenate([np.arange(p["tok_start"][v], p["tok_start"][v] + node_len[v]) for v in path]
                          ).astype(np.int64)


def _pairs(p, node_len, labels, ignore_index):
    """(t, u) for every consecutive pair on every path with a supervised u, with repetition
    (a pair on g_u paths appears g_u times)."""
    out = []
    for path in p["paths"]:
        toks = _path_tokens(p, node_len, path)
        for i in range(len(toks) - 1):
            u = int(toks[i + 1])
            if labels[u] != ignore_index:
                out.append((int(toks[i]), u))
    return out


def _lse(z):
    m = z.max(axis=-1, keepdims=True)
    return (m + np.log(np.exp(z - m).sum(axis=-1, keepdims=True)))[..., 0]


def ce_paths(parent, node_len, h, W, labels, ignore_index=-100, p=None):
    """h [N, D], W [V, D], labels [N] (ints).  Returns dict loss, lse [N], dz [N, V], dh [N, D],
    dW [V, D] in fp64."""
    node_len = np.asarray(node_len, dtype=np.int64)
    p = p if p is not None else _plan(parent, node_len)
    h = np.asarray(h, dtype=np.float64)
    W = np.asarray(W, dtype=np.float64)
    labels = np.asarray(labels, dtype=np.int64)
    z = h @ W.T
    lse = _lse(z)
    K = p["n_paths"]
    dz = np.zeros_like(z)
    loss = 0.0
    for t, u in _pairs(p, node_len, labels, ignore_index):
        y = labels[u]
        loss += (lse[t] - z[t, y]) / K
        dz[t] += np.exp(z[t] - lse[t]) / K
        dz[t, y] -= 1.0 / K
    return dict(loss=loss, lse=lse, dz=dz, dh=dz @ W, dW=dz.T @ h)


def ce_rows(parent, node_len, h, W, labels, rows, ignore_index=-100, p=None):
    """The same definition restricted to the logits rows `rows`: their logsumexp, their
    pairs' loss, and their rows of dh.  W may be large: only len(rows) logits rows are formed."""
    node_len = np.asarray(node_len, dtype=np.int64)
    p = p if p is not None else _plan(parent, node_len)
    labels = np.asarray(labels, dtype=np.int64)
    rows = [int(r) for r in rows]
    W = np.asarray(W, dtype=np.float64)
    z = np.asarray(h, dtype=np.float64)[rows] @ W.T
    lse = _lse(z)
    K = p["n_paths"]
    where = {t: i for i, t in enumerate(rows)}
    dz = np.zeros_like(z)
    loss = np.zeros(len(rows))
    for t, u in _pairs(p, node_len, labels, ignore_index):
        if t in where:
            i, y = where[t], labels[u]
            loss[i] += (lse[i] - z[i, y]) / K
            dz[i] += np.exp(z[i] - lse[i]) / K
            dz[i, y] -= 1.0 / K
    return dict(lse=lse, loss=loss, dh=dz @ W)
