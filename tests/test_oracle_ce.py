"""Pins of the cross-entropy oracle ("Tree Training 技术详解" sections 6.2, 6.3, 12) against
things other than itself:

* a chain is one sequence: torch's cross_entropy on the shifted logits/labels with
  ignore_index, summed, with autograd for dh and dW (fp64);
* any tree: the average over root-to-leaf paths of torch's cross_entropy of each path, each
  path built as its own sequence from parent pointers (not from the packed order), with
  autograd - the definition of section 6.2 computed by a library routine;
* brute force on the pairing: the logits gradient equals the sum over tokens u of
  (g_u/K)(softmax(z_p) - e_label_u) with p found by walking parent pointers;
* all labels ignored: zero loss and zero gradients; the sampled-row form agrees with the
  whole form.
"""
import numpy as np
import pytest
import torch

import oracle
from workloads import random_tree

IGN = -100


def _data(N, D, V, seed, ignore_frac=0.2):
    rng = np.random.default_rng(seed)
    h = rng.standard_normal((N, D))
    W = rng.standard_normal((V, D)) / np.sqrt(D)
    labels = rng.integers(0, V, size=N)
    labels[rng.random(N) < ignore_frac] = IGN
    return h, W, labels


def test_chain_equals_library_cross_entropy():
    node_len = np.array([4, 6, 5])
    parent = np.array([-1, 0, 1])
    N, D, V = int(node_len.sum()), 8, 11
    h, W, labels = _data(N, D, V, 1)
    r = oracle.ce_paths(parent, node_len, h, W, labels, IGN)
    ht = torch.tensor(h, requires_grad=True)
    Wt = torch.tensor(W, requires_grad=True)
    z = ht @ Wt.T
    loss = torch.nn.functional.cross_entropy(z[:-1], torch.tensor(labels[1:]), ignore_index=IGN, reduction="sum")
    loss.backward()
    assert abs(loss.item() - r["loss"]) < 1e-12
    assert np.abs(ht.grad.numpy() - r["dh"]).max() < 1e-12
    assert np.abs(Wt.grad.numpy() - r["dW"]).max() < 1e-12
    assert np.abs(torch.logsumexp(z, 1).detach().numpy() - r["lse"]).max() < 1e-12


def _root_paths_by_parent(parent, node_len, tok_start):
    """token sequences of every root-to-leaf path, built by walking parent pointers up from
    each leaf (children never consulted)"""
    n = len(parent)
    has_child = np.zeros(n, dtype=bool)
    for c in range(n):
        if parent[c] >= 0:
            has_child[parent[c]] = True
    seqs = []
    for leaf in np.nonzero(~has_child)[0]:
        chain, v = [], int(leaf)
        while v >= 0:
            chain.append(v)
            v = int(parent[v])
        toks = [t for v in reversed(chain) for t in range(tok_start[v], tok_start[v] + node_len[v])]
        seqs.append(np.array(toks, dtype=np.int64))
    return seqs


@pytest.mark.parametrize("seed", range(5))
def test_path_average_of_library_cross_entropy(seed):
    parent, node_len = random_tree(10 + seed, n_nodes=6 + 2 * seed, max_len=5, zero_prob=0.2, n_roots=1 + seed % 2)
    p = oracle.plan(parent, node_len)
    N, D, V = p["n_tokens"], 6, 9
    h, W, labels = _data(N, D, V, seed)
    r = oracle.ce_paths(parent, node_len, h, W, labels, IGN, p=p)
    seqs = _root_paths_by_parent(parent, node_len, p["tok_start"])
    assert len(seqs) == p["n_paths"]
    ht = torch.tensor(h, requires_grad=True)
    Wt = torch.tensor(W, requires_grad=True)
    z = ht @ Wt.T
    loss = 0
    for s in seqs:
        if len(s) > 1:
            loss = loss + torch.nn.functional.cross_entropy(z[s[:-1]], torch.tensor(labels[s[1:]]), ignore_index=IGN,
                                                            reduction="sum")
    loss = loss / len(seqs)
    loss.backward()
    assert abs(float(loss) - r["loss"]) < 1e-12
    assert np.abs(ht.grad.numpy() - r["dh"]).max() < 1e-12
    assert np.abs(Wt.grad.numpy() - r["dW"]).max() < 1e-12


@pytest.mark.parametrize("seed", range(4))
def test_logits_gradient_by_parent_walk(seed):
    parent, node_len = random_tree(30 + seed, n_nodes=10, max_len=4, zero_prob=0.3, n_roots=2)
    p = oracle.plan(parent, node_len)
    N, D, V = p["n_tokens"], 5, 7
    h, W, labels = _data(N, D, V, seed)
    r = oracle.ce_paths(parent, node_len, h, W, labels, IGN, p=p)
    z = h @ W.T
    sm = np.exp(z - z.max(1, keepdims=True))
    sm /= sm.sum(1, keepdims=True)
    dz = np.zeros_like(z)
    for u in range(N):
        v = p["tok_node"][u]
        if u > p["tok_start"][v]:
            t = u - 1
        else:
            a = parent[v]
            while a >= 0 and node_len[a] == 0:
                a = parent[a]
            if a < 0:
                continue
            t = p["tok_start"][a] + node_len[a] - 1
        if labels[u] == IGN:
            continue
        c = p["g"][u] / p["n_paths"]
        dz[t] += c * sm[t]
        dz[t, labels[u]] -= c
    assert np.abs(dz - r["dz"]).max() < 1e-12


def test_all_ignored_and_sampled_rows():
    parent, node_len = random_tree(3, n_nodes=9, max_len=6, zero_prob=0.1)
    p = oracle.plan(parent, node_len)
    N = p["n_tokens"]
    h, W, labels = _data(N, 4, 6, 3)
    r0 = oracle.ce_paths(parent, node_len, h, W, np.full(N, IGN), IGN, p=p)
    assert r0["loss"] == 0 and not r0["dh"].any() and not r0["dW"].any()
    r = oracle.ce_paths(parent, node_len, h, W, labels, IGN, p=p)
    rows = [0, N // 2, N - 1]
    s = oracle.ce_rows(parent, node_len, h, W, labels, rows, IGN, p=p)
    assert np.abs(s["lse"] - r["lse"][rows]).max() < 1e-12
    assert np.abs(s["dh"] - r["dh"][rows]).max() < 1e-12
    every = oracle.ce_rows(parent, node_len, h, W, labels, range(N), IGN, p=p)
    assert abs(every["loss"].sum() - r["loss"]) < 1e-12
