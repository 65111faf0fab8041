"""Pins of the partition bookkeeping and of the gateway decomposition ("Tree Training 技术详解",
section 8.2), on the CPU oracle alone:

* a partitioned tree's tokens are the whole tree's, each once; child positions continue the
  gateway's (pos = A + position inside the child partition);
* a child partition needs nothing but the gateway: the oracle on the tree "root-to-cut path +
  the child's subtree" gives the whole tree's O and LSE at the child's tokens;
* the relay is exact: gradients are linear in dO, so the whole tree's dK, dV at the parent
  partition's tokens are the sum of the run with the loss on parent tokens only and the run
  with the loss on child tokens only (the child part reaches the ancestors through the gateway).
"""
import numpy as np
import pytest
import torch

import oracle
from _gateway import gateway_tree, partition


def _tensors(N, Hq, Hkv, d, seed=1):
    g = torch.Generator().manual_seed(seed)
    mk = lambda h: torch.randn(N, h, d, generator=g).to(torch.bfloat16)
    return dict(q=mk(Hq), k=mk(Hkv), v=mk(Hkv), u=mk(Hq))


CASES = [(0, [37, 20, 11], 30, 14), (1, [64, 64], 25, 10), (2, [5], 40, 8)]


@pytest.mark.parametrize("seed,gw,max_len,n_extra", CASES)
def test_partition_bookkeeping(seed, gw, max_len, n_extra):
    parent, lens, cut = gateway_tree(seed, gw, branch_len=23, n_extra=n_extra, max_len=max_len)
    P = partition(parent, lens, cut)
    full = P["full"]
    toks = np.concatenate([P["parent"].tokens] + [c.tokens for c in P["children"]])
    assert sorted(toks.tolist()) == list(range(full["n_tokens"]))
    assert P["A"] == sum(gw)
    assert np.array_equal(full["pos"][P["gw_tokens"]], np.arange(P["A"]))      # the path, root first
    assert np.array_equal(P["parent"].tokens[P["gw_rows"]], P["gw_tokens"])
    for ch in P["children"]:
        sub = oracle.plan(ch.parent, ch.node_len)
        assert np.array_equal(full["pos"][ch.tokens], sub["pos"] + P["A"])
    sub = oracle.plan(P["parent"].parent, P["parent"].node_len)
    assert np.array_equal(full["pos"][P["parent"].tokens], sub["pos"])


@pytest.mark.parametrize("seed,gw,max_len,n_extra", CASES)
def test_child_sees_only_the_gateway(seed, gw, max_len, n_extra):
    parent, lens, cut = gateway_tree(seed, gw, branch_len=23, n_extra=n_extra, max_len=max_len)
    P = partition(parent, lens, cut)
    N = P["full"]["n_tokens"]
    t = _tensors(N, 2, 1, 16)
    ref = oracle.attention_nodes(parent, lens, t["q"], t["k"], t["v"], t["u"], heads=[0, 1], theta=10000.0)
    for ch in P["children"]:
        # the tree "path root..cut as a chain, then this child's subtree"
        path_nodes = list(range(len(gw)))
        nodes = path_nodes + [int(v) for v in ch.nodes]
        remap = {v: i for i, v in enumerate(nodes)}
        par = np.array([-1 if v == 0 else remap[int(parent[v])] for v in nodes])
        ln = np.asarray(lens)[nodes]
        toks = np.concatenate([P["gw_tokens"], ch.tokens])
        sub = {k: t[k][toks].contiguous() for k in t}
        r = oracle.attention_nodes(par, ln, sub["q"], sub["k"], sub["v"], sub["u"], heads=[0, 1], theta=10000.0)
        A = P["A"]
        assert np.abs(r["o"][A:] - ref["o"][ch.tokens]).max() < 1e-12
        assert np.abs(r["lse"][:, A:] - ref["lse"][:, ch.tokens]).max() < 1e-12


@pytest.mark.parametrize("seed,gw,max_len,n_extra", CASES[:2])
def test_relay_is_the_sum_of_the_partition_losses(seed, gw, max_len, n_extra):
    parent, lens, cut = gateway_tree(seed, gw, branch_len=23, n_extra=n_extra, max_len=max_len)
    P = partition(parent, lens, cut)
    N = P["full"]["n_tokens"]
    t = _tensors(N, 2, 1, 16, seed=7)
    run = lambda u: oracle.attention_nodes(parent, lens, t["q"], t["k"], t["v"], u, heads=[0, 1], theta=10000.0)
    whole = run(t["u"])
    child_tok = np.concatenate([c.tokens for c in P["children"]])
    u_par, u_chi = t["u"].clone(), t["u"].clone()
    u_par[torch.as_tensor(child_tok)] = 0
    u_chi[torch.as_tensor(P["parent"].tokens)] = 0
    a, b = run(u_par), run(u_chi)
    for name in ("dq", "dk", "dv"):
        assert np.abs(a[name] + b[name] - whole[name]).max() < 1e-9 * max(1.0, np.abs(whole[name]).max())
    # the child loss reaches parent-partition keys only through the gateway (the path)
    off_path = np.setdiff1d(P["parent"].tokens, P["gw_tokens"])
    assert np.abs(b["dk"][off_path]).max() == 0 and np.abs(b["dv"][off_path]).max() == 0


@pytest.mark.parametrize("seed,gw,max_len,n_extra", CASES)
def test_library_partitioner_matches_the_test_bookkeeping(seed, gw, max_len, n_extra):
    """The package's host partitioner (own depth-first packing) against the oracle-plan-based
    bookkeeping of these tests."""
    from tree_masked_attention_plan_gb300.partition import partition_tree
    parent, lens, cut = gateway_tree(seed, gw, branch_len=23, n_extra=n_extra, max_len=max_len)
    P, Q = partition(parent, lens, cut), partition_tree(parent, lens, cut)
    assert P["A"] == Q["A"]
    assert np.array_equal(P["gw_tokens"], Q["gw_tokens"]) and np.array_equal(P["gw_rows"], Q["gw_rows"])
    kids = [c for c in P["children"] if c.node_len.sum() > 0]
    assert len(kids) == len(Q["children"])
    for a, b in zip([P["parent"]] + kids, [Q["parent"]] + Q["children"]):
        assert np.array_equal(a.parent, b.parent) and np.array_equal(a.node_len, b.node_len)
        assert np.array_equal(a.tokens, b.tokens) and a.pos_offset == b.pos_offset
