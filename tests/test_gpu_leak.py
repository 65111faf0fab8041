"""Leak and permutation properties of the tree mask on the GPU ("Tree Training 技术详解",
section 14.2), on the Fig. 2 tree with every node 20x longer (1280 tokens, 10 tiles, so node
boundaries fall inside tiles):

* a future child: perturbing n3's inputs leaves the output of every other node (its ancestors
  n0, n1, its sibling n4 and the other branch) bit for bit unchanged;
* a sibling branch: perturbing n1's branch leaves n2's branch unchanged bit for bit, in the
  forward (O, LSE) and in the gradients of n2's branch keys (dK, dV, reduced on chip in a
  fixed order, where the masked pairs contribute exact zeros);
* an ancestor: perturbing one root token changes every descendant's output;
* sibling order: relabelling siblings (which reorders the depth-first packing, so tokens land
  in other tiles) gives the same per-token results within the target tolerances.
"""
import numpy as np
import pytest
import torch

import oracle
from workloads import make_tensors, tiny_tree
from workloads.trees import Workload

from _gpu import GRAD_TOL, O_TOL, f64, rel_err, run_gpu

pytestmark = pytest.mark.gpu


def _setup():
    parent, lens = tiny_tree()
    lens = lens * 20
    wl = Workload(name="tiny20", parent=parent, node_len=lens, Hq=4, Hkv=2, d=128)
    return wl, make_tensors(wl), oracle.plan(wl.parent, wl.node_len)


def _toks(p, lens, nodes):
    return torch.from_numpy(np.concatenate([np.arange(p["tok_start"][x], p["tok_start"][x] + lens[x])
                                            for x in nodes]))


def _perturb(t, tok):
    t2 = dict(t)
    for key, f in (("q", lambda x: x + 1), ("k", lambda x: x * -2), ("v", lambda x: x * 3)):
        t2[key] = t[key].clone()
        t2[key][tok] = f(t[key][tok].float()).to(torch.bfloat16)
    return t2


def test_future_child_leaves_other_nodes_bitwise():
    wl, t, p = _setup()
    base = run_gpu(wl.parent, wl.node_len, t)
    pert = run_gpu(wl.parent, wl.node_len, _perturb(t, _toks(p, wl.node_len, [3])))
    keep = _toks(p, wl.node_len, [0, 1, 4, 2, 5]).cuda()
    assert torch.equal(pert["o"][keep], base["o"][keep])
    assert torch.equal(pert["lse"][:, keep], base["lse"][:, keep])
    n3 = _toks(p, wl.node_len, [3]).cuda()
    assert not torch.equal(pert["o"][n3], base["o"][n3])


def test_sibling_branch_bitwise_forward_and_key_gradients():
    wl, t, p = _setup()
    base = run_gpu(wl.parent, wl.node_len, t)
    pert = run_gpu(wl.parent, wl.node_len, _perturb(t, _toks(p, wl.node_len, [1, 3, 4])))
    br2 = _toks(p, wl.node_len, [2, 5]).cuda()
    assert torch.equal(pert["o"][br2], base["o"][br2])
    assert torch.equal(pert["lse"][:, br2], base["lse"][:, br2])
    assert torch.equal(pert["dk"][br2], base["dk"][br2])
    assert torch.equal(pert["dv"][br2], base["dv"][br2])
    # dQ goes through fp32 reduce-adds in arbitrary order: equal within rounding only
    assert rel_err(f64(pert["dq"][br2]), f64(base["dq"][br2])) < 1e-2


def test_ancestor_changes_every_descendant():
    wl, t, p = _setup()
    base = run_gpu(wl.parent, wl.node_len, t, backward=False)
    pert = run_gpu(wl.parent, wl.node_len, _perturb(t, torch.tensor([0])), backward=False)
    desc = _toks(p, wl.node_len, [1, 2, 3, 4, 5]).cuda()
    assert torch.all((pert["o"][desc].float() - base["o"][desc].float()).abs().amax(dim=(1, 2)) > 0)


def test_sibling_order_permutation():
    wl, t, p1 = _setup()
    perm = np.array([0, 2, 1, 5, 4, 3])            # new id of old node: n2's branch first in DFS
    inv = np.argsort(perm)
    parent2 = np.array([-1 if wl.parent[inv[i]] < 0 else perm[wl.parent[inv[i]]] for i in range(6)])
    len2 = wl.node_len[inv]
    p2 = oracle.plan(parent2, len2)
    N = wl.n_tokens
    tmap = np.empty(N, dtype=np.int64)             # old packed index -> new packed index
    for x in range(6):
        s1, s2 = p1["tok_start"][x], p2["tok_start"][perm[x]]
        tmap[s1:s1 + wl.node_len[x]] = np.arange(s2, s2 + wl.node_len[x])
    assert not np.array_equal(tmap, np.arange(N))
    t2 = {}
    for key in ("q", "k", "v", "u"):
        t2[key] = torch.empty_like(t[key])
        t2[key][torch.from_numpy(tmap)] = t[key]
    a = run_gpu(wl.parent, wl.node_len, t)
    b = run_gpu(parent2, len2, t2)
    ref = oracle.attention_paths(wl.parent, wl.node_len, t["q"], t["k"], t["v"], t["u"], p=p1)
    idx = torch.from_numpy(tmap).cuda()
    for key in ("o", "dq", "dk", "dv"):
        got_b = f64(b[key][idx])
        tol = O_TOL if key == "o" else GRAD_TOL
        err_ref = np.abs(got_b - ref[key]).max() if key == "o" else rel_err(got_b, ref[key])
        err_ab = np.abs(got_b - f64(a[key])).max() if key == "o" else rel_err(got_b, f64(a[key]))
        print(f"{key}: permuted vs oracle {err_ref:.2e}, permuted vs original layout {err_ab:.2e}")
        assert err_ref <= tol and err_ab <= tol
    lse_b = f64(b["lse"])[:, tmap]
    assert np.abs(lse_b - ref["lse"]).max() <= O_TOL
