"""RoPE and attention forward on the GPU against the fp64 oracle.

Tolerances: O and LSE max-abs <= 2e-2; RoPE outputs within bf16 output rounding plus the
fp32 angle (|delta| <= 1e-2 (|x_c| + |x_c+d/2|) + 1e-3)."""
import numpy as np
import pytest
import torch

import oracle
import tree_masked_attention_plan_gb300 as tam
from workloads import make_tensors, make_workload, random_tree
from workloads.trees import Workload

from _gpu import O_TOL, compare_fwd, f64, oracle_ref, run_gpu

pytestmark = pytest.mark.gpu


def _wl(parent, node_len, Hq, Hkv, d, name="rand"):
    return Workload(name=name, parent=np.asarray(parent, np.int32), node_len=np.asarray(node_len, np.int32),
                    Hq=Hq, Hkv=Hkv, d=d)


SMALL = [("ragged_d128", random_tree(7, 12, max_len=90), 4, 2, 128),
         ("ragged_d64", random_tree(8, 20, max_len=60, zero_prob=0.1), 2, 2, 64),
         ("forest_d128", random_tree(9, 9, max_len=150, n_roots=3), 4, 1, 128),
         ("deep_d128", random_tree(10, 40, max_len=25), 2, 1, 128),
         ("one_token", (np.array([-1]), np.array([1])), 2, 1, 128)]


@pytest.mark.parametrize("name,tree,Hq,Hkv,d", SMALL, ids=[s[0] for s in SMALL])
def test_fwd_small_trees(name, tree, Hq, Hkv, d):
    wl = _wl(*tree, Hq, Hkv, d)
    t = make_tensors(wl)
    g = run_gpu(wl.parent, wl.node_len, t, backward=False)
    ref = oracle_ref(wl.parent, wl.node_len, t, heads=range(Hq))
    eo, el = compare_fwd(g, ref, range(Hq), wl.n_tokens)
    print(f"{name}: N={wl.n_tokens} O err {eo:.3e} LSE err {el:.3e}")
    assert eo <= O_TOL and el <= O_TOL


def test_rope_matches_oracle():
    wl = make_workload("caterpillar")
    t = make_tensors(wl)
    p = oracle.plan(wl.parent, wl.node_len)
    g = run_gpu(wl.parent, wl.node_len, t, backward=False)
    for key, src in (("qr", "q"), ("kr", "k")):
        x = f64(t[src])
        ref = oracle.rope(x, p["pos"], 10000.0)
        got = f64(g[key])
        half = x.shape[-1] // 2
        bound = 1e-2 * (np.abs(x) + np.abs(np.concatenate([x[..., half:], x[..., :half]], -1))) + 1e-3
        assert np.all(np.abs(got - ref) <= bound), key


def test_fwd_tiny_example():
    wl = make_workload("tiny")
    t = make_tensors(wl)
    g = run_gpu(wl.parent, wl.node_len, t, backward=False)
    ref = oracle_ref(wl.parent, wl.node_len, t, heads=[0])
    eo, el = compare_fwd(g, ref, [0], wl.n_tokens)
    print(f"tiny: O err {eo:.3e} LSE err {el:.3e}")
    assert eo <= O_TOL and el <= O_TOL


@pytest.mark.parametrize("name,heads", [("caterpillar", [0, 1, 2, 3, 28, 29, 30, 31]),
                                        ("rollout32k", [0, 1, 2, 3, 31]),
                                        ("forest", [0, 5]),
                                        ("large128k", [0])])
def test_fwd_configs(name, heads):
    """Full-size workloads; the oracle evaluates the listed q heads (per-node tree-mask form)."""
    wl = make_workload(name)
    t = make_tensors(wl)
    g = run_gpu(wl.parent, wl.node_len, t, backward=False)
    ref = oracle_ref(wl.parent, wl.node_len, t, heads=heads, use_nodes=True)
    eo, el = compare_fwd(g, ref, heads, wl.n_tokens)
    print(f"{name}: O err {eo:.3e} LSE err {el:.3e}")
    assert eo <= O_TOL and el <= O_TOL


def test_fwd_leak_sibling_bitwise():
    """Section 14.2 leak test on the GPU: changing a sibling branch leaves this branch's O and
    LSE bit-for-bit unchanged; changing an ancestor changes every descendant."""
    wl = make_workload("tiny")
    wl = _wl(wl.parent, wl.node_len * 20, 4, 2, 128)       # 1280 tokens, 10 tiles
    t = make_tensors(wl)
    p = oracle.plan(wl.parent, wl.node_len)
    base = run_gpu(wl.parent, wl.node_len, t, backward=False)

    def toks(nodes):
        return np.concatenate([np.arange(p["tok_start"][x], p["tok_start"][x] + wl.node_len[x]) for x in nodes])

    n2_branch = torch.from_numpy(toks([2, 5]))
    t2 = dict(t)
    for key in ("q", "k", "v"):
        t2[key] = t[key].clone()
        t2[key][torch.from_numpy(toks([1, 3, 4]))] *= -2
    pert = run_gpu(wl.parent, wl.node_len, t2, backward=False)
    assert torch.equal(pert["o"][n2_branch.cuda()], base["o"][n2_branch.cuda()])
    assert torch.equal(pert["lse"][:, n2_branch.cuda()], base["lse"][:, n2_branch.cuda()])
    t3 = dict(t)
    t3["v"] = t["v"].clone()
    t3["v"][0] += 1
    pert = run_gpu(wl.parent, wl.node_len, t3, backward=False)
    desc = torch.from_numpy(toks([1, 2, 3, 4, 5])).cuda()
    assert torch.all((pert["o"][desc] - base["o"][desc]).abs().amax(dim=(1, 2)) > 0)


def test_timeout_selftest():
    st = tam.new_status()
    tam.tree_selftest_timeout(st, 2_000_000)
    torch.cuda.synchronize()
    assert st.item() == -5
    # the context is still usable afterwards
    x = torch.ones(4, device="cuda") * 2
    assert x.sum().item() == 8
