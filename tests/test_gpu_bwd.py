"""Backward on the GPU against the fp64 oracle: dQ, dK, dV within 5e-2 of max|reference|.

The oracle's gradient is that of the per-path average loss (1/K) sum_k sum_{t in p_k}
<U_t, O_t>; the GPU path is fed dO_t = (g_t/K) U_t from tree_apply_weights.  Equality of the
two is the explainer's section 6.2 identity."""
import numpy as np
import pytest
import torch

import oracle
import tree_masked_attention_plan_gb300 as tam
from workloads import make_tensors, make_workload, random_tree
from workloads.trees import Workload

from _gpu import GRAD_TOL, O_TOL, compare_bwd, compare_fwd, f64, oracle_ref, run_gpu

pytestmark = pytest.mark.gpu


def _wl(parent, node_len, Hq, Hkv, d):
    return Workload(name="t", parent=np.asarray(parent, np.int32), node_len=np.asarray(node_len, np.int32),
                    Hq=Hq, Hkv=Hkv, d=d)


SMALL = [("ragged_d128", random_tree(7, 12, max_len=90), 4, 2, 128),
         ("ragged_d64", random_tree(8, 20, max_len=60, zero_prob=0.1), 2, 2, 64),
         ("forest_d128", random_tree(9, 9, max_len=150, n_roots=3), 4, 1, 128),
         ("deep_d128", random_tree(10, 40, max_len=25), 2, 1, 128),
         ("one_token", (np.array([-1]), np.array([1])), 2, 1, 128)]


@pytest.mark.parametrize("name,tree,Hq,Hkv,d", SMALL, ids=[s[0] for s in SMALL])
def test_bwd_small_trees(name, tree, Hq, Hkv, d):
    wl = _wl(*tree, Hq, Hkv, d)
    t = make_tensors(wl)
    g = run_gpu(wl.parent, wl.node_len, t)
    ref = oracle_ref(wl.parent, wl.node_len, t, heads=range(Hq))
    e = compare_bwd(g, ref, range(Hq), Hq, Hkv)
    print(f"{name}: N={wl.n_tokens} grad rel errs {e}")
    assert max(e.values()) <= GRAD_TOL


def test_bwd_tiny_example():
    wl = make_workload("tiny")
    t = make_tensors(wl)
    g = run_gpu(wl.parent, wl.node_len, t)
    ref = oracle_ref(wl.parent, wl.node_len, t, heads=[0])
    e = compare_bwd(g, ref, [0], 1, 1)
    print(f"tiny grads {e}")
    assert max(e.values()) <= GRAD_TOL


@pytest.mark.parametrize("name,heads", [("caterpillar", [0, 1, 2, 3, 28, 29, 30, 31]),
                                        ("rollout32k", [0, 1, 2, 3]),
                                        ("forest", [4, 5, 6, 7]),
                                        ("large128k", [28, 29, 30, 31])])
def test_bwd_configs(name, heads):
    """Full-size workloads in the bench's launch configuration; the oracle evaluates one or two
    whole kv-head groups (every q head reading those kv heads) with the per-node tree-mask form."""
    wl = make_workload(name)
    t = make_tensors(wl)
    g = run_gpu(wl.parent, wl.node_len, t)
    ref = oracle_ref(wl.parent, wl.node_len, t, heads=heads, use_nodes=True)
    eo, el = compare_fwd(g, ref, heads, wl.n_tokens)
    e = compare_bwd(g, ref, heads, wl.Hq, wl.Hkv)
    print(f"{name}: O {eo:.3e} LSE {el:.3e} grads {e}")
    assert eo <= O_TOL and el <= O_TOL
    assert max(e.values()) <= GRAD_TOL


def test_dkdv_deterministic():
    """dK and dV are reduced on chip per key tile (no atomics): two runs agree bit for bit."""
    wl = make_workload("caterpillar")
    t = make_tensors(wl)
    a = run_gpu(wl.parent, wl.node_len, t)
    b = run_gpu(wl.parent, wl.node_len, t)
    assert torch.equal(a["dk"], b["dk"]) and torch.equal(a["dv"], b["dv"])
    assert torch.equal(a["o"], b["o"]) and torch.equal(a["lse"], b["lse"])


def test_bwd_without_rope_inverse():
    """rope_theta <= 0 returns gradients w.r.t. the rotated inputs: rotating them back on the
    host (oracle RoPE transpose at the plan positions) gives the rope_theta > 0 result."""
    wl = _wl(*random_tree(3, 10, max_len=80), 2, 1, 128)
    t = make_tensors(wl)
    g = run_gpu(wl.parent, wl.node_len, t)
    plan, dev = g["plan"], torch.device("cuda", 0)
    dq2, dk2, dv2 = tam.tree_attn_bwd(plan, g["qr"], g["kr"], t["v"].to(dev), g["o"], g["lse"], g["dO"],
                                      rope_theta=0.0)
    torch.cuda.synchronize()
    pos = oracle.plan(wl.parent, wl.node_len)["pos"]
    back = oracle.rope_transpose(f64(dk2), pos, 10000.0)
    assert np.abs(back - f64(g["dk"])).max() <= 2e-2 * np.abs(f64(g["dk"])).max()
    assert torch.equal(dv2, g["dv"])


WEIGHTED = SMALL[:4] + [("caterpillar", None, None, None, None)]


@pytest.mark.parametrize("name,tree,Hq,Hkv,d", WEIGHTED, ids=[s[0] for s in WEIGHTED])
def test_bwd_weighted_matches_oracle_and_unfused(name, tree, Hq, Hkv, d):
    """tree_attn_bwd_weighted (the weights g_t/K folded into the backward's probabilities, no
    dO formed) against the fp64 oracle of the path-averaged loss (section 6.2) at the target
    tolerance, and against tree_apply_weights + tree_attn_bwd: the same sums, where the unfused
    path rounds dO = w U to bf16 first, so within a few bf16 steps of max |grad|."""
    wl = make_workload(name) if tree is None else _wl(*tree, Hq, Hkv, d)
    Hq = wl.Hq
    heads = [0, 1, 2, 3] if tree is None else range(Hq)
    t = make_tensors(wl)
    g = run_gpu(wl.parent, wl.node_len, t)                 # unfused: dO from tree_apply_weights
    status = tam.new_status()
    u = t["u"].cuda().contiguous()
    dq, dk, dv = tam.tree_attn_bwd_weighted(g["plan"], g["qr"], g["kr"], t["v"].cuda(), g["o"], g["lse"], u,
                                            status=status)
    torch.cuda.synchronize()
    tam.check_status(status, "tree_attn_bwd_weighted")
    fused = dict(dq=dq, dk=dk, dv=dv)
    ref = oracle_ref(wl.parent, wl.node_len, t, heads=heads, use_nodes=tree is None)
    e = compare_bwd(fused, ref, heads, Hq, wl.Hkv)
    diffs = {x: float((f64(fused[x]) - f64(g[x])).__abs__().max() / max(np.abs(f64(g[x])).max(), 1e-30))
             for x in ("dq", "dk", "dv")}
    print(f"{name}: fused vs oracle {e}; fused vs unfused {diffs}")
    assert max(e.values()) <= GRAD_TOL
    assert max(diffs.values()) <= 2e-2
