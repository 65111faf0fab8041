"""Split rows and columns (Tree Attention page, the associativity of the (max, numerator,
denominator) softmax state over disjoint key subsets).

Forward split-KV: a query tile's key tiles are dealt to the CTAs of a cluster, each keeps its
own online-softmax state, and rank 0 merges the states by the associative rule.  Backward: the
query steps of one key tile's column are dealt to the CTAs of a cluster and their dK / dV
partials are summed in fixed rank order.

For split = 1, 2 and 4 (forced), O, LSE, dQ, dK, dV match the fp64 oracle at the target
tolerances on trees with ragged tiles, many node runs, GQA 4:1 and 1:1, and gateway partitions
(whose gateway tiles are dealt like the row's own); with a backward split, two runs give
bit-identical dK and dV."""
import numpy as np
import pytest
import torch

import tree_masked_attention_plan_gb300 as tam
from workloads import make_tensors, make_workload, random_tree
from workloads.trees import Workload

from _gpu import GRAD_TOL, O_TOL, compare_bwd, compare_fwd, oracle_ref, run_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _automatic_split_afterwards():
    yield
    tam.tree_set_bwd_split(0)
    tam.tree_set_fwd_split(0)


def _wl(parent, node_len, Hq, Hkv, d):
    return Workload(name="t", parent=np.asarray(parent, np.int32), node_len=np.asarray(node_len, np.int32),
                    Hq=Hq, Hkv=Hkv, d=d)


TREES = [("ragged_d128_gqa4", random_tree(51, 14, max_len=120), 8, 2, 128),
         ("tiny_nodes_d64", random_tree(52, 250, max_len=5, zero_prob=0.1), 2, 2, 64),
         ("forest_d128_gqa1", random_tree(53, 10, max_len=200, n_roots=3), 2, 2, 128),
         ("one_tile_d64", (np.array([-1, 0]), np.array([40, 50])), 4, 1, 64)]


@pytest.mark.parametrize("split", [1, 2, 4])
@pytest.mark.parametrize("name,tree,Hq,Hkv,d", TREES, ids=[t[0] for t in TREES])
def test_split_columns_match_oracle(name, tree, Hq, Hkv, d, split):
    tam.tree_set_bwd_split(split)
    tam.tree_set_fwd_split(split)
    wl = _wl(*tree, Hq, Hkv, d)
    t = make_tensors(wl)
    g = run_gpu(wl.parent, wl.node_len, t)
    ref = oracle_ref(wl.parent, wl.node_len, t, heads=range(Hq))
    eo, el = compare_fwd(g, ref, range(Hq), wl.n_tokens)
    e = compare_bwd(g, ref, range(Hq), Hq, Hkv)
    print(f"{name} split {split}: grads {e}")
    assert eo <= O_TOL and el <= O_TOL
    assert max(e.values()) <= GRAD_TOL


@pytest.mark.parametrize("split", [2, 4])
def test_split_dkdv_deterministic(split):
    tam.tree_set_bwd_split(split)
    wl = make_workload("caterpillar")
    t = make_tensors(wl)
    a = run_gpu(wl.parent, wl.node_len, t)
    b = run_gpu(wl.parent, wl.node_len, t)
    assert torch.equal(a["dk"], b["dk"]) and torch.equal(a["dv"], b["dv"])


def test_caterpillar_split_matches_oracle():
    """The small benchmark tree takes the automatic split (2 on 152 SMs); two kv-head groups
    against the per-node oracle."""
    wl = make_workload("caterpillar")
    t = make_tensors(wl)
    g = run_gpu(wl.parent, wl.node_len, t)
    heads = [0, 1, 2, 3, 28, 29, 30, 31]
    ref = oracle_ref(wl.parent, wl.node_len, t, heads=heads, use_nodes=True)
    e = compare_bwd(g, ref, heads, wl.Hq, wl.Hkv)
    print(f"caterpillar automatic split: grads {e}")
    assert max(e.values()) <= GRAD_TOL


@pytest.mark.parametrize("split", [2, 4])
def test_split_gateway_partition(split):
    """Gateway key tiles (every query tile of the partition in their column) split too; the
    cluster's rank 0 adds the summed fp32 gradients to the caller's accumulators."""
    from _gateway import gateway_tree
    import oracle
    from _gpu import f64, rel_err
    from test_gpu_gateway import _tensors, run_partitioned
    tam.tree_set_bwd_split(split)
    dev = torch.device("cuda", 0)
    parent, lens, cut = gateway_tree(8, [200, 70], branch_len=30, n_extra=60, max_len=40)
    N = int(np.sum(lens))
    t = _tensors(N, 4, 2, 128, seed=23)
    P, got = run_partitioned(parent, lens, cut, t, dev)
    ref = oracle.attention_nodes(parent, lens, t["q"], t["k"], t["v"], t["u"], heads=list(range(4)), theta=10000.0)
    errs = {x: rel_err(f64(got[x]), ref[x]) for x in ("dq", "dk", "dv")}
    print(f"gateway split {split}: {errs}")
    assert max(errs.values()) <= GRAD_TOL


@pytest.mark.parametrize("split", [1, 2, 4])
def test_forward_split_long_rows(split):
    """A chain of 24 tiles (rows of up to 24 key tiles) with one q-head pair: few CTAs, long rows."""
    tam.tree_set_fwd_split(split)
    wl = _wl(np.array([-1] + list(range(11))), np.full(12, 250), 2, 1, 128)
    t = make_tensors(wl)
    g = run_gpu(wl.parent, wl.node_len, t, backward=False)
    ref = oracle_ref(wl.parent, wl.node_len, t, heads=[0, 1])
    eo, el = compare_fwd(g, ref, [0, 1], wl.n_tokens)
    print(f"chain fwd split {split}: O {eo:.2e} LSE {el:.2e}")
    assert eo <= O_TOL and el <= O_TOL


@pytest.mark.parametrize("split", [2, 4])
def test_forward_split_gateway(split):
    """A small child partition below a long gateway (9 gateway tiles, 1-2 own tiles): the
    gateway tiles are dealt to the cluster's CTAs with the row's own tiles."""
    from _gateway import gateway_tree
    import oracle
    from _gpu import f64
    from test_gpu_gateway import _tensors, run_partitioned
    tam.tree_set_fwd_split(split)
    dev = torch.device("cuda", 0)
    parent, lens, cut = gateway_tree(9, [700, 430], branch_len=40, n_extra=30, max_len=12)
    N = int(np.sum(lens))
    t = _tensors(N, 4, 1, 128, seed=29)
    P, got = run_partitioned(parent, lens, cut, t, dev)
    ref = oracle.attention_nodes(parent, lens, t["q"], t["k"], t["v"], t["u"], heads=list(range(4)), theta=10000.0)
    eo = np.abs(f64(got["o"]) - ref["o"]).max()
    el = np.abs(f64(got["lse"]) - ref["lse"]).max()
    print(f"gateway fwd split {split}: A={P['A']} O {eo:.2e} LSE {el:.2e}")
    assert eo <= O_TOL and el <= O_TOL
