"""The CUDA plan (host node pass + expansion + tile kernels) is bit-exact against the oracle."""
import numpy as np
import pytest
import torch

import oracle
import tree_masked_attention_plan_gb300 as tam
from workloads import CONFIGS, make_workload, random_tree

pytestmark = pytest.mark.gpu


def _trees():
    out = [("single", (np.array([-1]), np.array([1]))),
           ("one_tile", (np.array([-1, 0]), np.array([100, 28]))),
           ("ragged129", (np.array([-1, 0, 0]), np.array([1, 64, 64]))),
           ("chain", (np.array([-1] + list(range(299))), np.full(300, 3))),
           ("star", (np.array([-1] + [0] * 400), np.r_[50, np.arange(400) % 7])),
           ("zero_root", (np.array([-1, 0, 0, 1]), np.array([0, 5, 0, 300]))),
           ("star_1100_tiles", (np.array([-1] + [0] * 1100), np.full(1101, 128))),
           ("forest_1200_tiles", (np.full(600, -1), np.full(600, 256)))]
    for s in range(24):
        out.append((f"rand{s}", random_tree(1000 + s, n_nodes=2 + 7 * s, max_len=40 + 10 * s,
                                            zero_prob=0.1 if s % 3 == 0 else 0.0, n_roots=1 + (s % 5 == 2) * 3)))
    return out


def _check_plan(parent, node_len):
    ref = oracle.plan(parent, node_len)
    plan = tam.tree_plan(parent, node_len)
    torch.cuda.synchronize()
    a = {k: v.cpu().numpy() for k, v in plan.arrays().items()}
    N, T = ref["n_tokens"], ref["n_tiles"]
    assert plan.n_tokens == N and plan.n_tiles == T and plan.n_paths == ref["n_paths"]
    for f in ("order", "dfs_in", "dfs_out", "tok_start", "depth_off", "leaves"):
        assert np.array_equal(a[f], ref[f]), f
    for f in ("tok_node", "pos", "g", "tok_in", "tok_out", "hi"):
        assert np.array_equal(a[f][:N], ref[f]), f
    assert np.array_equal(a["w"][:N].view(np.uint32), ref["w"].view(np.uint32))   # bitwise
    # padding values documented in the header
    assert np.all(a["tok_in"][N:] == -1) and np.all(a["tok_out"][N:] == -2) and np.all(a["tok_node"][N:] == -1)
    assert np.array_equal(a["tile_class"], ref["tile_class"])
    for f in ("row_ptr", "col_ptr", "row_order", "col_order"):
        assert np.array_equal(a[f], ref[f]), f
    nnz = ref["nnz"]
    assert np.array_equal(a["row_idx"][:nnz], ref["row_idx"]) and np.array_equal(a["col_idx"][:nnz], ref["col_idx"])
    assert a["counts"][:3].tolist() == [nnz, ref["n_full"], ref["n_partial"]]
    assert np.array_equal(a["tile_nruns"], ref["tile_nruns"])
    runs = a["tile_runs"].reshape(T, tam.MAX_RUNS, 4)
    for t in range(T):
        k = min(len(ref["tile_runs"][t]), tam.MAX_RUNS)
        assert runs[t, :k].tolist() == [list(r) for r in ref["tile_runs"][t][:k]], t


@pytest.mark.parametrize("name,tree", _trees(), ids=[t[0] for t in _trees()])
def test_plan_bit_exact_random(name, tree):
    _check_plan(*tree)


@pytest.mark.parametrize("name", list(CONFIGS))
def test_plan_bit_exact_configs(name):
    wl = make_workload(name)
    _check_plan(wl.parent, wl.node_len)


def test_invalid_trees_rejected():
    for parent, lens in (([0], [3]), ([1, 0], [1, 1]), ([-1, 0], [1, -1]), ([-1, 0], [0, 0])):
        with pytest.raises(tam.TreeError) as e:
            tam.tree_plan(parent, lens)
        assert e.value.code == -1
