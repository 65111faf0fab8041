"""Parity of the hybrid-layer kernels ("Tree Training 技术详解", section 9) with the oracle.

* tree convolution forward and backward against the oracle's path expansion (every root-to-
  leaf path convolved as its own sequence), on random trees with zero-length nodes, several
  roots, ragged token counts and channel counts that leave partial channel slabs; ~90K tokens on
  one slab (each block walks many staged tiles); a chain of
  one-token nodes with empty nodes between them (every tap crosses nodes); one token;
* the rollout32k tree at full size with 8192 channels, on 64 sampled channels (channels are
  independent in a depthwise convolution, so the oracle on a channel subset is exact);
* state routing and its transpose against the oracle.

The upstream gradient is the path-weighted one, dy_t = (g_t / K) u_t rounded to bf16; the
oracle, which averages over paths itself, gets u_t = dy_t K / g_t.

Tolerances: y and dx are fp32 sums rounded to bf16, so |err| <= 2^-8 |ref| plus 1e-4 of the
largest |ref| for the fp32 summation; dw and dbias are fp32 sums of exact bf16 products over at
most a few thousand partials, bounded by 1e-4 of the sum of the terms' magnitudes (computed by
running the oracle on |x|, |u|)."""
import numpy as np
import pytest
import torch

import oracle
import tree_masked_attention_plan_gb300 as tam
from workloads import make_conv_tensors, make_workload, random_tree

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda", 0)


def _f64(t):
    return t.detach().to(torch.float64).cpu().numpy()


def _dy(p, u):
    """path-weighted upstream gradient (bf16) and the oracle's matching per-path u (fp64)"""
    wgt = torch.tensor(p["g"], dtype=torch.float64)[:, None] / p["n_paths"]
    dy = (u.double() * wgt).to(torch.bfloat16)
    return dy, _f64(dy) / wgt.numpy()


def _check_conv(parent, node_len, C, K, seed, with_bias=True, channels=None):
    p = oracle.plan(parent, node_len)
    N = p["n_tokens"]
    t = make_conv_tensors(N, C, K, seed, with_bias)
    dy, u_or = _dy(p, t["u"])
    plan = tam.tree_plan(parent, node_len, device=DEV)
    tree = tam.tree_arrays(parent, node_len, DEV)
    x, w = t["x"].to(DEV), t["w"].to(DEV)
    b = t["bias"].to(DEV) if with_bias else None
    status = tam.new_status(DEV)
    y = tam.tree_conv1d_fwd(plan, tree, x, w, b, status=status)
    dx, dw, db = tam.tree_conv1d_bwd(plan, tree, x, w, dy.to(DEV), with_bias=with_bias, status=status)
    torch.cuda.synchronize()
    tam.check_status(status, "tree conv")
    ch = np.arange(C) if channels is None else channels
    xs, ws = _f64(t["x"])[:, ch], _f64(t["w"])[:, ch]
    bs = _f64(t["bias"])[ch] if with_bias else None
    ref = oracle.conv_paths(parent, node_len, xs, ws, bs, u_or[:, ch], p=p)
    mag = oracle.conv_paths(parent, node_len, np.abs(xs), np.abs(ws), None, np.abs(u_or[:, ch]), p=p)
    gy, gdx, gdw = _f64(y)[:, ch], _f64(dx)[:, ch], _f64(dw)[:, ch]
    for name, got, exp in (("y", gy, ref["y"]), ("dx", gdx, ref["dx"])):
        tol = 2.0 ** -8 * np.abs(exp) + 1e-4 * np.abs(exp).max()
        bad = np.abs(got - exp) > tol
        assert not bad.any(), (name, np.argwhere(bad)[:5], np.abs(got - exp).max())
    assert (np.abs(gdw - ref["dw"]) <= 1e-4 * mag["dw"] + 1e-30).all(), np.abs(gdw - ref["dw"]).max()
    if with_bias:
        gdb = _f64(db)[ch]
        assert (np.abs(gdb - ref["db"]) <= 1e-4 * mag["db"] + 1e-30).all(), np.abs(gdb - ref["db"]).max()
    return ref


@pytest.mark.parametrize("seed,C,K", [(0, 64, 4), (1, 8, 1), (2, 264, 8), (3, 2056, 3), (4, 128, 6)])
def test_conv_random_trees(seed, C, K):
    parent, node_len = random_tree(100 + seed, n_nodes=40 + 20 * seed, max_len=60, zero_prob=0.2,
                                   n_roots=1 + seed % 3)
    _check_conv(parent, node_len, C, K, seed, with_bias=seed % 2 == 0)


def test_conv_many_tiles_per_block():
    """~90K tokens over 8 channels: one channel slab, so every block walks many token tiles
    through both staging buffers."""
    parent, node_len = random_tree(300, n_nodes=3000, max_len=60, zero_prob=0.1, n_roots=3)
    _check_conv(parent, node_len, 8, 4, 10)


def test_conv_chain_of_single_tokens_through_empty_nodes():
    n = 120
    parent = np.arange(-1, n - 1)
    node_len = np.where(np.arange(n) % 3 == 1, 0, 1)       # every third node holds no tokens
    _check_conv(parent, node_len, 16, 8, 7)


def test_conv_single_token():
    _check_conv(np.array([-1]), np.array([1]), 8, 4, 8)


def test_conv_rollout32k_full_size_sampled_channels():
    wl = make_workload("rollout32k")
    C = 8192
    ch = np.arange(0, C, C // 64)
    _check_conv(wl.parent, wl.node_len, C, 4, 9, channels=ch)


def test_conv_rejects_bad_shapes():
    parent, node_len = random_tree(5, n_nodes=6, max_len=10)
    plan = tam.tree_plan(parent, node_len, device=DEV)
    tree = tam.tree_arrays(parent, node_len, DEV)
    N = plan.n_tokens
    x = torch.zeros(N, 12, dtype=torch.bfloat16, device=DEV)
    with pytest.raises(tam.TreeError):
        tam.tree_conv1d_fwd(plan, tree, x, torch.zeros(4, 12, device=DEV))          # C % 8 != 0
    x = torch.zeros(N, 16, dtype=torch.bfloat16, device=DEV)
    with pytest.raises(tam.TreeError):
        tam.tree_conv1d_fwd(plan, tree, x, torch.zeros(9, 16, device=DEV))          # K > 8


@pytest.mark.parametrize("seed", range(3))
def test_route_states(seed):
    parent, node_len = random_tree(200 + seed, n_nodes=300, max_len=20, zero_prob=0.3, n_roots=1 + seed)
    n, S = len(parent), 516
    g = torch.Generator().manual_seed(seed)
    fin = torch.randn(n, S, generator=g)
    d_init = torch.randn(n, S, generator=g)
    tree = tam.tree_arrays(parent, node_len, DEV)
    init = tam.tree_route_states(tree, fin.to(DEV))
    d_fin = tam.tree_route_states_bwd(tree, d_init.to(DEV))
    torch.cuda.synchronize()
    assert np.array_equal(_f64(init), oracle.route_states(parent, node_len, fin.double().numpy()))
    ref = oracle.route_states_bwd(parent, node_len, d_init.double().numpy())
    assert np.abs(_f64(d_fin) - ref).max() <= 1e-5 * max(1.0, np.abs(ref).max())
