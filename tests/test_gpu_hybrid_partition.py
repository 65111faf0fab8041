"""Hybrid-layer context across a gateway partition cut ("Tree Training 技术详解", section 8.2 with
section 9): a tree cut below one node runs as a parent partition plus child partitions, and
the layers that carry context along root paths must see, in each child partition, the context
the whole tree would give it.

* Causal convolution (section 9.2): each child partition runs on its context tree (a root node
  holding the gateway path's last K-1 tokens, gathered from the parent partition, with zero
  upstream gradient); the gradient those context rows receive is added to the parent
  partition's dx rows, and dw, dbias are summed over the partitions.  y, dx, dw, dbias of the
  assembled partitions match the fp64 oracle of the whole tree.
* Recurrent-state routing (section 9.1): each child partition's context node carries the final
  state of the gateway path's last token-holding node; the routed initial states of every node
  and the routing backward (the context node's gradient added to that gateway node) match the
  oracle on the whole tree.
"""
import numpy as np
import pytest
import torch

import oracle
import tree_masked_attention_plan_gb300 as tam
from tree_masked_attention_plan_gb300.partition import context_tree, gateway_state_node, partition_tree
from workloads import make_conv_tensors

from _gateway import gateway_tree

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda", 0)


def _f64(t):
    return t.detach().to(torch.float64).cpu().numpy()


CASES = [("ragged", 11, [70, 45], 30, 40, 12, 4),     # seed, gateway path, side branch, extra nodes, max len, K
         ("k8_short_gateway", 12, [3], 25, 30, 10, 8),  # gateway shorter than K - 1
         ("empty_nodes", 13, [20, 0, 9], 15, 35, 6, 3)]


@pytest.mark.parametrize("name,seed,gw,side,n_extra,max_len,K", CASES, ids=[c[0] for c in CASES])
def test_conv_across_partitions(name, seed, gw, side, n_extra, max_len, K):
    C = 64
    parent, lens, cut = gateway_tree(seed, gw, branch_len=side, n_extra=n_extra, max_len=max_len)
    P = partition_tree(parent, lens, cut)
    p = oracle.plan(parent, lens)
    N = p["n_tokens"]
    t = make_conv_tensors(N, C, K, seed=seed)
    wgt = torch.tensor(p["g"], dtype=torch.float64)[:, None] / p["n_paths"]
    dy = (t["u"].double() * wgt).to(torch.bfloat16)                 # path-weighted upstream gradient
    ref = oracle.conv_paths(parent, lens, _f64(t["x"]), _f64(t["w"]), _f64(t["bias"]), _f64(dy) / wgt.numpy(), p=p)
    x, w, b, dyd = t["x"].to(DEV), t["w"].to(DEV), t["bias"].to(DEV), dy.to(DEV)
    y_all = torch.zeros(N, C, dtype=torch.float32, device=DEV)
    dx_all = torch.zeros(N, C, dtype=torch.float32, device=DEV)
    dw_sum = torch.zeros(K, C, dtype=torch.float32, device=DEV)
    db_sum = torch.zeros(C, dtype=torch.float32, device=DEV)
    st = tam.new_status(DEV)

    def run(tree_parent, tree_len, xs, dys):
        plan = tam.tree_plan(tree_parent, tree_len, device=DEV)
        tree = tam.tree_arrays(tree_parent, tree_len, DEV)
        y = tam.tree_conv1d_fwd(plan, tree, xs, w, b, status=st)
        dx, dw, db = tam.tree_conv1d_bwd(plan, tree, xs, w, dys, with_bias=True, status=st)
        return y, dx, dw, db

    pp = P["parent"]
    idx = torch.as_tensor(pp.tokens, device=DEV)
    y, dx, dw, db = run(pp.parent, pp.node_len, x[idx].contiguous(), dyd[idx].contiguous())
    y_all[idx] = y.float()
    dx_all.index_add_(0, idx, dx.float())
    dw_sum += dw
    db_sum += db
    ctx = min(K - 1, P["A"])
    ctx_tok = torch.as_tensor(P["gw_tokens"][len(P["gw_tokens"]) - ctx:], device=DEV)   # whole-tree ids
    for ch in P["children"]:
        cpar, clen = context_tree(ch, ctx)
        cidx = torch.as_tensor(ch.tokens, device=DEV)
        xs = torch.cat([x[ctx_tok], x[cidx]]).contiguous()
        dys = torch.cat([torch.zeros(ctx, C, dtype=torch.bfloat16, device=DEV), dyd[cidx]]).contiguous()
        y, dx, dw, db = run(cpar, clen, xs, dys)
        y_all[cidx] = y[ctx:].float()
        dx_all.index_add_(0, cidx, dx[ctx:].float())
        dx_all.index_add_(0, ctx_tok, dx[:ctx].float())        # relayed to the gateway tokens
        dw_sum += dw
        db_sum += db
    torch.cuda.synchronize()
    tam.check_status(st, "partitioned conv")
    # y: one bf16 rounding; dx: a sum of up to two bf16-rounded parts (own partition + relay)
    ey = np.abs(_f64(y_all) - ref["y"]).max() / np.abs(ref["y"]).max()
    edx = np.abs(_f64(dx_all) - ref["dx"]).max() / np.abs(ref["dx"]).max()
    edw = np.abs(_f64(dw_sum) - ref["dw"]).max() / np.abs(ref["dw"]).max()
    edb = np.abs(_f64(db_sum) - ref["db"]).max() / np.abs(ref["db"]).max()
    print(f"{name}: A={P['A']} ctx={ctx} children={len(P['children'])} y {ey:.2e} dx {edx:.2e} dw {edw:.2e} db {edb:.2e}")
    assert ey < 1e-2 and edx < 2e-2 and edw < 1e-3 and edb < 1e-3


@pytest.mark.parametrize("name,seed,gw,side,n_extra,max_len", [c[:6] for c in CASES], ids=[c[0] for c in CASES])
def test_state_routing_across_partitions(name, seed, gw, side, n_extra, max_len):
    S = 16
    parent, lens, cut = gateway_tree(seed, gw, branch_len=side, n_extra=n_extra, max_len=max_len)
    P = partition_tree(parent, lens, cut)
    n = len(parent)
    rng = np.random.default_rng(seed)
    final = rng.standard_normal((n, S)).astype(np.float32)
    d_init = rng.standard_normal((n, S)).astype(np.float32)
    ref_init = oracle.route_states(parent, lens, final)
    ref_dfin = oracle.route_states_bwd(parent, lens, d_init)
    init_all = np.zeros((n, S))
    dfin_all = np.zeros((n, S))
    pp = P["parent"]
    tree = tam.tree_arrays(pp.parent, pp.node_len, DEV)
    fin_p = torch.as_tensor(final[pp.nodes], device=DEV)
    init_all[pp.nodes] = _f64(tam.tree_route_states(tree, fin_p))
    dfin_p = tam.tree_route_states_bwd(tree, torch.as_tensor(d_init[pp.nodes], device=DEV))
    g = gateway_state_node(P, parent, lens)
    for ch in P["children"]:
        cpar, clen = context_tree(ch, 1)                 # node 0 stands for the gateway's last node
        ctree = tam.tree_arrays(cpar, clen, DEV)
        fin_c = torch.zeros(len(cpar), S, device=DEV)
        if g >= 0:
            fin_c[0] = fin_p[g]
        fin_c[1:] = torch.as_tensor(final[ch.nodes], device=DEV)
        init_all[ch.nodes] = _f64(tam.tree_route_states(ctree, fin_c))[1:]
        d_in = torch.zeros(len(cpar), S, device=DEV)
        d_in[1:] = torch.as_tensor(d_init[ch.nodes], device=DEV)
        dfin_c = tam.tree_route_states_bwd(ctree, d_in)
        dfin_all[ch.nodes] += _f64(dfin_c)[1:]
        if g >= 0:
            dfin_p[g] += dfin_c[0]                      # the context node's gradient, relayed
    dfin_all[pp.nodes] += _f64(dfin_p)
    torch.cuda.synchronize()
    assert np.array_equal(init_all, ref_init.astype(np.float32).astype(np.float64))
    assert np.abs(dfin_all - ref_dfin).max() < 1e-5 * max(1.0, np.abs(ref_dfin).max())
