"""Gateway partitions on the GPU ("Tree Training 技术详解", section 8.2): a tree cut below one
node runs as a parent partition plus one child partition per child of the cut node.  The
children read the parent's rotated K/V of the root-to-cut path as a gateway, add their
gradients w.r.t. it into one fp32 accumulator, and the relay adds that into the parent's dK,
dV.  Every token's O, LSE, dQ, dK, dV must match the fp64 oracle of the WHOLE tree."""
import numpy as np
import pytest
import torch

import oracle
import tree_masked_attention_plan_gb300 as tam
from _gateway import gateway_tree, partition
from _gpu import GRAD_TOL, O_TOL, f64, rel_err

pytestmark = pytest.mark.gpu

THETA = 10000.0


def _tensors(N, Hq, Hkv, d, seed=1):
    g = torch.Generator().manual_seed(seed)
    mk = lambda h: torch.randn(N, h, d, generator=g).to(torch.bfloat16)
    return dict(q=mk(Hq), k=mk(Hkv), v=mk(Hkv), u=mk(Hq))


def run_partitioned(parent, lens, cut, t, dev):
    P = partition(parent, lens, cut)
    N = P["full"]["n_tokens"]
    Hq, d = t["q"].shape[1], t["q"].shape[2]
    Hkv = t["k"].shape[1]
    st = tam.new_status(dev)
    # loss weights g_t / K of the WHOLE tree, gathered per partition
    full_plan = tam.tree_plan(parent, lens, device=dev)
    dO_full = tam.tree_apply_weights(full_plan, t["u"].to(dev))
    out = {x: torch.zeros(N, H, d, dtype=torch.bfloat16, device=dev)
           for x, H in (("o", Hq), ("dq", Hq), ("dk", Hkv), ("dv", Hkv))}
    lse = torch.zeros(Hq, N, dtype=torch.float32, device=dev)

    def inputs(part):
        idx = torch.as_tensor(part.tokens, device=dev)
        return [t[x].to(dev)[idx].contiguous() for x in ("q", "k", "v")] + [dO_full[idx].contiguous(), idx]

    # parent partition: an ordinary tree
    pp = P["parent"]
    plan_p = tam.tree_plan(pp.parent, pp.node_len, device=dev)
    q, k, v, dO, idx_p = inputs(pp)
    qr, kr = tam.tree_rope_fwd(plan_p, q, k, THETA)
    o_p, lse_p = tam.tree_attn_fwd(plan_p, qr, kr, v, status=st)
    dq_p, dk_p, dv_p = tam.tree_attn_bwd(plan_p, qr, kr, v, o_p, lse_p, dO, rope_theta=THETA, status=st)
    rows = torch.as_tensor(P["gw_rows"], device=dev)
    k_gw, v_gw = kr[rows].contiguous(), v[rows].contiguous()
    dk_gw = torch.zeros(P["A"], Hkv, d, dtype=torch.float32, device=dev)
    dv_gw = torch.zeros_like(dk_gw)
    # child partitions below the gateway
    for ch in P["children"]:
        plan_c = tam.tree_plan(ch.parent, ch.node_len, device=dev, pos_offset=P["A"])
        q, k, v, dO, idx = inputs(ch)
        qr_c, kr_c = tam.tree_rope_fwd(plan_c, q, k, THETA)
        o_c, lse_c = tam.tree_attn_fwd_gateway(plan_c, k_gw, v_gw, qr_c, kr_c, v, status=st)
        dq_c, dk_c, dv_c = tam.tree_attn_bwd_gateway(plan_c, k_gw, v_gw, qr_c, kr_c, v, o_c, lse_c, dO, dk_gw, dv_gw,
                                                     rope_theta=THETA, status=st)
        out["o"][idx], out["dq"][idx], out["dk"][idx], out["dv"][idx] = o_c, dq_c, dk_c, dv_c
        lse[:, idx] = lse_c[:, :len(ch.tokens)]
    tam.tree_relay_add(rows.to(torch.int32), dk_gw, dv_gw, dk_p, dv_p)
    out["o"][idx_p], out["dq"][idx_p], out["dk"][idx_p], out["dv"][idx_p] = o_p, dq_p, dk_p, dv_p
    lse[:, idx_p] = lse_p[:, :len(pp.tokens)]
    torch.cuda.synchronize()
    tam.check_status(st, "gateway partitions")
    out["lse"] = lse
    return P, out


CASES = [
    # seed, gateway path lengths, side branch, extra nodes, max node length, Hq, Hkv, d
    ("ragged", 0, [150, 90, 57], 200, 18, 160, 4, 2, 128),
    ("aligned", 1, [128, 128], 300, 14, 200, 4, 2, 128),
    ("long_gateway", 2, [700, 420], 64, 12, 120, 4, 2, 128),
    ("short_gateway", 3, [3], 40, 16, 150, 4, 2, 128),
    ("one_head_d64", 4, [77, 50], 90, 12, 140, 2, 2, 64),
]


@pytest.mark.parametrize("name,seed,gw,side,n_extra,max_len,Hq,Hkv,d", CASES, ids=[c[0] for c in CASES])
def test_partitioned_tree_matches_whole_tree(name, seed, gw, side, n_extra, max_len, Hq, Hkv, d):
    dev = torch.device("cuda", 0)
    parent, lens, cut = gateway_tree(seed, gw, branch_len=side, n_extra=n_extra, max_len=max_len)
    N = int(np.sum(lens))
    t = _tensors(N, Hq, Hkv, d, seed=seed + 11)
    P, got = run_partitioned(parent, lens, cut, t, dev)
    ref = oracle.attention_nodes(parent, lens, t["q"], t["k"], t["v"], t["u"], heads=list(range(Hq)), theta=THETA)
    eo = np.abs(f64(got["o"]) - ref["o"]).max()
    el = np.abs(f64(got["lse"]) - ref["lse"]).max()
    errs = {x: rel_err(f64(got[x]), ref[x]) for x in ("dq", "dk", "dv")}
    gw_err = {x: rel_err(f64(got[x])[P["gw_tokens"]], ref[x][P["gw_tokens"]]) for x in ("dk", "dv")}
    print(f"{name}: N={N} A={P['A']} children={len(P['children'])} O {eo:.2e} LSE {el:.2e} "
          f"grads {errs} gateway rows {gw_err}")
    assert eo <= O_TOL and el <= O_TOL
    assert all(e <= GRAD_TOL for e in errs.values()), errs
    assert all(e <= GRAD_TOL for e in gw_err.values()), gw_err


def test_gateway_argument_errors():
    dev = torch.device("cuda", 0)
    parent, lens, cut = gateway_tree(5, [40], branch_len=10, n_extra=5, max_len=10)
    plan = tam.tree_plan(parent, lens, device=dev, pos_offset=40)
    N = plan.n_tokens
    q = torch.zeros(N, 2, 64, dtype=torch.bfloat16, device=dev)
    k = torch.zeros(N, 1, 64, dtype=torch.bfloat16, device=dev)
    empty = torch.zeros(0, 1, 64, dtype=torch.bfloat16, device=dev)
    with pytest.raises(tam.TreeError) as e:
        tam.tree_attn_fwd_gateway(plan, empty, empty, q, k, k)
    assert e.value.code == -6
    with pytest.raises(tam.TreeError) as e:
        tam.tree_plan(parent, lens, device=dev, pos_offset=-3)
    assert e.value.code == -6
