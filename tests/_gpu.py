"""Shared helpers of the GPU parity tests: run the CUDA path through the C-ABI binding and the
CPU oracle on the same seeded inputs, and compare."""
from __future__ import annotations

import numpy as np
import torch

import oracle
import tree_masked_attention_plan_gb300 as tam
from workloads import make_tensors

O_TOL = 2e-2          # max-abs on O and LSE against the fp64 oracle
GRAD_TOL = 5e-2       # max-abs on dQ, dK, dV relative to max |reference|


def run_gpu(parent, node_len, t, theta=10000.0, backward=True, Hq=None):
    """Plan -> RoPE -> forward (-> weights -> backward) on cuda:0; returns CPU float64 arrays."""
    dev = torch.device("cuda", 0)
    status = tam.new_status(dev)
    plan = tam.tree_plan(parent, node_len, device=dev)
    q, k, v, u = (t[x].to(dev).contiguous() for x in ("q", "k", "v", "u"))
    qr, kr = tam.tree_rope_fwd(plan, q, k, theta)
    o, lse = tam.tree_attn_fwd(plan, qr, kr, v, status=status)
    out = dict(plan=plan, qr=qr, kr=kr, o=o, lse=lse)
    if backward:
        dO = tam.tree_apply_weights(plan, u)
        dq, dk, dv = tam.tree_attn_bwd(plan, qr, kr, v, o, lse, dO, rope_theta=theta, status=status)
        out.update(dO=dO, dq=dq, dk=dk, dv=dv)
    torch.cuda.synchronize()
    tam.check_status(status, "attention kernels")
    return out


def f64(x):
    return x.detach().to(torch.float64).cpu().numpy()


def oracle_ref(parent, node_len, t, heads, plan=None, use_nodes=False, theta=10000.0):
    fn = oracle.attention_nodes if use_nodes else oracle.attention_paths
    return fn(parent, node_len, t["q"], t["k"], t["v"], t["u"], heads=heads, theta=theta, p=plan)


def kv_heads_covered(heads, Hq, Hkv):
    """kv heads whose whole q-head group is in `heads` (their dK/dV are fully determined)."""
    grp = Hq // Hkv
    hs = set(heads)
    return [g for g in range(Hkv) if all(g * grp + i in hs for i in range(grp))]


def compare_fwd(gpu, ref, heads, N):
    o = f64(gpu["o"])
    lse = f64(gpu["lse"])[:, :N]
    eo = max(np.abs(o[:, h] - ref["o"][:, h]).max() for h in heads)
    el = max(np.abs(lse[h] - ref["lse"][h]).max() for h in heads)
    return eo, el


def rel_err(got, ref):
    """max|got - ref| / max|ref|; where the exact gradient is identically zero (a lone token:
    dS = P (dP - delta) = 0) the absolute error is returned instead."""
    scale = np.abs(ref).max()
    err = np.abs(got - ref).max()
    return err / scale if scale > 1e-6 else err


def compare_bwd(gpu, ref, heads, Hq, Hkv):
    errs = {}
    dq = f64(gpu["dq"])
    errs["dq"] = max(rel_err(dq[:, h], ref["dq"][:, h]) for h in heads)
    kvs = kv_heads_covered(heads, Hq, Hkv)
    for name in ("dk", "dv"):
        g = f64(gpu[name])
        errs[name] = max(rel_err(g[:, x], ref[name][:, x]) for x in kvs)
    return errs


def tensors_for(wl, n_tokens=None):
    return make_tensors(wl, n_tokens)


def oracle_head_job(job):
    """Worker for a spawn pool: the oracle's per-node form for one q head of a named workload,
    optionally restricted to some query nodes; returns only the rows / keys asked for."""
    name, h, nodes, rows = job
    from workloads import make_workload
    wl = make_workload(name)
    t = make_tensors(wl)
    p = oracle.plan(wl.parent, wl.node_len)
    g = h // (wl.Hq // wl.Hkv)
    one = lambda x, i: x[:, i:i + 1].contiguous()          # this head only: [N, 1, d]
    r = oracle.attention_nodes(wl.parent, wl.node_len, one(t["q"], h), one(t["k"], g), one(t["v"], g),
                               one(t["u"], h), heads=[0], p=p, nodes=nodes, theta=wl.theta)
    sel = slice(None) if rows is None else rows
    return dict(h=h, o=r["o"][sel, 0], lse=r["lse"][0, sel], dq=r["dq"][sel, 0], dk=r["dk"][sel, 0],
                dv=r["dv"][sel, 0])


def oracle_heads_parallel(name, heads, nodes=None, rows=None, workers=None):
    import multiprocessing as mp
    ctx = mp.get_context("spawn")
    jobs = [(name, h, nodes, rows) for h in heads]
    with ctx.Pool(workers or min(len(jobs), 8)) as pool:
        return pool.map(oracle_head_job, jobs)
