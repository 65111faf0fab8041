"""The non-allocating backward entry point, called through the C ABI.

tree_attn_bwd_noalloc serves callers that cannot allocate device memory (a host runtime that
owns every allocation, or a path that must not pay cudaMalloc's synchronisation): it takes
its scratch from a fixed 64 MiB array inside the library instead of a caller workspace.
This test compares it, on two calls in a row, with tree_attn_bwd given a PyTorch workspace:
dK and dV bit for bit (both reduce on chip in a fixed order), dQ (fp32 reduce-adds in
arbitrary order, then one rounding to bf16) element by element within one bf16 rounding step,
and all three against the fp64 oracle within the
gradient tolerance of the other tests.  It also checks that an oversized problem is refused
before anything runs.  It is self-contained, so it passes alone in a fresh process
and after the rest of the suite.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import tree_masked_attention_plan_gb300 as tam
from workloads import make_tensors, make_workload

pytestmark = pytest.mark.gpu

GRAD_TOL = 5e-2       # against the fp64 oracle, relative to max|reference|
BF16_STEP = 2.0 ** -7  # relative spacing of bf16 values: two roundings of nearly equal fp32 sums
ORACLE_HEADS = [0, 1, 2, 3]   # one whole kv-head group, so its dK / dV are fully determined


def _noalloc_fn():
    lib = ctypes.CDLL(tam.LIB_PATH)
    fn = lib.tree_attn_bwd_noalloc
    vp, i32, f32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_float
    fn.restype = i32
    fn.argtypes = [ctypes.POINTER(tam.PlanT), vp, vp, vp, vp, vp, vp, i32, i32, i32, f32, f32, vp, vp, vp, vp, vp]
    return fn


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


def _forward(name):
    wl = make_workload(name)
    t = make_tensors(wl)
    dev = torch.device("cuda", 0)
    plan = tam.tree_plan(wl.parent, wl.node_len, device=dev)
    q, k, v, u = (t[x].to(dev) for x in ("q", "k", "v", "u"))
    qr, kr = tam.tree_rope_fwd(plan, q, k, wl.theta)
    o, lse = tam.tree_attn_fwd(plan, qr, kr, v)
    dO = tam.tree_apply_weights(plan, u)
    return wl, plan, qr, kr, v, o, lse, dO, t


def _rel(a, b):
    a, b = a.double(), b.double()
    return ((a - b).abs().max() / b.abs().max()).item()


def test_noalloc_matches_workspace_backward_twice():
    wl, plan, qr, kr, v, o, lse, dO, t = _forward("caterpillar")   # 3456 tokens, 57 MB of scratch
    assert tam.tree_attn_bwd_workspace(plan, wl.Hq, wl.d) <= 64 << 20
    ref = tam.tree_attn_bwd(plan, qr, kr, v, o, lse, dO, rope_theta=wl.theta)
    torch.cuda.synchronize()
    exact = oracle.attention_nodes(wl.parent, wl.node_len, t["q"], t["k"], t["v"], t["u"], heads=ORACLE_HEADS,
                                   theta=wl.theta)
    fn = _noalloc_fn()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for call in range(2):
        status = tam.new_status()
        dq, dk, dv = torch.empty_like(qr), torch.empty_like(kr), torch.empty_like(v)
        rc = fn(plan.ref(), _p(qr), _p(kr), _p(v), _p(o), _p(lse), _p(dO), wl.Hq, wl.Hkv, wl.d, 0.0,
                float(wl.theta), _p(dq), _p(dk), _p(dv), _p(status), stream)
        assert rc == 0, rc
        torch.cuda.synchronize()
        assert status.item() == 0
        assert torch.equal(dk, ref[1]) and torch.equal(dv, ref[2]), "dK / dV differ from the workspace call"
        e_dq = _rel(dq, ref[0])
        a, b = dq.double(), ref[0].double()
        bound = BF16_STEP * torch.maximum(a.abs(), b.abs()) + 1e-6 * b.abs().max()
        assert bool(((a - b).abs() <= bound).all()), f"dQ differs from the workspace call by more than one bf16 step"
        errs = {}
        for name, got, g in (("dq", dq, ORACLE_HEADS), ("dk", dk, [0]), ("dv", dv, [0])):
            a = got.double().cpu().numpy()[:, g]
            b = exact[name][:, g]
            errs[name] = float(np.abs(a - b).max() / np.abs(b).max())
        print(f"call {call}: dq vs workspace call {e_dq:.2e}; vs fp64 oracle {errs}")
        assert max(errs.values()) <= GRAD_TOL


def test_noalloc_rejects_oversized_problem():
    wl = make_workload("rollout32k")                               # needs ~0.5 GB of scratch
    plan = tam.tree_plan(wl.parent, wl.node_len)
    x = torch.zeros(16, dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros(16, dtype=torch.float32, device="cuda")
    status = tam.new_status()
    fn = _noalloc_fn()
    rc = fn(plan.ref(), _p(x), _p(x), _p(x), _p(x), _p(lse), _p(x), wl.Hq, wl.Hkv, wl.d, 0.0, 10000.0,
            _p(x), _p(x), _p(x), _p(status), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == -7                                                 # TREE_ERR_SCRATCH, nothing launched
    torch.cuda.synchronize()
    assert status.item() == 0
