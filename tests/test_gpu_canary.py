"""Out-of-bounds write checks without a sanitizer: every buffer the library writes is placed
between guard regions filled with a canary byte, and the payload itself is pre-filled with
the canary.  After plan, RoPE, forward, loss weights and backward:

* every guard byte before and after O, LSE, dQ, dK, dV, the rotated Q/K, the weighted dO, the
  plan buffer and the backward workspace is unchanged (nothing writes past a buffer's end or
  before its start, including the ragged last tile's rows >= N);
* every 16-byte unit of the token-major outputs was written (no leftover canary unit);
* LSE padding columns [N, N_pad) hold the documented 0.

Run on small ragged trees (N not a multiple of 128, tiles with many node runs, a forest) at
d = 64 and 128."""
import ctypes

import numpy as np
import pytest
import torch

import tree_masked_attention_plan_gb300 as tam
from workloads import make_tensors, random_tree
from workloads.trees import Workload

pytestmark = pytest.mark.gpu

CANARY = 0xA5
GUARD = 4096           # bytes on each side (keeps the payload's alignment)


class Guarded:
    def __init__(self, shape, dtype, dev):
        n = int(np.prod(shape)) * torch.tensor([], dtype=dtype).element_size()
        self.n = n
        self.raw = torch.full((GUARD + n + GUARD,), CANARY, dtype=torch.uint8, device=dev)
        self.t = self.raw[GUARD:GUARD + n].view(dtype).view(*shape)

    def guards_intact(self):
        return bool((self.raw[:GUARD] == CANARY).all()) and bool((self.raw[GUARD + self.n:] == CANARY).all())

    def units_written(self):
        """No 16-byte unit of the payload is still entirely canary."""
        u = self.raw[GUARD:GUARD + self.n].view(-1, 16)
        return not bool((u == CANARY).all(dim=1).any())


def _plan_into(parent, lens, dev):
    lib = tam._lib()
    par, nl = tam._host_i32(parent), tam._host_i32(lens)
    info = tam.PlanInfo()
    tam._check(lib.tree_plan_query(par.ctypes.data, nl.ctypes.data, len(par), ctypes.byref(info)), "query")
    g = Guarded((int(info.plan_bytes),), torch.uint8, dev)
    c = tam.PlanT()
    tam._check(lib.tree_plan_bind(ctypes.byref(info), tam._ptr(g.t), ctypes.byref(c)), "bind")
    tam._check(lib.tree_plan(par.ctypes.data, nl.ctypes.data, len(par), ctypes.byref(c), tam._stream()), "plan")
    return tam.TreePlan(info=info, buf=g.t, c=c, device=dev), g


CASES = [("ragged_d128", random_tree(31, 15, max_len=70), 4, 2, 128),
         ("tiny_nodes_d64", random_tree(32, 200, max_len=5, zero_prob=0.1), 2, 1, 64),
         ("forest_d128", random_tree(33, 12, max_len=100, n_roots=4), 2, 2, 128),
         ("one_token_d64", (np.array([-1]), np.array([1])), 1, 1, 64)]


@pytest.mark.parametrize("name,tree,Hq,Hkv,d", CASES, ids=[c[0] for c in CASES])
def test_no_write_outside_buffers(name, tree, Hq, Hkv, d):
    dev = torch.device("cuda", 0)
    wl = Workload(name=name, parent=np.asarray(tree[0], np.int32), node_len=np.asarray(tree[1], np.int32),
                  Hq=Hq, Hkv=Hkv, d=d)
    N = wl.n_tokens
    t = make_tensors(wl)
    q, k, v, u = (t[x].to(dev) for x in ("q", "k", "v", "u"))
    plan, gplan = _plan_into(wl.parent, wl.node_len, dev)
    Np = plan.n_pad
    bufs = {name_: Guarded(shape, dt, dev) for name_, shape, dt in (
        ("qr", (N, Hq, d), torch.bfloat16), ("kr", (N, Hkv, d), torch.bfloat16),
        ("o", (N, Hq, d), torch.bfloat16), ("lse", (Hq, Np), torch.float32), ("dO", (N, Hq, d), torch.bfloat16),
        ("dq", (N, Hq, d), torch.bfloat16), ("dk", (N, Hkv, d), torch.bfloat16), ("dv", (N, Hkv, d), torch.bfloat16),
        ("ws", (tam.tree_attn_bwd_workspace(plan, Hq, d),), torch.uint8))}
    b = {x: g.t for x, g in bufs.items()}
    status = tam.new_status(dev)
    tam.tree_rope_fwd(plan, q, k, 10000.0, qr=b["qr"], kr=b["kr"])
    tam.tree_attn_fwd(plan, b["qr"], b["kr"], v, o=b["o"], lse=b["lse"], status=status)
    tam.tree_apply_weights(plan, u, out=b["dO"])
    tam.tree_attn_bwd(plan, b["qr"], b["kr"], v, b["o"], b["lse"], b["dO"], rope_theta=10000.0, workspace=b["ws"],
                      dq=b["dq"], dk=b["dk"], dv=b["dv"], status=status)
    torch.cuda.synchronize()
    tam.check_status(status, name)
    assert gplan.guards_intact(), "plan buffer"
    for x, g in bufs.items():
        assert g.guards_intact(), f"{x}: a guard byte changed"
    for x in ("qr", "kr", "o", "dO", "dq", "dk", "dv"):
        assert bufs[x].units_written(), f"{x}: some 16-byte unit was never written"
    assert bool((b["lse"][:, N:] == 0).all()), "LSE padding"
    assert bool(torch.isfinite(b["lse"][:, :N]).all())
