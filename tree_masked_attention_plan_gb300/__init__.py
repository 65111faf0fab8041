"""Python binding of the tree-masked attention library (GB300, sm_103a).

Thin ctypes layer over ``_lib/libtreeattn.so``: it allocates outputs with PyTorch, passes
``data_ptr()`` and the current CUDA stream, and turns status codes into exceptions.  Every
step of the computation runs in the library's CUDA kernels; there is no fallback.  The
functions carry the C entry points' names (``include/tree_attn.h``):

  tree_plan_query, tree_plan (pos_offset -> tree_plan_offset), tree_rope_fwd,
  tree_apply_weights, tree_attn_fwd, tree_attn_bwd_workspace, tree_attn_bwd,
  tree_attn_fwd_gateway, tree_attn_bwd_gateway, tree_relay_add, tree_gather_rows, tree_conv1d_fwd,
  tree_conv1d_bwd_workspace, tree_conv1d_bwd, tree_route_states, tree_route_states_bwd, tree_ce_workspace,
  tree_ce_fwd_bwd, tree_selftest_timeout, tree_set_wait_limit_ns (and diag_gemm -> tree_diag_gemm)

Semantics follow "Tree Training 技术详解" (tingdeliu.github.io): DFS packing (section 3.2),
tree mask (4.2), block table (4.3), depth positions (5), path-count weights (6.2), the
path-averaged next-token loss (6.2, 6.3, 12), hybrid layers (9).
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_lib", "libtreeattn.so")
TILE = 128
MAX_RUNS = 16

TREE_OK = 0
ERROR_NAMES = {-1: "TREE_ERR_INVALID_TREE", -2: "TREE_ERR_SHAPE", -3: "TREE_ERR_ARCH", -4: "TREE_ERR_CUDA",
               -5: "TREE_ERR_TIMEOUT", -6: "TREE_ERR_ARG", -7: "TREE_ERR_SCRATCH"}

_i32, _i64, _vp, _f32 = ctypes.c_int32, ctypes.c_int64, ctypes.c_void_p, ctypes.c_float


class TreeError(RuntimeError):
    def __init__(self, code, where):
        self.code = code
        msg = f"{where}: {ERROR_NAMES.get(code, code)}"
        try:
            msg += f" ({_lib().tree_strerror(code).decode()})"
            if code == -4:
                msg += f": {_lib().tree_last_cuda_error().decode()}"
        except Exception:  # pragma: no cover - message decoration only
            pass
        super().__init__(msg)


class PlanInfo(ctypes.Structure):
    _fields_ = [("n_nodes", _i32), ("n_tokens", _i32), ("n_tiles", _i32), ("n_paths", _i32),
                ("max_nnz", _i64), ("plan_bytes", _i64)]


PLAN_PTR_FIELDS = ["order", "dfs_in", "dfs_out", "tok_start", "depth_off", "leaves", "dfs_tok_start", "sub_end",
                   "tok_node", "pos", "g", "tok_in", "tok_out", "hi", "w", "tile_class", "row_ptr", "row_idx",
                   "col_ptr", "col_idx", "row_order", "col_order", "tile_hi_min", "tile_hi_max", "tile_runs",
                   "tile_nruns", "counts"]


class PlanT(ctypes.Structure):
    _fields_ = [(f, _vp) for f in PLAN_PTR_FIELDS] + [("n_nodes", _i32), ("n_tokens", _i32),
                                                      ("n_tiles", _i32), ("n_paths", _i32)]


class Gateway(ctypes.Structure):
    _fields_ = [("k", _vp), ("v", _vp), ("len", _i32)]


_LIB = None


def _lib():
    """Load the in-tree library; fails loudly when it has not been built."""
    global _LIB
    if _LIB is not None:
        return _LIB
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is missing: build it with "
                          "`python -m tree_masked_attention_plan_gb300.build_lib`")
    lib = ctypes.CDLL(LIB_PATH)
    P = ctypes.POINTER
    sig = {
        "tree_plan_query": (_i32, [_vp, _vp, _i32, P(PlanInfo)]),
        "tree_plan_bind": (_i32, [P(PlanInfo), _vp, P(PlanT)]),
        "tree_plan_nodes": (_i32, [_vp, _vp, _i32, _vp]),
        "tree_plan": (_i32, [_vp, _vp, _i32, P(PlanT), _vp]),
        "tree_plan_offset": (_i32, [_vp, _vp, _i32, _i32, P(PlanT), _vp]),
        "tree_rope_fwd": (_i32, [P(PlanT), _vp, _vp, _vp, _vp, _i32, _i32, _i32, _f32, _vp]),
        "tree_apply_weights": (_i32, [P(PlanT), _vp, _vp, _i32, _i32, _vp]),
        "tree_attn_fwd": (_i32, [P(PlanT), _vp, _vp, _vp, _i32, _i32, _i32, _f32, _vp, _vp, _vp, _vp]),
        "tree_attn_bwd_workspace": (ctypes.c_size_t, [P(PlanT), _i32, _i32]),
        "tree_attn_bwd": (_i32, [P(PlanT), _vp, _vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32, _f32, _f32, _vp,
                                 _vp, _vp, _vp, _vp, _vp]),
        "tree_attn_bwd_weighted": (_i32, [P(PlanT), _vp, _vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32, _f32, _f32,
                                          _vp, _vp, _vp, _vp, _vp, _vp]),
        "tree_attn_fwd_gateway": (_i32, [P(PlanT), P(Gateway), _vp, _vp, _vp, _i32, _i32, _i32, _f32, _vp, _vp,
                                         _vp, _vp]),
        "tree_attn_bwd_gateway": (_i32, [P(PlanT), P(Gateway), _vp, _vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32,
                                         _f32, _f32, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp]),
        "tree_relay_add": (_i32, [_vp, _i32, _vp, _vp, _i32, _i32, _vp, _vp, _vp]),
        "tree_gather_rows": (_i32, [_vp, _i32, _vp, _vp, _i32, _vp]),
        "tree_conv1d_fwd": (_i32, [P(PlanT), _vp, _vp, _vp, _vp, _vp, _i32, _i32, _vp, _vp, _vp]),
        "tree_conv1d_bwd_workspace": (ctypes.c_size_t, [P(PlanT), _i32]),
        "tree_conv1d_bwd": (_i32, [P(PlanT), _vp, _vp, _vp, _vp, _vp, _i32, _i32, _vp, _vp, _vp, _vp, _vp, _vp]),
        "tree_route_states": (_i32, [_vp, _vp, _i32, _vp, _i32, _vp, _vp]),
        "tree_route_states_bwd": (_i32, [_vp, _vp, _i32, _vp, _i32, _vp, _vp]),
        "tree_ce_workspace": (ctypes.c_size_t, [P(PlanT), _i32, _i32, _i32]),
        "tree_ce_fwd_bwd": (_i32, [P(PlanT), _vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32, _i32, _vp, _vp, _vp, _vp,
                                   _vp, _vp, _vp]),
        "tree_diag_gemm": (_i32, [_vp, _vp, _i32, _i32, _i32, _i32, _i32, _vp, _vp, _vp]),
        "tree_set_wait_limit_ns": (_i32, [_i64]),
        "tree_set_bwd_split": (_i32, [_i32]),
        "tree_set_fwd_split": (_i32, [_i32]),
        "tree_set_timing_events": (_i32, [ctypes.POINTER(_vp), _i32]),
        "tree_selftest_timeout": (_i32, [_vp, _i64, _vp]),
        "tree_strerror": (ctypes.c_char_p, [_i32]),
        "tree_last_cuda_error": (ctypes.c_char_p, []),
        "tree_version": (_i32, []),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _LIB = lib
    return lib


def _check(code, where):
    if code != TREE_OK:
        raise TreeError(code, where)


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def _host_i32(a):
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32))


def tree_plan_query(parent, node_len) -> dict:
    """Validate a tree and return its sizes (host only)."""
    par, nl = _host_i32(parent), _host_i32(node_len)
    if par.shape != nl.shape:
        raise ValueError("parent and node_len differ in length")
    info = PlanInfo()
    _check(_lib().tree_plan_query(par.ctypes.data, nl.ctypes.data, len(par), ctypes.byref(info)),
           "tree_plan_query")
    return {f: getattr(info, f) for f, _ in PlanInfo._fields_}


NODE_FIELDS = ["order", "dfs_in", "dfs_out", "tok_start", "depth_off", "leaves", "dfs_tok_start", "sub_end"]


def tree_plan_nodes(parent, node_len) -> dict:
    """The plan's per-node arrays (depth-first order, intervals, token starts, depth offsets,
    leaf counts, subtree ends) from the library's host pass, as int64 NumPy arrays by name."""
    par, nl = _host_i32(parent), _host_i32(node_len)
    if par.shape != nl.shape:
        raise ValueError("parent and node_len differ in length")
    out = np.empty(8 * len(par), dtype=np.int32)
    _check(_lib().tree_plan_nodes(par.ctypes.data, nl.ctypes.data, len(par), out.ctypes.data), "tree_plan_nodes")
    return {f: out[i * len(par):(i + 1) * len(par)].astype(np.int64) for i, f in enumerate(NODE_FIELDS)}


@dataclass
class TreePlan:
    """A plan resident in device memory (one buffer) plus its C descriptor."""
    info: PlanInfo
    buf: torch.Tensor
    c: PlanT
    device: torch.device

    @property
    def n_tokens(self):
        return self.info.n_tokens

    @property
    def n_tiles(self):
        return self.info.n_tiles

    @property
    def n_pad(self):
        return self.info.n_tiles * TILE

    @property
    def n_paths(self):
        return self.info.n_paths

    def ref(self):
        return ctypes.byref(self.c)

    def arrays(self) -> dict:
        """Device tensor views of every plan array (for inspection and tests)."""
        n, Np, T, nnz = self.info.n_nodes, self.n_pad, self.n_tiles, self.info.max_nnz
        sizes = dict(order=n, dfs_in=n, dfs_out=n, tok_start=n, depth_off=n, leaves=n, dfs_tok_start=n,
                     sub_end=n, tok_node=Np, pos=Np, g=Np, tok_in=Np, tok_out=Np, hi=Np, w=Np,
                     tile_class=T * T, row_ptr=T + 1, row_idx=nnz, col_ptr=T + 1, col_idx=nnz, row_order=T,
                     col_order=T, tile_hi_min=T, tile_hi_max=T, tile_runs=T * MAX_RUNS * 4, tile_nruns=T, counts=4)
        base = self.buf.data_ptr()
        out = {}
        for f in PLAN_PTR_FIELDS:
            off = getattr(self.c, f) - base
            if f == "tile_class":
                out[f] = self.buf[off:off + sizes[f]]
            else:
                view = self.buf[off:off + 4 * sizes[f]]
                out[f] = view.view(torch.float32 if f == "w" else torch.int32)
        return out


def tree_plan(parent, node_len, device=None, stream=None, pos_offset=0) -> TreePlan:
    """Build the plan of a tree on the GPU (DFS order, intervals, positions, g, w, tile table).
    pos_offset > 0: the tree is a partition below a gateway of that many tokens (positions
    continue from it; tree_plan_offset)."""
    par, nl = _host_i32(parent), _host_i32(node_len)
    if par.shape != nl.shape:
        raise ValueError("parent and node_len differ in length")
    lib = _lib()
    info = PlanInfo()
    _check(lib.tree_plan_query(par.ctypes.data, nl.ctypes.data, len(par), ctypes.byref(info)), "tree_plan_query")
    dev = torch.device(device) if device is not None else torch.device("cuda", torch.cuda.current_device())
    buf = torch.empty(int(info.plan_bytes), dtype=torch.uint8, device=dev)
    c = PlanT()
    _check(lib.tree_plan_bind(ctypes.byref(info), _ptr(buf), ctypes.byref(c)), "tree_plan_bind")
    with torch.cuda.device(dev):
        if pos_offset:
            _check(lib.tree_plan_offset(par.ctypes.data, nl.ctypes.data, len(par), int(pos_offset), ctypes.byref(c),
                                        _stream(stream)), "tree_plan_offset")
        else:
            _check(lib.tree_plan(par.ctypes.data, nl.ctypes.data, len(par), ctypes.byref(c), _stream(stream)),
                   "tree_plan")
    return TreePlan(info=info, buf=buf, c=c, device=dev)


def _need(t, shape, dtype, name):
    if t.dtype != dtype or tuple(t.shape) != tuple(shape) or not t.is_contiguous() or not t.is_cuda:
        raise ValueError(f"{name}: expected contiguous CUDA {dtype} {tuple(shape)}, got {t.dtype} "
                         f"{tuple(t.shape)} contiguous={t.is_contiguous()} cuda={t.is_cuda}")


def _heads(plan, q, k):
    N = plan.n_tokens
    if q.dim() != 3 or k.dim() != 3:
        raise ValueError("q, k must be [N, heads, d]")
    Hq, d = q.shape[1], q.shape[2]
    Hkv = k.shape[1]
    _need(q, (N, Hq, d), torch.bfloat16, "q")
    _need(k, (N, Hkv, d), torch.bfloat16, "k")
    return Hq, Hkv, d


def tree_rope_fwd(plan: TreePlan, q, k, theta=10000.0, qr=None, kr=None, stream=None):
    """Rotate-half RoPE at depth positions: returns (qr, kr); pass qr=q, kr=k for in place."""
    Hq, Hkv, d = _heads(plan, q, k)
    qr = torch.empty_like(q) if qr is None else qr
    kr = torch.empty_like(k) if kr is None else kr
    _check(_lib().tree_rope_fwd(plan.ref(), _ptr(q), _ptr(k), _ptr(qr), _ptr(kr), Hq, Hkv, d, float(theta),
                                _stream(stream)), "tree_rope_fwd")
    return qr, kr


def tree_apply_weights(plan: TreePlan, u, out=None, stream=None):
    """dO = (g_t / K) * U_t for u [N, H, d] bf16."""
    N, H, d = u.shape
    _need(u, (plan.n_tokens, H, d), torch.bfloat16, "u")
    out = torch.empty_like(u) if out is None else out
    _check(_lib().tree_apply_weights(plan.ref(), _ptr(u), _ptr(out), H, d, _stream(stream)), "tree_apply_weights")
    return out


def tree_attn_fwd(plan: TreePlan, q, k, v, scale=0.0, o=None, lse=None, status=None, stream=None):
    """Tree-masked attention forward: returns (o [N,Hq,d] bf16, lse [Hq, N_pad] fp32)."""
    Hq, Hkv, d = _heads(plan, q, k)
    _need(v, k.shape, torch.bfloat16, "v")
    o = torch.empty_like(q) if o is None else o
    lse = torch.empty(Hq, plan.n_pad, dtype=torch.float32, device=q.device) if lse is None else lse
    _need(lse, (Hq, plan.n_pad), torch.float32, "lse")
    _check(_lib().tree_attn_fwd(plan.ref(), _ptr(q), _ptr(k), _ptr(v), Hq, Hkv, d, float(scale), _ptr(o), _ptr(lse),
                                _ptr(status), _stream(stream)), "tree_attn_fwd")
    return o, lse


def tree_attn_bwd_workspace(plan: TreePlan, Hq: int, d: int) -> int:
    return int(_lib().tree_attn_bwd_workspace(plan.ref(), Hq, d))


def tree_attn_bwd(plan: TreePlan, q, k, v, o, lse, dO, scale=0.0, rope_theta=10000.0, workspace=None,
                  dq=None, dk=None, dv=None, status=None, stream=None):
    """Backward: returns (dq, dk, dv); with rope_theta > 0 dq/dk are w.r.t. the un-rotated q, k."""
    Hq, Hkv, d = _heads(plan, q, k)
    _need(v, k.shape, torch.bfloat16, "v")
    _need(o, q.shape, torch.bfloat16, "o")
    _need(dO, q.shape, torch.bfloat16, "dO")
    _need(lse, (Hq, plan.n_pad), torch.float32, "lse")
    if workspace is None:
        workspace = torch.empty(tree_attn_bwd_workspace(plan, Hq, d), dtype=torch.uint8, device=q.device)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    _check(_lib().tree_attn_bwd(plan.ref(), _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dO), Hq, Hkv, d,
                                float(scale), float(rope_theta), _ptr(workspace), _ptr(dq), _ptr(dk), _ptr(dv),
                                _ptr(status), _stream(stream)), "tree_attn_bwd")
    return dq, dk, dv


def tree_attn_bwd_weighted(plan: TreePlan, q, k, v, o, lse, u, scale=0.0, rope_theta=10000.0, workspace=None,
                           dq=None, dk=None, dv=None, status=None, stream=None):
    """Backward for dO = w U with the plan's weights w = g/K applied inside (no dO is formed):
    returns (dq, dk, dv) as tree_attn_bwd(plan, ..., tree_apply_weights(plan, u)) does."""
    Hq, Hkv, d = _heads(plan, q, k)
    _need(v, k.shape, torch.bfloat16, "v")
    _need(o, q.shape, torch.bfloat16, "o")
    _need(u, q.shape, torch.bfloat16, "u")
    _need(lse, (Hq, plan.n_pad), torch.float32, "lse")
    if workspace is None:
        workspace = torch.empty(tree_attn_bwd_workspace(plan, Hq, d), dtype=torch.uint8, device=q.device)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    _check(_lib().tree_attn_bwd_weighted(plan.ref(), _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(u), Hq, Hkv,
                                         d, float(scale), float(rope_theta), _ptr(workspace), _ptr(dq), _ptr(dk),
                                         _ptr(dv), _ptr(status), _stream(stream)), "tree_attn_bwd_weighted")
    return dq, dk, dv


def tree_set_timing_events(events):
    """Register torch.cuda.Event objects (up to 4, enable_timing=True) that tree_attn_bwd records
    around its kernels: before delta, before dK/dV, after dK/dV, after dQ finalize.  [] clears."""
    for e in events:                       # torch creates the CUDA event on first record
        if not e.cuda_event:
            e.record()
    arr = (_vp * 4)(*[ctypes.c_void_p(e.cuda_event) for e in events])
    _check(_lib().tree_set_timing_events(arr, len(events)), "tree_set_timing_events")


def tree_set_bwd_split(split: int = 0):
    """CTAs per key-tile column in the backward: 0 automatic (default), or 1, 2, 4 forced."""
    _check(_lib().tree_set_bwd_split(int(split)), "tree_set_bwd_split")


def tree_set_fwd_split(split: int = 0):
    """CTAs per query-tile row in the forward (split-KV): 0 automatic (default), or 1, 2, 4."""
    _check(_lib().tree_set_fwd_split(int(split)), "tree_set_fwd_split")


def tree_set_wait_limit_ns(ns: int):
    _check(_lib().tree_set_wait_limit_ns(int(ns)), "tree_set_wait_limit_ns")


def tree_selftest_timeout(status, ns: int = 1_000_000, stream=None):
    _check(_lib().tree_selftest_timeout(_ptr(status), int(ns), _stream(stream)), "tree_selftest_timeout")


def new_status(device=None):
    """A zeroed int32 device status word for the kernels' error reports."""
    return torch.zeros(1, dtype=torch.int32, device=device or "cuda")


def check_status(status, where="device"):
    """Raise TreeError if a kernel stored an error code in `status` (synchronizes)."""
    code = int(status.item())
    if code != TREE_OK:
        raise TreeError(code, where)


__all__ = ["TreeError", "TreePlan", "tree_plan_query", "tree_plan_nodes", "tree_plan", "tree_rope_fwd", "tree_apply_weights",
           "tree_attn_fwd", "tree_attn_bwd_workspace", "tree_attn_bwd", "tree_attn_bwd_weighted", "tree_set_wait_limit_ns", "tree_set_bwd_split", "tree_set_fwd_split",
           "tree_selftest_timeout", "tree_set_timing_events", "new_status", "check_status", "LIB_PATH", "TILE"]


def _gateway(k_gw, v_gw, Hkv, d):
    if k_gw.dim() != 3:
        raise ValueError("k_gw must be [len, Hkv, d]")
    A = k_gw.shape[0]
    _need(k_gw, (A, Hkv, d), torch.bfloat16, "k_gw")
    _need(v_gw, (A, Hkv, d), torch.bfloat16, "v_gw")
    return Gateway(k=_ptr(k_gw), v=_ptr(v_gw), len=A)


def tree_attn_fwd_gateway(plan: TreePlan, k_gw, v_gw, q, k, v, scale=0.0, o=None, lse=None, status=None,
                          stream=None):
    """Forward of a partition below a gateway (ancestor K/V [len, Hkv, d], rotated, root first)."""
    Hq, Hkv, d = _heads(plan, q, k)
    _need(v, k.shape, torch.bfloat16, "v")
    gw = _gateway(k_gw, v_gw, Hkv, d)
    o = torch.empty_like(q) if o is None else o
    lse = torch.empty(Hq, plan.n_pad, dtype=torch.float32, device=q.device) if lse is None else lse
    _need(lse, (Hq, plan.n_pad), torch.float32, "lse")
    _check(_lib().tree_attn_fwd_gateway(plan.ref(), ctypes.byref(gw), _ptr(q), _ptr(k), _ptr(v), Hq, Hkv, d,
                                        float(scale), _ptr(o), _ptr(lse), _ptr(status), _stream(stream)),
           "tree_attn_fwd_gateway")
    return o, lse


def tree_attn_bwd_gateway(plan: TreePlan, k_gw, v_gw, q, k, v, o, lse, dO, dk_gw, dv_gw, scale=0.0,
                          rope_theta=10000.0, workspace=None, dq=None, dk=None, dv=None, status=None,
                          stream=None):
    """Backward of a partition below a gateway: returns (dq, dk, dv) and ADDS the gateway keys'
    gradients from this partition into the fp32 accumulators dk_gw, dv_gw [len, Hkv, d]."""
    Hq, Hkv, d = _heads(plan, q, k)
    _need(v, k.shape, torch.bfloat16, "v")
    _need(o, q.shape, torch.bfloat16, "o")
    _need(dO, q.shape, torch.bfloat16, "dO")
    _need(lse, (Hq, plan.n_pad), torch.float32, "lse")
    gw = _gateway(k_gw, v_gw, Hkv, d)
    _need(dk_gw, tuple(k_gw.shape), torch.float32, "dk_gw")
    _need(dv_gw, tuple(k_gw.shape), torch.float32, "dv_gw")
    if workspace is None:
        workspace = torch.empty(tree_attn_bwd_workspace(plan, Hq, d), dtype=torch.uint8, device=q.device)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    _check(_lib().tree_attn_bwd_gateway(plan.ref(), ctypes.byref(gw), _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse),
                                        _ptr(dO), Hq, Hkv, d, float(scale), float(rope_theta), _ptr(workspace),
                                        _ptr(dq), _ptr(dk), _ptr(dv), _ptr(dk_gw), _ptr(dv_gw), _ptr(status),
                                        _stream(stream)), "tree_attn_bwd_gateway")
    return dq, dk, dv


def tree_relay_add(rows, dk_gw, dv_gw, dk, dv, stream=None):
    """dk[rows[r]] += dk_gw[r] (and dv), fp32 sum rounded once to bf16; rows int32 CUDA [len]."""
    A, Hkv, d = dk_gw.shape
    _need(rows, (A,), torch.int32, "rows")
    _need(dv_gw, (A, Hkv, d), torch.float32, "dv_gw")
    _need(dk, (dk.shape[0], Hkv, d), torch.bfloat16, "dk")
    _need(dv, tuple(dk.shape), torch.bfloat16, "dv")
    _check(_lib().tree_relay_add(_ptr(rows), A, _ptr(dk_gw), _ptr(dv_gw), Hkv, d, _ptr(dk), _ptr(dv),
                                 _stream(stream)), "tree_relay_add")


def tree_gather_rows(rows, src, out=None, stream=None):
    """out[r] = src[rows[r]] for bf16 src [M, ...]; rows int32 CUDA [n]."""
    n = rows.shape[0]
    _need(rows, (n,), torch.int32, "rows")
    if not (src.is_cuda and src.is_contiguous() and src.dtype == torch.bfloat16):
        raise ValueError("src: expected contiguous CUDA bf16")
    row_elems = src[0].numel()
    out = torch.empty((n,) + tuple(src.shape[1:]), dtype=src.dtype, device=src.device) if out is None else out
    _need(out, (n,) + tuple(src.shape[1:]), torch.bfloat16, "out")
    _check(_lib().tree_gather_rows(_ptr(rows), n, _ptr(src), _ptr(out), row_elems, _stream(stream)),
           "tree_gather_rows")
    return out


def tree_arrays(parent, node_len, device):
    """The tree as device int32 arrays (parent, node_len), as the hybrid-layer entry points take it."""
    return (torch.as_tensor(_host_i32(parent), device=device), torch.as_tensor(_host_i32(node_len), device=device))


def tree_conv1d_fwd(plan: TreePlan, tree, x, w, bias=None, out=None, status=None, stream=None):
    """Causal depthwise convolution along root paths: x [N, C] bf16, w [K, C] fp32, bias [C] fp32."""
    parent, node_len = tree
    N, C = x.shape
    K = w.shape[0]
    _need(x, (plan.n_tokens, C), torch.bfloat16, "x")
    _need(w, (K, C), torch.float32, "w")
    if bias is not None:
        _need(bias, (C,), torch.float32, "bias")
    out = torch.empty_like(x) if out is None else out
    _check(_lib().tree_conv1d_fwd(plan.ref(), _ptr(parent), _ptr(node_len), _ptr(x), _ptr(w), _ptr(bias), C, K,
                                  _ptr(out), _ptr(status), _stream(stream)), "tree_conv1d_fwd")
    return out


def tree_conv1d_bwd_workspace(plan: TreePlan, C):
    """Bytes of workspace tree_conv1d_bwd needs for C channels."""
    return int(_lib().tree_conv1d_bwd_workspace(plan.ref(), C))


def tree_conv1d_bwd(plan: TreePlan, tree, x, w, dy, with_bias=False, workspace=None, status=None, stream=None):
    """Backward: returns (dx bf16 [N, C], dw fp32 [K, C], dbias fp32 [C] or None)."""
    parent, node_len = tree
    N, C = x.shape
    K = w.shape[0]
    _need(x, (plan.n_tokens, C), torch.bfloat16, "x")
    _need(dy, (plan.n_tokens, C), torch.bfloat16, "dy")
    _need(w, (K, C), torch.float32, "w")
    if workspace is None:
        workspace = torch.empty(tree_conv1d_bwd_workspace(plan, C), dtype=torch.uint8, device=x.device)
    dx = torch.empty_like(x)
    dw = torch.empty_like(w)
    db = torch.empty(C, dtype=torch.float32, device=x.device) if with_bias else None
    _check(_lib().tree_conv1d_bwd(plan.ref(), _ptr(parent), _ptr(node_len), _ptr(x), _ptr(w), _ptr(dy), C, K,
                                  _ptr(workspace), _ptr(dx), _ptr(dw), _ptr(db), _ptr(status), _stream(stream)),
           "tree_conv1d_bwd")
    return dx, dw, db


def tree_route_states(tree, final_states, stream=None):
    """init[v] = final[nearest ancestor of v holding tokens] (zeros for roots); fp32 [n_nodes, S]."""
    parent, node_len = tree
    n, S = final_states.shape
    _need(final_states, (parent.shape[0], S), torch.float32, "final_states")
    init = torch.empty_like(final_states)
    _check(_lib().tree_route_states(_ptr(parent), _ptr(node_len), n, _ptr(final_states), S, _ptr(init),
                                    _stream(stream)), "tree_route_states")
    return init


def tree_route_states_bwd(tree, d_init, d_final=None, stream=None):
    """d_final[ancestor(v)] += d_init[v]; returns d_final (zeros first when not given)."""
    parent, node_len = tree
    n, S = d_init.shape
    _need(d_init, (parent.shape[0], S), torch.float32, "d_init")
    d_final = torch.zeros_like(d_init) if d_final is None else d_final
    _check(_lib().tree_route_states_bwd(_ptr(parent), _ptr(node_len), n, _ptr(d_init), S, _ptr(d_final),
                                        _stream(stream)), "tree_route_states_bwd")
    return d_final


def tree_ce_workspace(plan: TreePlan, D, V, chunk):
    """Bytes of workspace tree_ce_fwd_bwd needs."""
    return int(_lib().tree_ce_workspace(plan.ref(), D, V, chunk))


def tree_ce_fwd_bwd(plan: TreePlan, tree, h, W, labels, chunk=8192, ignore_index=-100, workspace=None, out=None,
                    status=None, stream=None):
    """Path-averaged next-token cross-entropy fused with the vocabulary projection.
    h [N, D] bf16, W [V, D] bf16, labels [N] int32.  Returns (loss [1] fp32, lse [N] fp32,
    dh [N, D] bf16, dW [V, D] fp32); `out` may supply those four tensors."""
    parent, node_len = tree
    N, D = h.shape
    V = W.shape[0]
    _need(h, (plan.n_tokens, D), torch.bfloat16, "h")
    _need(W, (V, D), torch.bfloat16, "W")
    _need(labels, (plan.n_tokens,), torch.int32, "labels")
    if workspace is None:
        workspace = torch.empty(tree_ce_workspace(plan, D, V, chunk), dtype=torch.uint8, device=h.device)
    if out is None:
        out = (torch.empty(1, dtype=torch.float32, device=h.device),
               torch.empty(N, dtype=torch.float32, device=h.device), torch.empty_like(h),
               torch.empty(V, D, dtype=torch.float32, device=h.device))
    loss, lse, dh, dW = out
    _check(_lib().tree_ce_fwd_bwd(plan.ref(), _ptr(parent), _ptr(node_len), _ptr(h), _ptr(W), _ptr(labels), D, V,
                                  chunk, ignore_index, _ptr(workspace), _ptr(loss), _ptr(lse), _ptr(dh), _ptr(dW),
                                  _ptr(status), _stream(stream)), "tree_ce_fwd_bwd")
    return loss, lse, dh, dW


def diag_gemm(A, B, M, N, K, a_mn, b_mn, status=None, stream=None):
    """C [M, N] fp32 = op(A) op(B)^T on the library's GEMM kernel (a_mn: A is [K, M]; b_mn: B is [K, N])."""
    C = torch.empty(M, N, dtype=torch.float32, device=A.device)
    _check(_lib().tree_diag_gemm(_ptr(A), _ptr(B), M, N, K, int(a_mn), int(b_mn), _ptr(C), _ptr(status),
                                 _stream(stream)), "tree_diag_gemm")
    return C
