"""CPU-side checks of the C ABI: the library builds, loads without a GPU, exports every entry
point include/tree_attn.h declares, and its host-only functions validate trees."""
import ctypes
import os
import re

import numpy as np
import pytest

import oracle
import tree_masked_attention_plan_gb300 as tam
from workloads import CONFIGS, make_workload, random_tree

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(tam.LIB_PATH):
        from tree_masked_attention_plan_gb300 import build_lib
        build_lib.build()
    return ctypes.CDLL(tam.LIB_PATH)


def declared_functions():
    src = open(os.path.join(ROOT, "include", "tree_attn.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[a-z_0-9]+\*?\s+\**(tree_[a-z_0-9]+)\s*\(", src, flags=re.M)))


def test_header_declares_entry_points():
    names = declared_functions()
    for n in ("tree_plan_query", "tree_plan_bind", "tree_plan", "tree_rope_fwd", "tree_attn_fwd",
              "tree_attn_bwd", "tree_attn_bwd_workspace", "tree_strerror", "tree_plan_offset",
              "tree_attn_fwd_gateway", "tree_attn_bwd_gateway", "tree_relay_add"):
        assert n in names


def test_every_declared_symbol_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_plan_query_sizes_match_oracle(lib):
    for name in CONFIGS:
        wl = make_workload(name)
        info = tam.tree_plan_query(wl.parent, wl.node_len)
        p = oracle.plan(wl.parent, wl.node_len)
        assert (info["n_nodes"], info["n_tokens"], info["n_tiles"], info["n_paths"]) == \
            (len(wl.parent), p["n_tokens"], p["n_tiles"], p["n_paths"])
        assert info["max_nnz"] == p["n_tiles"] * (p["n_tiles"] + 1) // 2


@pytest.mark.parametrize("parent,lens", [([0], [3]), ([-1, 5], [1, 1]), ([1, 0], [1, 1]), ([-1, 2, 1], [1, 1, 1]),
                                         ([-1, 0], [1, -1]), ([-1, 0], [0, 0]), ([-1], [2 ** 31 - 1])])
def test_plan_query_rejects(parent, lens):
    if lens == [2 ** 31 - 1]:
        info = tam.tree_plan_query(parent, lens)     # exactly at the limit: accepted
        assert info["n_tokens"] == 2 ** 31 - 1
        with pytest.raises(tam.TreeError):
            tam.tree_plan_query([-1, 0], [2 ** 31 - 1, 1])
        return
    with pytest.raises(tam.TreeError) as e:
        tam.tree_plan_query(parent, lens)
    assert e.value.code == -1


def test_plan_query_agrees_with_oracle_validation():
    for s in range(40):
        rng = np.random.default_rng(s)
        n = int(rng.integers(1, 12))
        parent = rng.integers(-1, n, size=n)
        lens = rng.integers(-1, 4, size=n)
        try:
            oracle.validate_tree(parent, lens)
            ok = True
        except oracle.TreeError:
            ok = False
        try:
            tam.tree_plan_query(parent, lens)
            ok2 = True
        except tam.TreeError:
            ok2 = False
        assert ok == ok2, (parent, lens)


def test_strerror_and_version(lib):
    lib.tree_strerror.restype = ctypes.c_char_p
    for code in (0, -1, -2, -3, -4, -5, -6, 99):
        assert lib.tree_strerror(code)
    assert lib.tree_version() >= 1


def test_bind_rejects_misaligned(lib):
    wl = make_workload("tiny")
    info = tam.PlanInfo()
    par = np.asarray(wl.parent, np.int32)
    nl = np.asarray(wl.node_len, np.int32)
    assert tam._lib().tree_plan_query(par.ctypes.data, nl.ctypes.data, len(par), ctypes.byref(info)) == 0
    c = tam.PlanT()
    assert tam._lib().tree_plan_bind(ctypes.byref(info), ctypes.c_void_p(4096 + 8), ctypes.byref(c)) == -6
    assert tam._lib().tree_plan_bind(ctypes.byref(info), ctypes.c_void_p(4096 * 16), ctypes.byref(c)) == 0
    # carved pointers stay inside the buffer and are 256-byte aligned
    for f in tam.PLAN_PTR_FIELDS:
        off = getattr(c, f) - 4096 * 16
        assert 0 <= off < info.plan_bytes and off % 4 == 0


def test_gateway_entry_points_reject_bad_arguments_without_a_gpu(lib):
    """Argument checks run before any CUDA call."""
    lib.tree_relay_add.restype = ctypes.c_int
    lib.tree_relay_add.argtypes = [ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int,
                                   ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
    assert lib.tree_relay_add(None, 4, None, None, 1, 64, None, None, None) == -6
    lib.tree_plan_offset.restype = ctypes.c_int
    lib.tree_plan_offset.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32,
                                     ctypes.c_void_p, ctypes.c_void_p]
    par = np.array([-1, 0], dtype=np.int32)
    ln = np.array([3, 4], dtype=np.int32)
    plan = ctypes.create_string_buffer(512)
    assert lib.tree_plan_offset(par.ctypes.data, ln.ctypes.data, 2, -1, plan, None) == -6
    assert lib.tree_attn_fwd_gateway(None, None, None, None, None, 1, 1, 64, ctypes.c_float(0.0), None, None,
                                     None, None) != 0


def test_hybrid_entry_points_reject_bad_arguments_without_a_gpu(lib):
    """Shape and pointer checks of the hybrid-layer entry points run before any CUDA call."""
    f = lib.tree_route_states
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p,
                  ctypes.c_void_p]
    buf = ctypes.create_string_buffer(4096)
    a = ctypes.addressof(buf) + (-ctypes.addressof(buf)) % 16
    assert f(a, a, 4, a, 6, a, None) == -2                      # S not a multiple of 4: TREE_ERR_SHAPE
    assert f(None, a, 4, a, 8, a, None) == -6                   # NULL: TREE_ERR_ARG
    assert f(a, a, 4, a + 4, 8, a, None) == -6                  # misaligned
    g = lib.tree_route_states_bwd
    g.restype = ctypes.c_int
    g.argtypes = f.argtypes
    assert g(a, a, 0, a, 8, a, None) == -6
    assert lib.tree_conv1d_fwd(None, None, None, None, None, None, 8, 4, None, None, None) != 0
    assert lib.tree_conv1d_bwd_workspace(None, 8) == 0


def _fake_plan(n_tokens=300, n_paths=2, n_nodes=4):
    """A plan descriptor whose pointers are never dereferenced by the host-side checks."""
    c = tam.PlanT()
    for f in tam.PLAN_PTR_FIELDS:
        setattr(c, f, 4096 * 16)
    c.n_nodes, c.n_tokens, c.n_tiles, c.n_paths = n_nodes, n_tokens, (n_tokens + 127) // 128, n_paths
    return c


def test_loss_and_conv_entry_points_check_shapes_before_any_cuda_call(lib):
    L = tam._lib()
    plan = ctypes.byref(_fake_plan())
    a = 4096 * 64                                     # 16-byte aligned stand-in address
    ce = lambda D, V, chunk, h=a, W=a: L.tree_ce_fwd_bwd(plan, a, a, h, W, a, D, V, chunk, -100, a, a, a, a, a, None,
                                                         None)
    assert ce(200, 1000, 256) == -2                   # D not a multiple of 256
    assert ce(256, 1001, 256) == -2                   # V not a multiple of 8
    assert ce(256, 1000, 100) == -2                   # chunk not a multiple of 128
    assert ce(256, 1000, 256, h=a + 8) == -6          # misaligned
    assert ce(256, 1000, 256, W=None) == -6           # NULL
    conv = lambda C, K, par=a: L.tree_conv1d_fwd(plan, par, a, a, a, None, C, K, a, None, None)
    assert conv(12, 4) == -2 and conv(16, 9) == -2 and conv(16, 0) == -2
    assert conv(16, 4, par=None) == -6
    bwd = L.tree_conv1d_bwd(plan, a, a, a, a, a, 16, 4, None, a, a, None, None, None)
    assert bwd == -6                                  # no workspace
    assert L.tree_diag_gemm(a, a, 7, 8, 8, 0, 0, a, None, None) == -2
    assert L.tree_diag_gemm(None, a, 8, 8, 8, 0, 0, a, None, None) == -6
    assert L.tree_conv1d_fwd(None, a, a, a, a, None, 16, 4, a, None, None) == -6   # no plan


def test_loss_workspace_size_is_host_arithmetic(lib):
    L = tam._lib()
    N = 300
    plan = ctypes.byref(_fake_plan(N))
    small = L.tree_ce_workspace(plan, 256, 1000, 128)
    whole = L.tree_ce_workspace(plan, 256, 1000, 1 << 20)
    assert 0 < small < whole
    assert whole == L.tree_ce_workspace(plan, 256, 1000, N)          # chunks longer than the tree clamp to N
    # the per-chunk logits gradient dominates: growing the chunk by 128 rows adds 128 x V bf16
    assert L.tree_ce_workspace(plan, 256, 1000, 256) - small >= 128 * 1000 * 2
    assert L.tree_ce_workspace(None, 256, 1000, 128) == 0
    assert L.tree_conv1d_bwd_workspace(plan, 64) == N * 64 * 4
