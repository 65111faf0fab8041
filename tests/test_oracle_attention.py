"""Pins for the oracle's attention against formulations it does not share code with.

* a dense N x N mask built by walking parent pointers (section 4.2 of the explainer) with
  torch float64 autograd for the backward and RoPE written as complex rotation;
* the block-diagonal special case against torch's scaled_dot_product_attention (the
  agent-RL tutorial's packing section 14.1: packed == per-sequence causal attention);
* central finite differences of the per-path average loss (section 6.1);
* RoPE closed forms: unit vectors, norm preservation, relative-position invariance;
* the Tree Attention page's associative (max, numerator, denominator) merge against the
  unsplit softmax;
* the leak and permutation properties of section 14.2.
"""
import numpy as np
import pytest
import torch

import oracle
from workloads import caterpillar_tree, random_tree, tiny_tree


def _walk_anc(parent, v):
    out = [v]
    while parent[v] != -1:
        v = parent[v]
        out.append(v)
    return out


def _dense_mask_reference(parent, node_len, q, k, v, u, theta, scale):
    """Packed attention with an explicit N x N mask from parent walks, depth positions from
    parent walks, weights from leaf walks; backward by torch autograd (float64)."""
    parent = list(map(int, parent))
    node_len = list(map(int, node_len))
    n = len(parent)
    # packing order: a stack-based preorder, children ascending (independent of the oracle)
    kids = {i: sorted(c for c in range(n) if parent[c] == i) for i in range(n)}
    order, stack = [], sorted([i for i in range(n) if parent[i] == -1], reverse=True)
    while stack:
        x = stack.pop()
        order.append(x)
        stack.extend(sorted(kids[x], reverse=True))
    tok_node = [x for x in order for _ in range(node_len[x])]
    N = len(tok_node)
    start = {}
    acc = 0
    for x in order:
        start[x] = acc
        acc += node_len[x]
    pos = torch.tensor([sum(node_len[a] for a in _walk_anc(parent, tok_node[t])[1:]) + t - start[tok_node[t]]
                        for t in range(N)], dtype=torch.float64)
    leaves = [x for x in range(n) if not kids[x]]
    g = np.zeros(n)
    for lf in leaves:
        for a in _walk_anc(parent, lf):
            g[a] += 1
    w = torch.tensor([g[tok_node[t]] / len(leaves) for t in range(N)], dtype=torch.float64)
    allowed = torch.zeros(N, N, dtype=torch.bool)
    for i in range(N):
        anc = set(_walk_anc(parent, tok_node[i]))
        for j in range(i + 1):
            allowed[i, j] = tok_node[j] in anc
    Hq, Hkv, d = q.shape[1], k.shape[1], q.shape[2]
    half = d // 2
    inv = theta ** (-(2.0 * torch.arange(half, dtype=torch.float64)) / d)
    rot = torch.polar(torch.ones(N, half, dtype=torch.float64), pos[:, None] * inv[None, :])   # e^{i pos theta_c}

    def crope(x):       # (x_c + i x_{c+d/2}) * e^{i pos theta_c}
        z = torch.complex(x[..., :half], x[..., half:]) * rot[:, None, :]
        return torch.cat([z.real, z.imag], dim=-1)

    qt, kt, vt = (torch.tensor(a).requires_grad_() for a in (q, k, v))
    qr, kr = crope(qt), crope(kt)
    kr = kr.repeat_interleave(Hq // Hkv, dim=1)
    vv = vt.repeat_interleave(Hq // Hkv, dim=1)
    S = torch.einsum("ihc,jhc->hij", qr, kr) * scale
    S = S.masked_fill(~allowed[None], float("-inf"))
    lse = torch.logsumexp(S, dim=-1)
    O = torch.einsum("hij,jhc->ihc", torch.softmax(S, dim=-1), vv)
    loss = (w[:, None, None] * torch.tensor(u) * O).sum()
    loss.backward()
    return dict(o=O.detach().numpy(), lse=lse.detach().numpy(), dq=qt.grad.numpy(),
                dk=kt.grad.numpy(), dv=vt.grad.numpy())


def _inputs(N, Hq, Hkv, d, seed):
    rng = np.random.default_rng(seed)
    return (rng.standard_normal((N, Hq, d)), rng.standard_normal((N, Hkv, d)),
            rng.standard_normal((N, Hkv, d)), rng.standard_normal((N, Hq, d)))


TREES = [tiny_tree(), caterpillar_tree(p=6, T=5, delta=4, a=3)] + [
    random_tree(s, n_nodes=5 + 3 * s, max_len=8, zero_prob=0.2 if s % 2 else 0.0,
                n_roots=1 + (s == 3)) for s in range(5)]


@pytest.mark.parametrize("tree", TREES)
def test_dense_mask_bruteforce(tree):
    parent, node_len = tree
    N = int(np.sum(node_len))
    Hq, Hkv, d = (2, 1, 16) if N > 40 else (4, 2, 8)
    q, k, v, u = _inputs(N, Hq, Hkv, d, seed=N)
    ref = _dense_mask_reference(parent, node_len, q, k, v, u, theta=10000.0, scale=1 / np.sqrt(d))
    got = oracle.attention_paths(parent, node_len, q, k, v, u)
    for key in ("o", "lse", "dq", "dk", "dv"):
        assert np.abs(got[key] - ref[key]).max() < 1e-10, key
    got2 = oracle.attention_nodes(parent, node_len, q, k, v, u, row_chunk=5)
    for key in ("o", "lse", "dq", "dk", "dv"):
        assert np.abs(got2[key] - ref[key]).max() < 1e-10, key


def test_block_diagonal_equals_sdpa():
    """Forest of single-node chains == per-sequence causal attention (library routine)."""
    lens = [5, 17, 1, 9, 12]
    parent = [-1] * len(lens)
    N, Hq, Hkv, d = sum(lens), 4, 2, 16
    q, k, v, u = _inputs(N, Hq, Hkv, d, seed=3)
    got = oracle.attention_paths(parent, lens, q, k, v, u, use_rope=False)
    K = len(lens)
    s = 0
    for L in lens:
        sl = slice(s, s + L)
        qt = torch.tensor(q[sl]).transpose(0, 1).requires_grad_()
        kt = torch.tensor(k[sl]).transpose(0, 1).requires_grad_()
        vt = torch.tensor(v[sl]).transpose(0, 1).requires_grad_()
        o = torch.nn.functional.scaled_dot_product_attention(
            qt, kt.repeat_interleave(2, 0), vt.repeat_interleave(2, 0), is_causal=True)
        (o * torch.tensor(u[sl]).transpose(0, 1) / K).sum().backward()
        assert np.abs(got["o"][sl] - o.detach().transpose(0, 1).numpy()).max() < 1e-10
        assert np.abs(got["dq"][sl] - qt.grad.transpose(0, 1).numpy()).max() < 1e-10
        assert np.abs(got["dk"][sl] - kt.grad.transpose(0, 1).numpy()).max() < 1e-10
        assert np.abs(got["dv"][sl] - vt.grad.transpose(0, 1).numpy()).max() < 1e-10
        s += L


def test_finite_differences():
    """Central differences of L = (1/K) sum_k sum_{t in p_k} <U_t, O_t> (section 6.1)."""
    parent, node_len = tiny_tree()
    node_len = np.array([3, 2, 2, 3, 1, 2])
    N, Hq, Hkv, d = int(node_len.sum()), 2, 1, 8
    q, k, v, u = _inputs(N, Hq, Hkv, d, seed=11)
    plan = oracle.plan(parent, node_len)

    def loss(q_, k_, v_):
        o = oracle.attention_paths(parent, node_len, q_, k_, v_, u, p=plan)["o"]
        tot = 0.0
        for path in plan["paths"]:
            for x in path:
                s = plan["tok_start"][x]
                tot += (u[s:s + node_len[x]] * o[s:s + node_len[x]]).sum()
        return tot / plan["n_paths"]

    got = oracle.attention_paths(parent, node_len, q, k, v, u, p=plan)
    rng = np.random.default_rng(0)
    eps = 1e-6
    for name, arr, gk in (("q", q, "dq"), ("k", k, "dk"), ("v", v, "dv")):
        for _ in range(12):
            idx = tuple(rng.integers(0, s) for s in arr.shape)
            a1, a2 = arr.copy(), arr.copy()
            a1[idx] += eps
            a2[idx] -= eps
            args1 = {"q": (a1, k, v), "k": (q, a1, v), "v": (q, k, a1)}[name]
            args2 = {"q": (a2, k, v), "k": (q, a2, v), "v": (q, k, a2)}[name]
            fd = (loss(*args1) - loss(*args2)) / (2 * eps)
            assert abs(fd - got[gk][idx]) <= 1e-6 * max(1.0, abs(fd)), (name, idx)


def test_rope_closed_forms():
    d, theta = 16, 10000.0
    pos = np.array([0, 1, 7, 1000, 131071])
    for c in range(d // 2):
        e = np.zeros((len(pos), d))
        e[:, c] = 1.0
        r = oracle.rope(e, pos, theta)
        ang = pos * theta ** (-2.0 * c / d)
        assert np.allclose(r[:, c], np.cos(ang), atol=1e-12)
        assert np.allclose(r[:, c + d // 2], np.sin(ang), atol=1e-12)
        r2 = np.delete(r, [c, c + d // 2], axis=1)
        assert np.all(r2 == 0)
    rng = np.random.default_rng(1)
    x = rng.standard_normal((5, 3, d))
    y = rng.standard_normal((5, 3, d))
    rx = oracle.rope(x, pos, theta)
    assert np.allclose(np.linalg.norm(rx, axis=-1), np.linalg.norm(x, axis=-1), atol=1e-12)
    assert np.allclose(oracle.rope(x, np.zeros(5), theta), x)
    assert np.allclose(oracle.rope_transpose(rx, pos, theta), x, atol=1e-12)
    # adjoint: <R x, y> = <x, R^T y>
    assert np.isclose((rx * y).sum(), (x * oracle.rope_transpose(y, pos, theta)).sum())
    # relative position: <R(m) q, R(n) k> depends on m - n only
    q, k = rng.standard_normal((1, d)), rng.standard_normal((1, d))
    for m, n, s in ((5, 2, 40), (100, 100, 7), (3, 9, 1000)):
        a = (oracle.rope(q, [m], theta) * oracle.rope(k, [n], theta)).sum()
        b = (oracle.rope(q, [m + s], theta) * oracle.rope(k, [n + s], theta)).sum()
        assert abs(a - b) < 1e-9


def test_softmax_state_merge_associative():
    rng = np.random.default_rng(5)
    s = rng.standard_normal(37) * 4
    v = rng.standard_normal((37, 6))
    full = oracle.softmax_state(s, v)
    o_ref = np.exp(s - s.max()) / np.exp(s - s.max()).sum() @ v
    lse_ref = np.log(np.exp(s).sum())
    for cut in (1, 10, 36):
        m, n_, d_ = oracle.merge_softmax_state(oracle.softmax_state(s[:cut], v[:cut]),
                                               oracle.softmax_state(s[cut:], v[cut:]))
        assert np.abs(n_ / d_ - o_ref).max() < 1e-12
        assert abs(m + np.log(d_) - lse_ref) < 1e-12
    a, b, c = (oracle.softmax_state(s[x], v[x]) for x in (slice(0, 9), slice(9, 20), slice(20, 37)))
    m1, n1, d1 = oracle.merge_softmax_state(oracle.merge_softmax_state(a, b), c)
    m2, n2, d2 = oracle.merge_softmax_state(a, oracle.merge_softmax_state(c, b))
    assert np.abs(n1 / d1 - n2 / d2).max() < 1e-12 and abs(m1 + np.log(d1) - m2 - np.log(d2)) < 1e-12
    assert np.abs(n1 / d1 - full[1] / full[2]).max() < 1e-12


def _branch_tokens(plan, node_len, nodes):
    out = []
    for x in nodes:
        s = plan["tok_start"][x]
        out += list(range(s, s + node_len[x]))
    return np.array(out, dtype=np.int64)


def test_leak_properties():
    """Section 14.2: a sibling branch, a future child and an ancestor perturbation."""
    parent, node_len = tiny_tree()
    plan = oracle.plan(parent, node_len)
    N, Hq, Hkv, d = 64, 2, 1, 16
    q, k, v, u = _inputs(N, Hq, Hkv, d, seed=9)
    base = oracle.attention_paths(parent, node_len, q, k, v, u, p=plan)
    branch_n1 = _branch_tokens(plan, node_len, [1, 3, 4])
    branch_n2 = _branch_tokens(plan, node_len, [2, 5])
    root = _branch_tokens(plan, node_len, [0])

    def perturbed(tok):
        q2, k2, v2 = q.copy(), k.copy(), v.copy()
        q2[tok] += 1.0
        k2[tok] -= 0.5
        v2[tok] *= 3.0
        return oracle.attention_paths(parent, node_len, q2, k2, v2, u, p=plan)

    r = perturbed(branch_n1)                  # sibling of n2: n2's branch unchanged, bit for bit
    assert np.array_equal(r["o"][branch_n2], base["o"][branch_n2])
    assert np.array_equal(r["lse"][:, branch_n2], base["lse"][:, branch_n2])
    r = perturbed(_branch_tokens(plan, node_len, [3]))   # future child: ancestors + other branches
    keep = np.concatenate([root, _branch_tokens(plan, node_len, [1, 4, 2, 5])])
    assert np.array_equal(r["o"][keep], base["o"][keep])
    r = perturbed(root[:1])                    # ancestor: every descendant changes
    desc = np.concatenate([branch_n1, branch_n2])
    assert np.all(np.abs(r["o"][desc] - base["o"][desc]).max(axis=(1, 2)) > 0)


def test_sibling_order_permutation():
    """Swapping sibling ids (hence their DFS order) leaves positions and per-path outputs unchanged."""
    parent, node_len = tiny_tree()
    # relabel: swap n1 <-> n2 and n3 <-> n5 so n2's branch comes first in DFS
    perm = np.array([0, 2, 1, 5, 4, 3])        # new id of old node
    inv = np.argsort(perm)
    parent2 = np.array([-1 if parent[inv[i]] < 0 else perm[parent[inv[i]]] for i in range(6)])
    len2 = node_len[inv]
    p1, p2 = oracle.plan(parent, node_len), oracle.plan(parent2, len2)
    N, Hq, Hkv, d = 64, 2, 1, 16
    q, k, v, u = _inputs(N, Hq, Hkv, d, seed=2)
    # token t of old node x (offset o) moves to new node perm[x], same offset
    tmap = np.empty(N, dtype=np.int64)
    for x in range(6):
        s1, s2 = p1["tok_start"][x], p2["tok_start"][perm[x]]
        tmap[s1:s1 + node_len[x]] = np.arange(s2, s2 + node_len[x])
    assert np.array_equal(p1["pos"], p2["pos"][tmap])
    qq, kk, vv, uu = (np.empty_like(a) for a in (q, k, v, u))
    for a, b in ((q, qq), (k, kk), (v, vv), (u, uu)):
        b[tmap] = a
    r1 = oracle.attention_paths(parent, node_len, q, k, v, u, p=p1)
    r2 = oracle.attention_paths(parent2, len2, qq, kk, vv, uu, p=p2)
    for key in ("o", "dq", "dk", "dv"):
        assert np.abs(r1[key] - r2[key][tmap]).max() < 1e-12
    assert np.abs(r1["lse"] - r2["lse"][:, tmap]).max() < 1e-12


def test_nodes_formulation_matches_paths_caterpillar():
    """The per-node tree-mask formulation (used for the largest trees) equals the path expansion
    on the full caterpillar workload shape (3456 tokens, 40 paths), one head pair, d = 16."""
    parent, node_len = caterpillar_tree()
    N = int(node_len.sum())
    q, k, v, u = _inputs(N, 2, 1, 16, seed=21)
    plan = oracle.plan(parent, node_len)
    a = oracle.attention_paths(parent, node_len, q, k, v, u, p=plan)
    b = oracle.attention_nodes(parent, node_len, q, k, v, u, p=plan, row_chunk=100)
    for key in ("o", "lse", "dq", "dk", "dv"):
        assert np.abs(a[key] - b[key]).max() < 1e-10, key


def test_nodes_selection_exact_on_selected_leaf():
    """Restricting the per-node form to some query nodes leaves their rows (O, LSE, dQ) and
    the keys only they can see (a leaf's own dK, dV) exactly as in the full computation."""
    parent, node_len = caterpillar_tree(p=20, T=6, delta=9, a=5)
    N = int(node_len.sum())
    q, k, v, u = _inputs(N, 2, 1, 16, seed=4)
    plan = oracle.plan(parent, node_len)
    full = oracle.attention_nodes(parent, node_len, q, k, v, u, p=plan)
    leaves = [2, 12]
    part = oracle.attention_nodes(parent, node_len, q, k, v, u, p=plan, nodes=leaves)
    rows = np.concatenate([np.arange(plan["tok_start"][x], plan["tok_start"][x] + node_len[x]) for x in leaves])
    for key in ("o", "dq"):
        assert np.abs(full[key][rows] - part[key][rows]).max() < 1e-13
    assert np.abs(full["lse"][:, rows] - part["lse"][:, rows]).max() < 1e-13
    for key in ("dk", "dv"):
        assert np.abs(full[key][rows] - part[key][rows]).max() < 1e-13
