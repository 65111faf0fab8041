"""fp64 attention oracle: path-expanded causal attention forward + backward (TEST INFRASTRUCTURE ONLY).

Definition (from "Tree Training 技术详解", tingdeliu.github.io):
  * section 3.2 / 6.1 - the baseline runs every root-to-leaf path p_k as its own causal
    sequence and averages: L_sep-avg = (1/K) sum_k sum_{t in p_k} l_t;
  * section 4.2 - the tree mask gives every token exactly the context of its own path, so
    the packed result equals the per-path result;
  * section 5 - RoPE positions are the token's index on its path;
  * section 6.2 - since sum_k sum_{t in p_k} l_t = sum_t g_t l_t, the packed gradient with
    weights g_t/K equals the per-path average's gradient, and shared-ancestor gradients add up.
Per-token loss used here: l_t = <U_t, O_t> (U given), so dL/dO_t on path k is U_t / K.

RoPE reading (the pages only name RoPE): rotate-half pairing (c, c + d/2), angle
pos * theta^(-2c/d), theta = 10000.  Softmax scale 1/sqrt(d).  LSE is the natural log of
the sum of exp(scaled scores).  GQA: q head h reads kv head h // (Hq / Hkv).

The online-softmax state merge follows the Tree Attention page (t6page "Tree Attention",
the associativity equation and the six-step decode table): a partial result is
(m, n, d) = (running max, numerator o*exp(lse - m), denominator exp(lse - m)), and two
partials merge as m = max(m_A, m_B), n = n_A e^{m_A-m} + n_B e^{m_B-m}, d likewise.
"""
from __future__ import annotations

import numpy as np

from .tree import plan as _plan


def _f64(x):
    if hasattr(x, "detach"):                      # torch tensor (any dtype) -> float64 numpy
        import torch
        return x.detach().to(torch.float64).cpu().numpy()
    return np.asarray(x, dtype=np.float64)


def _angles(pos, d, theta):
    half = d // 2
    inv = theta ** (-(2.0 * np.arange(half)) / d)
    return np.asarray(pos, dtype=np.float64)[:, None] * inv[None, :]


def rope(x, pos, theta=10000.0):
    """Rotate-half RoPE of x [L, ..., d] at positions pos [L] (fp64)."""
    d = x.shape[-1]
    a = _angles(pos, d, theta)
    shape = (a.shape[0],) + (1,) * (x.ndim - 2) + (d // 2,)
    c, s = np.cos(a).reshape(shape), np.sin(a).reshape(shape)
    x1, x2 = x[..., : d // 2], x[..., d // 2:]
    return np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], axis=-1)


def rope_transpose(gr, pos, theta=10000.0):
    """Transpose (= inverse) of the RoPE rotation, applied to a gradient w.r.t. the rotated input."""
    d = gr.shape[-1]
    a = _angles(pos, d, theta)
    shape = (a.shape[0],) + (1,) * (gr.ndim - 2) + (d // 2,)
    c, s = np.cos(a).reshape(shape), np.sin(a).reshape(shape)
    g1, g2 = gr[..., : d // 2], gr[..., d // 2:]
    return np.concatenate([g1 * c + g2 * s, g2 * c - g1 * s], axis=-1)


def _causal_attention(qh, kh, vh, dO, scale):
    """Plain causal softmax attention and its backward on one sequence, fp64."""
    L = qh.shape[0]
    S = (qh @ kh.T) * scale
    S[np.triu_indices(L, 1)] = -np.inf
    m = S.max(axis=1)
    E = np.exp(S - m[:, None])
    l = E.sum(axis=1)
    P = E / l[:, None]
    O = P @ vh
    lse = m + np.log(l)
    dV = P.T @ dO
    dP = dO @ vh.T
    delta = (dO * O).sum(axis=1)
    dS = P * (dP - delta[:, None])
    dq = (dS @ kh) * scale
    dk = (dS.T @ qh) * scale
    return O, lse, dq, dk, dV


def attention_paths(parent, node_len, q, k, v, u, scale=None, theta=10000.0, heads=None,
                    use_rope=True, p=None, agree_tol=1e-12):
    """Path-expanded reference.  q,u: [N,Hq,d]; k,v: [N,Hkv,d], tokens in packed DFS order.

    Runs each of the K root-to-leaf paths as an independent causal sequence (positions
    0..|p|-1), backpropagates l = (1/K) sum_{t in p} <U_t, O_t>, and scatter-adds the gradients
    of the shared tokens.  Returns O [N,Hq,d], LSE [Hq,N], dQ, dK, dV (fp64, NaN/0 outside
    `heads`).  O and LSE of a token are checked to agree across all paths through it.
    """
    q, k, v, u = _f64(q), _f64(k), _f64(v), _f64(u)
    N, Hq, d = q.shape
    Hkv = k.shape[1]
    grp = Hq // Hkv
    scale = 1.0 / np.sqrt(d) if not scale else scale
    heads = range(Hq) if heads is None else heads
    p = _plan(parent, node_len) if p is None else p
    K = p["n_paths"]
    nl = np.asarray(node_len, dtype=np.int64)
    O = np.full((N, Hq, d), np.nan)
    LSE = np.full((Hq, N), np.nan)
    dQ = np.zeros((N, Hq, d))
    dK = np.zeros((N, Hkv, d))
    dV = np.zeros((N, Hkv, d))
    for path in p["paths"]:
        idx = np.concatenate([np.arange(p["tok_start"][v_], p["tok_start"][v_] + nl[v_])
                              for v_ in path]).astype(np.int64)
        if len(idx) == 0:
            continue
        pos = np.arange(len(idx))
        for h in heads:
            gk = h // grp
            qh, kh = q[idx, h], k[idx, gk]
            if use_rope:
                qh, kh = rope(qh, pos, theta), rope(kh, pos, theta)
            Oh, lse, dq, dk, dv = _causal_attention(qh, kh, v[idx, gk], u[idx, h] / K, scale)
            if use_rope:
                dq, dk = rope_transpose(dq, pos, theta), rope_transpose(dk, pos, theta)
            prev = O[idx, h]
            seen = ~np.isnan(prev[:, 0])
            if np.any(seen):
                err = max(np.abs(prev[seen] - Oh[seen]).max(),
                          np.abs(LSE[h, idx][seen] - lse[seen]).max())
                if err > agree_tol:
                    raise AssertionError(f"paths disagree on a shared token's output ({err:.3g})")
            O[idx, h] = Oh
            LSE[h, idx] = lse
            dQ[idx, h] += dq
            dK[idx, gk] += dk
            dV[idx, gk] += dv
    return dict(o=O, lse=LSE, dq=dQ, dk=dK, dv=dV)


def attention_nodes(parent, node_len, q, k, v, u, scale=None, theta=10000.0, heads=None,
                    use_rope=True, p=None, row_chunk=2048, nodes=None):
    """The same result written with the tree mask of section 4.2 instead of path expansion.

    For each node a, its tokens are the queries; the keys are the tokens of a's ancestors
    (in root-to-a order) followed by a's own tokens, causal inside a.  Key positions are
    their index in that list; the query gradient weight is g_t / K (section 6.2), with g_t
    counted from the paths.  Nothing is shared between nodes except the summed gradients.
    Rows of a long node are taken `row_chunk` at a time; each chunk is the full row set of
    those queries, so the result does not depend on the chunk size.
    With `nodes` given, only those nodes' tokens act as queries: their O, LSE and dQ are exact,
    and so are dK, dV of every key that no other node's tokens can see (e.g. a leaf's own keys).
    """
    q, k, v, u = _f64(q), _f64(k), _f64(v), _f64(u)
    N, Hq, d = q.shape
    Hkv = k.shape[1]
    grp = Hq // Hkv
    scale = 1.0 / np.sqrt(d) if not scale else scale
    heads = range(Hq) if heads is None else heads
    p = _plan(parent, node_len) if p is None else p
    K = p["n_paths"]
    nl = np.asarray(node_len, dtype=np.int64)
    chain = {}
    for path in p["paths"]:
        for a, v_ in enumerate(path):
            chain[v_] = path[: a + 1]
    O = np.full((N, Hq, d), np.nan)
    LSE = np.full((Hq, N), np.nan)
    dQ = np.zeros((N, Hq, d))
    dK = np.zeros((N, Hkv, d))
    dV = np.zeros((N, Hkv, d))
    for a, path in chain.items():
        if nl[a] == 0 or (nodes is not None and a not in nodes):
            continue
        kidx = np.concatenate([np.arange(p["tok_start"][b], p["tok_start"][b] + nl[b])
                               for b in path]).astype(np.int64)
        A = len(kidx) - nl[a]                          # ancestor tokens before a's own
        kpos = np.arange(len(kidx))
        wq = p["g"][kidx[A:]].astype(np.float64) / K   # g_t / K of a's tokens
        for h in heads:
            gk = h // grp
            kh = rope(k[kidx, gk], kpos, theta) if use_rope else k[kidx, gk]
            vh = v[kidx, gk]
            dk_acc = np.zeros_like(kh)
            dv_acc = np.zeros_like(vh)
            for r0 in range(0, nl[a], row_chunk):
                r1 = min(nl[a], r0 + row_chunk)
                qi = kidx[A + r0: A + r1]
                nk = A + r1                              # keys visible to the last row of the chunk
                qh = rope(q[qi, h], kpos[A + r0: A + r1], theta) if use_rope else q[qi, h]
                S = (qh @ kh[:nk].T) * scale
                rr = np.arange(r1 - r0)[:, None]
                cc = np.arange(nk)[None, :]
                S = np.where(cc <= A + r0 + rr, S, -np.inf)
                m = S.max(axis=1)
                E = np.exp(S - m[:, None])
                l = E.sum(axis=1)
                P = E / l[:, None]
                Oh = P @ vh[:nk]
                dO = wq[r0:r1, None] * u[qi, h]
                dv_acc[:nk] += P.T @ dO
                dP = dO @ vh[:nk].T
                delta = (dO * Oh).sum(axis=1)
                dS = P * (dP - delta[:, None])
                dq = (dS @ kh[:nk]) * scale
                dk_acc[:nk] += (dS.T @ qh) * scale
                if use_rope:
                    dq = rope_transpose(dq, kpos[A + r0: A + r1], theta)
                O[qi, h] = Oh
                LSE[h, qi] = m + np.log(l)
                dQ[qi, h] += dq
            if use_rope:
                dk_acc = rope_transpose(dk_acc, kpos, theta)
            dK[kidx, gk] += dk_acc
            dV[kidx, gk] += dv_acc
    return dict(o=O, lse=LSE, dq=dQ, dk=dK, dv=dV)


def softmax_state(scores, values):
    """Partial attention state of one query over a key subset: (m, n, d) with n = sum e^{s-m} v,
    d = sum e^{s-m} (the Tree Attention page's max / numerator / denominator)."""
    scores = np.asarray(scores, dtype=np.float64)
    m = scores.max()
    e = np.exp(scores - m)
    return m, e @ np.asarray(values, dtype=np.float64), e.sum()


def merge_softmax_state(a, b):
    """Associative merge of two partial states (m, n, d); the output is n / d, lse = m + log d."""
    ma, na, da = a
    mb, nb, db = b
    m = max(ma, mb)
    fa, fb = np.exp(ma - m), np.exp(mb - m)
    return m, na * fa + nb * fb, da * fa + db * fb
