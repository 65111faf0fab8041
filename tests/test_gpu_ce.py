"""Parity of the fused vocabulary-projection cross-entropy ("Tree Training 技术详解",
sections 6.2, 6.3, 12) with the oracle, and of the GEMM kernel under it.

* the GEMM alone (diagnostic entry): every operand layout (K-major / MN-major A and B) with
  ragged M, N and K, against NumPy on the same bf16 values;
* the loss on random trees (zero-length nodes, several roots, ignored labels) with chunks
  shorter than the tree (the last one ragged), one chunk, and all labels ignored: loss, row
  logsumexp, dh and dW against the fp64 oracle;
* rollout32k at full size (N = 32768, D = 4096, V = 128256, chunks of 8192): the oracle's
  logsumexp and dh on sampled rows (chunk edges and nodes' last tokens, which predict several
  children); over all of dW, the identity sum_v dW[v] = 0 (each row of the logits gradient
  sums to zero); the loss finite and positive (its value needs every row's logsumexp, which
  the small-size cases check against the oracle).

Tolerances: logits are fp32 sums of bf16 products (~1e-6 relative); the logits gradient is
stored in bf16 (2^-9 relative per element), so dh and dW are compared at 2e-2 of their largest
magnitude; LSE at 1e-3 absolute; the loss at 1e-4 relative.
"""
import numpy as np
import pytest
import torch

import oracle
import tree_masked_attention_plan_gb300 as tam
from workloads import make_workload, random_tree

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda", 0)
IGN = -100


def _f64(t):
    return t.detach().to(torch.float64).cpu().numpy()


@pytest.mark.parametrize("a_mn,b_mn", [(0, 0), (0, 1), (1, 0), (1, 1)])
@pytest.mark.parametrize("M,N,K", [(200, 264, 136), (512, 512, 1024)])
def test_diag_gemm_layouts(a_mn, b_mn, M, N, K):
    g = torch.Generator().manual_seed(M + N + K + 2 * a_mn + b_mn)
    A = torch.randn(K, M, generator=g) if a_mn else torch.randn(M, K, generator=g)
    B = torch.randn(K, N, generator=g) if b_mn else torch.randn(N, K, generator=g)
    A, B = A.to(torch.bfloat16), B.to(torch.bfloat16)
    status = tam.new_status(DEV)
    C = tam.diag_gemm(A.to(DEV), B.to(DEV), M, N, K, a_mn, b_mn, status=status)
    torch.cuda.synchronize()
    tam.check_status(status, "diag gemm")
    a = _f64(A).T if a_mn else _f64(A)
    b = _f64(B) if b_mn else _f64(B).T
    ref = a @ b
    err = np.abs(_f64(C) - ref).max()
    assert err <= 1e-4 * np.abs(ref).max(), err


def _ce_inputs(N, D, V, seed, ignore_frac=0.2):
    g = torch.Generator().manual_seed(seed)
    h = torch.randn(N, D, generator=g).to(torch.bfloat16)
    W = (torch.randn(V, D, generator=g) / D ** 0.5).to(torch.bfloat16)
    labels = torch.randint(0, V, (N,), generator=g, dtype=torch.int32)
    labels[torch.rand(N, generator=g) < ignore_frac] = IGN
    return h, W, labels


def _run(parent, node_len, h, W, labels, chunk):
    plan = tam.tree_plan(parent, node_len, device=DEV)
    tree = tam.tree_arrays(parent, node_len, DEV)
    status = tam.new_status(DEV)
    out = tam.tree_ce_fwd_bwd(plan, tree, h.to(DEV), W.to(DEV), labels.to(DEV), chunk=chunk, status=status)
    torch.cuda.synchronize()
    tam.check_status(status, "tree ce")
    return [_f64(x) for x in out]


@pytest.mark.parametrize("seed,chunk", [(0, 256), (1, 128), (2, 1 << 20)])
def test_ce_random_trees(seed, chunk):
    parent, node_len = random_tree(500 + seed, n_nodes=60, max_len=25, zero_prob=0.15, n_roots=1 + seed)
    N = int(np.sum(node_len))
    D, V = 256, 1000
    h, W, labels = _ce_inputs(N, D, V, seed)
    loss, lse, dh, dW = _run(parent, node_len, h, W, labels, chunk)
    r = oracle.ce_paths(parent, node_len, _f64(h), _f64(W), labels.numpy(), IGN)
    assert abs(loss[0] - r["loss"]) <= 1e-4 * abs(r["loss"]), (loss[0], r["loss"])
    assert np.abs(lse - r["lse"]).max() <= 1e-3
    assert np.abs(dh - r["dh"]).max() <= 2e-2 * np.abs(r["dh"]).max()
    assert np.abs(dW - r["dW"]).max() <= 2e-2 * np.abs(r["dW"]).max()


def test_ce_all_ignored():
    parent, node_len = random_tree(77, n_nodes=20, max_len=20)
    N = int(np.sum(node_len))
    h, W, labels = _ce_inputs(N, 256, 512, 3)
    labels[:] = IGN
    loss, lse, dh, dW = _run(parent, node_len, h, W, labels, 128)
    assert loss[0] == 0 and not dh.any() and not dW.any()


def test_ce_rollout32k_full_size():
    wl = make_workload("rollout32k")
    N, D, V = int(np.sum(wl.node_len)), 4096, 128256
    g = torch.Generator().manual_seed(41)
    h = torch.randn(N, D, generator=g).to(torch.bfloat16)
    W = (torch.randn(V, D, generator=g) / D ** 0.5).to(torch.bfloat16)
    labels = torch.randint(0, V, (N,), generator=g, dtype=torch.int32)
    labels[torch.rand(N, generator=g) < 0.1] = IGN
    loss, lse, dh, dW = _run(wl.parent, wl.node_len, h, W, labels, 8192)
    p = oracle.plan(wl.parent, wl.node_len)
    starts = [int(p["tok_start"][v] + wl.node_len[v] - 1) for v in range(len(wl.parent)) if wl.node_len[v] > 0]
    rows = sorted(set([0, 1, 8191, 8192, N - 1] + starts[:6]))      # chunk edges and nodes' last tokens
    r = oracle.ce_rows(wl.parent, wl.node_len, _f64(h), _f64(W), labels.numpy(), rows, IGN, p=p)
    assert np.abs(lse[rows] - r["lse"]).max() <= 1e-3
    assert np.abs(dh[rows] - r["dh"]).max() <= 2e-2 * np.abs(r["dh"]).max()
    colsum = dW.sum(axis=0)
    assert np.abs(colsum).max() <= 2e-2 * np.abs(dW).sum(axis=0).max()
    assert np.isfinite(loss[0]) and loss[0] > 0
