"""Seeded random activations for a workload: Q, K, V and the per-token loss gradient U.

All tensors are token-major ``[N, heads, d]`` in packed (depth-first) token order; the
values are i.i.d. N(0, 1) drawn in fp32 from a torch CPU generator and rounded to bf16,
which is the precision the kernels read.  The tiny example uses U = 1 (its per-token loss
is the sum of the output row).
"""
from __future__ import annotations

import torch


def _randn(seed: int, shape) -> torch.Tensor:
    gen = torch.Generator().manual_seed(seed)
    return torch.randn(*shape, generator=gen, dtype=torch.float32)


def make_tensors(wl, n_tokens: int | None = None, with_fp32: bool = False):
    """Returns dict q, k, v, u (bf16, CPU); with_fp32 adds the fp32 draws as q32/k32/v32."""
    N = wl.n_tokens if n_tokens is None else n_tokens
    s = wl.seeds
    q32 = _randn(s["q"], (N, wl.Hq, wl.d))
    k32 = _randn(s["k"], (N, wl.Hkv, wl.d))
    v32 = _randn(s["v"], (N, wl.Hkv, wl.d))
    if wl.uniform_grad:
        u32 = torch.ones(N, wl.Hq, wl.d, dtype=torch.float32)
    else:
        u32 = _randn(s["u"], (N, wl.Hq, wl.d))
    out = dict(q=q32.to(torch.bfloat16), k=k32.to(torch.bfloat16), v=v32.to(torch.bfloat16),
               u=u32.to(torch.bfloat16))
    if with_fp32:
        out.update(q32=q32, k32=k32, v32=v32)
    return out


def make_conv_tensors(n_tokens: int, C: int, K: int, seed: int = 0, with_bias: bool = True):
    """Seeded inputs of a depthwise causal convolution over the packed tokens: x [N, C] and the
    upstream gradient u [N, C] i.i.d. N(0, 1) rounded to bf16; taps w [K, C] N(0, 1/K) and
    bias [C] N(0, 1) in fp32 (or None)."""
    x = _randn(seed, (n_tokens, C)).to(torch.bfloat16)
    u = _randn(seed + 1, (n_tokens, C)).to(torch.bfloat16)
    w = _randn(seed + 2, (K, C)) / K ** 0.5
    b = _randn(seed + 3, (C,)) if with_bias else None
    return dict(x=x, w=w, bias=b, u=u)
