"""Oracle for the gradients of the differential-attention forward.

TEST INFRASTRUCTURE ONLY (tests, smoke check, benchmark baseline); never used
by the product path, and it shares no code with the CUDA library.

The pages define the forward only; the modules they print are trained
(lambda_q1 ... lambda_k2 and the sub-layer norm weight are nn.Parameters in
"DiffTransformer.py" and "LlamaDiffSdpaAttention.py", and the FlashDiffAttention
pull request targets training frameworks), so the gradients are the plain
derivatives of that forward. They are obtained here by torch autograd (a library
primitive) applied to a plain fp64 restatement of the forward in the
map-difference form of "DiffTransformer.py", MultiHeadDifferentialAttention.forward:
masked score maps, two softmaxes, (A1 - lambda A2) V, the per-head RMSNorm,
the weight and (1 - lambda_init), with lambda reparameterised from its four
vectors ("Compute lambda using reparameterization"). The tests pin these
gradients against central finite differences of the independent C oracle.
"""
from __future__ import annotations

from typing import Dict, Sequence

import torch


def _lambda(lq1, lk1, lq2, lk2, lambda_init, H):
    lam = torch.exp((lq1 * lk1).sum(-1)) - torch.exp((lq2 * lk2).sum(-1)) + lambda_init
    return lam.expand(H) if lam.dim() == 0 else lam


def forward(cu_seqlens: Sequence[int], q, k, v, lq1, lk1, lq2, lk2, w, lambda_init: float, eps: float,
            causal: bool) -> torch.Tensor:
    """fp64 forward, differentiable in q, k, v, the lambda vectors and w.
    q [tokens, H, 2d], k [tokens, Hkv, 2d], v [tokens, Hkv, dv] -> [tokens, H, dv]."""
    tokens, H, two_d = q.shape
    Hkv = k.shape[1]
    d = two_d // 2
    G = H // Hkv
    lam = _lambda(lq1, lk1, lq2, lk2, lambda_init, H)
    out = []
    cu = [int(x) for x in cu_seqlens]
    for s in range(len(cu) - 1):
        a, b = cu[s], cu[s + 1]
        n = b - a
        if n == 0:
            continue
        mask = torch.zeros(n, n, dtype=q.dtype)
        if causal:
            mask = mask.masked_fill(torch.ones(n, n, dtype=torch.bool).triu(1), float("-inf"))
        heads = []
        for h in range(H):
            g = h // G
            maps = []
            for c in range(2):
                qc = q[a:b, h, c * d:(c + 1) * d]
                kc = k[a:b, g, c * d:(c + 1) * d]
                maps.append(torch.softmax(qc @ kc.T * d ** -0.5 + mask, dim=-1))
            o = (maps[0] - lam[h] * maps[1]) @ v[a:b, g, :]
            rms = torch.sqrt((o * o).mean(-1, keepdim=True) + eps)
            heads.append(o / rms * w * (1.0 - lambda_init))
        out.append(torch.stack(heads, dim=1))
    return torch.cat(out, dim=0) if out else q.new_zeros(0, H, v.shape[-1])


def gradients(cu_seqlens, q, k, v, lq1, lk1, lq2, lk2, w, lambda_init: float, eps: float, causal: bool,
              dy) -> Dict[str, torch.Tensor]:
    """Gradients of sum(y * dy) with respect to q, k, v, the lambda vectors and w
    (all fp64 CPU tensors)."""
    leaves = {n: t.detach().to(torch.float64).clone().requires_grad_(True)
              for n, t in dict(q=q, k=k, v=v, lq1=lq1, lk1=lk1, lq2=lq2, lk2=lk2, w=w).items()}
    y = forward(cu_seqlens, leaves["q"], leaves["k"], leaves["v"], leaves["lq1"], leaves["lk1"],
                leaves["lq2"], leaves["lk2"], leaves["w"], lambda_init, eps, causal)
    grads = torch.autograd.grad(y, list(leaves.values()), grad_outputs=dy.to(torch.float64), allow_unused=True)
    return {n: (g if g is not None else torch.zeros_like(leaves[n])) for n, g in zip(leaves, grads)}
