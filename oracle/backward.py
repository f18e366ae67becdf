"""TEST INFRASTRUCTURE ONLY: the gradients of the KDA forward, in fp64.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this module.  The CUDA library never calls it.

"Autoresearch on Kimi Delta Attention", sections THE MECHANISM and OPTIMIZATION
TRACE, describes the training-side workload: a backward pass that carries the
gradient of the recurrent state backwards through the chunks.  What that backward
computes has a plain definition: the derivative of the forward's outputs (o and
h_T), contracted with given output gradients (do, dh_T), with respect to every
input (q, k, v, g, beta, h0).  This module writes the forward recurrence out
token by token in PyTorch fp64 (the same update as ``kda_oracle.c``: L2-normalised
q and k, alpha = exp(g) per key channel, S_t = (I - beta_t kh kh^T) Diag(alpha_t)
S_{t-1} + beta_t kh v_t^T, o_t = scale S_t^T qh_t) and lets PyTorch's autograd take
that derivative.  Tests pin it three ways: its forward equals the C oracle, its
gradients match central finite differences of the C oracle on tiny inputs, and the
beta = 0 case matches the closed form's derivative.
"""
from __future__ import annotations

from typing import Optional, Tuple

import numpy as np
import torch

from .recurrence import L2_EPS


def _t64(x) -> Optional[torch.Tensor]:
    if x is None:
        return None
    if isinstance(x, np.ndarray):
        x = torch.from_numpy(x)
    return x.detach().to(torch.float64).cpu()


def _spans(B: int, T: int, cu_seqlens) -> list:
    if cu_seqlens is None:
        return [(b, 0, T) for b in range(B)]
    cu = [int(c) for c in (cu_seqlens.cpu().tolist() if hasattr(cu_seqlens, "cpu") else cu_seqlens)]
    return [(0, cu[s], cu[s + 1]) for s in range(len(cu) - 1)]


def forward_torch(q, k, v, g, beta, h0, spans, scale, eps: float = L2_EPS):
    """The token recurrence on fp64 torch tensors (differentiable); all heads at once.
    q, k, g: [B, T, H, dk]; v: [B, T, H, dv]; beta: [B, T, H]; h0: [N, H, dk, dv] or
    None.  Returns o [B, T, H, dv] and h_T [N, H, dk, dv]."""
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    qh = q / torch.sqrt((q * q).sum(-1, keepdim=True) + eps)
    kh = k / torch.sqrt((k * k).sum(-1, keepdim=True) + eps)
    alpha = torch.exp(g)
    rows = [[None] * T for _ in range(B)]
    finals = []
    for s, (b, bos, eos) in enumerate(spans):
        S = h0[s] if h0 is not None else torch.zeros(H, dk, dv, dtype=torch.float64)
        for t in range(bos, eos):
            P = alpha[b, t][:, :, None] * S                                  # Diag(alpha) S
            kt = kh[b, t]                                                    # [H, dk]
            r = v[b, t] - torch.einsum("hc,hcn->hn", kt, P)                  # v - P^T kh
            S = P + beta[b, t][:, None, None] * kt[:, :, None] * r[:, None, :]
            rows[b][t] = scale * torch.einsum("hcn,hc->hn", S, qh[b, t])     # scale S^T qh
        finals.append(S)
    zero = torch.zeros(H, dv, dtype=torch.float64)
    o = torch.stack([torch.stack([rows[b][t] if rows[b][t] is not None else zero for t in range(T)])
                     for b in range(B)])
    hT = torch.stack(finals) if finals else torch.zeros(0, H, dk, dv, dtype=torch.float64)
    return o, hT


def kda_backward_fp64(q, k, v, g, beta, h0=None, cu_seqlens=None, scale=None, do=None, dhT=None,
                      eps: float = L2_EPS) -> Tuple[np.ndarray, ...]:
    """Gradients (dq, dk, dv, dg, dbeta, dh0) of sum(o * do) + sum(h_T * dh_T), fp64
    numpy arrays shaped like the inputs (dh0 zeros-shaped [N, H, dk, dv] even when
    h0 is None: the gradient with respect to a zero initial state).  ``do`` and
    ``dhT`` default to zero."""
    q, k, v, g, beta = (_t64(x) for x in (q, k, v, g, beta))
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    spans = _spans(B, T, cu_seqlens)
    N = len(spans)
    h0t = _t64(h0) if h0 is not None else torch.zeros(N, H, dk, dv, dtype=torch.float64)
    if scale is None:
        scale = dk ** -0.5
    leaves = [x.clone().requires_grad_(True) for x in (q, k, v, g, beta, h0t)]
    o, hT = forward_torch(*leaves, spans, float(scale), eps)
    loss = torch.zeros((), dtype=torch.float64)
    if do is not None:
        loss = loss + (o * _t64(do)).sum()
    if dhT is not None and N > 0:
        loss = loss + (hT * _t64(dhT)).sum()
    if loss.requires_grad:
        grads = torch.autograd.grad(loss, leaves, allow_unused=True)
    else:
        grads = [None] * 6
    return tuple((gr if gr is not None else torch.zeros_like(x)).numpy() for gr, x in zip(grads, leaves))
