"""TEST INFRASTRUCTURE ONLY: the chunkwise (WY) form of the KDA forward in fp64.

"Autoresearch on Kimi Delta Attention", section THE MECHANISM, points to the
chunkwise formulation of DeltaNet / Kimi Linear: the state still moves from one
block of tokens to the next in order, while the work inside a block becomes
matrix products.  "NVIDIA Kernel Design Agents optimize Kimi Delta Attention",
section 03 REWARD HACKING, names its pieces: the L2 normalisation of q and k, a
triangular matrix inverse, the initial state, the cumulative decay inside each
64-token chunk.  This module writes that form out plainly (numpy, fp64, direct
exponentials of decay differences, a library triangular solve) so that a test can
show it equals the token recurrence of ``kda_oracle.c`` for any chunk size.  The
CUDA kernels implement the same algebra independently.

For one chunk with rows 1..L, chunk-entry state S, and per-channel
Gamma_r = g_1 + ... + g_r:

  A[i, j] = beta_i * sum_c kh[i,c] kh[j,c] exp(Gamma[i,c] - Gamma[j,c])   (j < i)
  Tm      = (I + A)^-1                                    (unit lower triangular)
  w       = Tm Diag(beta) (kh * exp(Gamma))              L x dk
  u       = Tm Diag(beta) v                              L x dv
  U       = u - w S                                      (the corrections)
  P[i, j] = sum_c qh[i,c] kh[j,c] exp(Gamma[i,c] - Gamma[j,c])           (j <= i)
  O       = scale * ((qh * exp(Gamma)) S + P U)
  S'      = Diag(exp(Gamma_L)) S + (kh * exp(Gamma_L - Gamma))^T U
"""
from __future__ import annotations

import numpy as np
from scipy.linalg import solve_triangular

from .recurrence import L2_EPS, _f64


def _l2n(x: np.ndarray, eps: float) -> np.ndarray:
    return x / np.sqrt(np.sum(x * x, axis=-1, keepdims=True) + eps)


def chunk_step(qh, kh, v, g, beta, S, scale):
    """Advance one chunk.  qh, kh, g: [L, dk]; v: [L, dv]; beta: [L]; S: [dk, dv]."""
    L = qh.shape[0]
    if L == 0:
        return np.zeros((0, S.shape[1])), S
    G = np.cumsum(g, axis=0)                                  # [L, dk]
    diff = G[:, None, :] - G[None, :, :]                      # [i, j, c] = G_i - G_j
    lower_eq = np.tril(np.ones((L, L), dtype=bool))           # j <= i
    diff = np.where(lower_eq[:, :, None], diff, -np.inf)      # only causal pairs
    decay = np.exp(diff)                                      # exp(G_i - G_j), 0 above diag
    KK = np.einsum("ic,jc,ijc->ij", kh, kh, decay)
    A = np.tril(beta[:, None] * KK, k=-1)
    Tm = solve_triangular(np.eye(L) + A, np.eye(L), lower=True, unit_diagonal=True)
    gam = np.exp(G)
    w = Tm @ (beta[:, None] * (kh * gam))
    u = Tm @ (beta[:, None] * v)
    U = u - w @ S
    P = np.einsum("ic,jc,ijc->ij", qh, kh, decay)            # includes j == i
    O = scale * ((qh * gam) @ S + P @ U)
    Ktil = kh * np.exp(G[-1][None, :] - G)
    S_new = np.exp(G[-1])[:, None] * S + Ktil.T @ U
    return O, S_new


def kda_chunked_fp64(q, k, v, g, beta, h0=None, cu_seqlens=None, scale=None,
                     chunk: int = 64, eps: float = L2_EPS):
    """Chunkwise fp64 forward with arbitrary chunk size; same I/O as the oracle."""
    q, k, v, g, beta = (_f64(x) for x in (q, k, v, g, beta))
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    if cu_seqlens is not None:
        cu = np.asarray(cu_seqlens.cpu() if hasattr(cu_seqlens, "cpu") else cu_seqlens,
                        dtype=np.int64)
        spans = [(0, int(cu[s]), int(cu[s + 1])) for s in range(len(cu) - 1)]
    else:
        spans = [(b, 0, T) for b in range(B)]
    N = len(spans)
    h0a = _f64(h0)
    if scale is None:
        scale = dk ** -0.5
    o = np.zeros((B, T, H, dv))
    hT = np.zeros((N, H, dk, dv))
    qn, kn = _l2n(q, eps), _l2n(k, eps)
    for s, (b, bos, eos) in enumerate(spans):
        for h in range(H):
            S = h0a[s, h].copy() if h0a is not None else np.zeros((dk, dv))
            for c0 in range(bos, eos, chunk):
                c1 = min(c0 + chunk, eos)
                O, S = chunk_step(qn[b, c0:c1, h], kn[b, c0:c1, h], v[b, c0:c1, h],
                                  g[b, c0:c1, h], beta[b, c0:c1, h], S, scale)
                o[b, c0:c1, h] = O
            hT[s, h] = S
    return o, hT


def kda_segmented_fp64(q, k, v, g, beta, h0=None, cu_seqlens=None, scale=None,
                       seg_chunks: int = 4, chunk: int = 64, eps: float = L2_EPS):
    """The exact inter-chunk split in fp64: same I/O as the oracle.

    The chunk step above is affine in the entry state: S' = M S + D with
    M = Diag(exp(Gamma_L)) - Ktil^T w and D = Ktil^T u.  A run of chunks (a segment)
    is therefore the map S -> F S + Z, F the product of its M (the step applied to
    the identity with v = 0, so u = 0) and Z its final state from S = 0.  Each
    (sequence, head) chain is cut into segments of seg_chunks chunks; the first
    runs from h0; the start state of segment k + 1 is F_k E_k + Z_k (a sequential
    scan over the segments); every later segment is then rerun from its start state
    for its outputs.  This is the legal counterpart of the history truncation that
    "NVIDIA Kernel Design Agents optimize Kimi Delta Attention", section 03 REWARD
    HACKING, describes: nothing is dropped, only regrouped."""
    q, k, v, g, beta = (_f64(x) for x in (q, k, v, g, beta))
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    if cu_seqlens is not None:
        cu = np.asarray(cu_seqlens.cpu() if hasattr(cu_seqlens, "cpu") else cu_seqlens,
                        dtype=np.int64)
        spans = [(0, int(cu[s]), int(cu[s + 1])) for s in range(len(cu) - 1)]
    else:
        spans = [(b, 0, T) for b in range(B)]
    N = len(spans)
    h0a = _f64(h0)
    if scale is None:
        scale = dk ** -0.5
    o = np.zeros((B, T, H, dv))
    hT = np.zeros((N, H, dk, dv))
    qn, kn = _l2n(q, eps), _l2n(k, eps)
    span = chunk * seg_chunks
    for s, (b, bos, eos) in enumerate(spans):
        for h in range(H):
            segs = [(a, min(a + span, eos)) for a in range(bos, eos, span)]

            def run(a, e, S, vv, out):
                for c0 in range(a, e, chunk):
                    c1 = min(c0 + chunk, e)
                    O, S = chunk_step(qn[b, c0:c1, h], kn[b, c0:c1, h], vv[c0 - a:c1 - a],
                                      g[b, c0:c1, h], beta[b, c0:c1, h], S, scale)
                    if out:
                        o[b, c0:c1, h] = O
                return S

            S0 = h0a[s, h].copy() if h0a is not None else np.zeros((dk, dv))
            if not segs:
                hT[s, h] = S0
                continue
            a, e = segs[0]
            E = run(a, e, S0, v[b, a:e, h], True)       # the first segment, from h0
            starts = [None, E]                           # start state of each segment
            for a, e in segs[1:-1]:                      # the middle segments: F, Z, scan
                F = run(a, e, np.eye(dk), np.zeros((e - a, dk)), False)
                Z = run(a, e, np.zeros((dk, dv)), v[b, a:e, h], False)
                starts.append(F @ starts[-1] + Z)
            for i, (a, e) in enumerate(segs[1:], start=1):  # every later segment, rerun
                S = run(a, e, starts[i], v[b, a:e, h], True)
                if i == len(segs) - 1:
                    hT[s, h] = S
            if len(segs) == 1:
                hT[s, h] = E
    return o, hT
