"""TEST INFRASTRUCTURE ONLY: deliberately wrong variants of the KDA forward.

"NVIDIA Kernel Design Agents optimize Kimi Delta Attention", section 03 REWARD
HACKING, lists shortcuts that passed a weak test suite but were wrong on real
inputs; section 01 RESULTS adds the bf16 recurrent state of an earlier kernel.
Each is restated here as a fp64 CPU variant of the chunkwise form in
``chunked.py`` (never as GPU code).  The test suite requires every one of them
to FAIL the parity gates on at least one input recipe: this is what shows that
the synthetic inputs and the tolerances can tell a correct kernel from these.

  M1  constant reciprocal norm 0.1778209953 in place of the L2 normalisation
  M2  some initial-state key channels zeroed
  M2b the triangular inverse skipped (Tm = I)
  M3  cu_seqlens ignored; sequence boundaries assumed to be an even split
  M4  history truncated: each sequence cut into independent 32-token pieces
  M5  in-chunk decay formed as exp(Gamma_i) * exp(-Gamma_j) in fp32
  M6  cumulative decay looked up in an fp16 table
  M7  recurrent state rounded to bf16 after every chunk
"""
from __future__ import annotations

import numpy as np
import torch
from scipy.linalg import solve_triangular

from .chunked import _l2n
from .recurrence import L2_EPS, _f64

KINDS = ("M1", "M2", "M2b", "M3", "M4", "M5", "M6", "M7")
HACK_RSQRT = 0.1778209953


def _round_bf16(x: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.asarray(x, dtype=np.float32)).to(torch.bfloat16).double().numpy()


def _decay_exact(G):
    L = G.shape[0]
    diff = G[:, None, :] - G[None, :, :]
    mask = np.tril(np.ones((L, L), dtype=bool))
    return np.exp(np.where(mask[:, :, None], diff, -np.inf)), np.exp(G), np.exp(G[-1][None, :] - G)


def _decay_naive_fp32(G):
    """M5: exp(G_i) * exp(-G_j) in fp32; exp(-G_j) overflows once decay is deep."""
    with np.errstate(over="ignore", invalid="ignore", under="ignore"):
        Gf = G.astype(np.float32)
        e_pos = np.exp(Gf)
        e_neg = np.exp(-Gf)
        L = G.shape[0]
        mask = np.tril(np.ones((L, L), dtype=bool))
        dec = (e_pos[:, None, :] * e_neg[None, :, :]).astype(np.float64)
        dec = np.where(mask[:, :, None], dec, 0.0)
        last = (e_pos[-1][None, :] * e_neg).astype(np.float64)
    return dec, e_pos.astype(np.float64), last


def _decay_fp16_table(G):
    """M6: a table of exp(Gamma) in fp16; ratios of table entries as decays."""
    with np.errstate(over="ignore", invalid="ignore", under="ignore", divide="ignore"):
        tab = np.exp(G).astype(np.float16).astype(np.float64)
        L = G.shape[0]
        mask = np.tril(np.ones((L, L), dtype=bool))
        dec = tab[:, None, :] / tab[None, :, :]
        dec = np.where(mask[:, :, None], dec, 0.0)
        last = tab[-1][None, :] / tab
    return dec, tab, last


def _chunk(qh, kh, v, g, beta, S, scale, decay_fn, skip_inverse):
    L = qh.shape[0]
    G = np.cumsum(g, axis=0)
    with np.errstate(over="ignore", invalid="ignore"):
        decay, gam, last = decay_fn(G)
        A = np.tril(beta[:, None] * np.einsum("ic,jc,ijc->ij", kh, kh, decay), k=-1)
        if skip_inverse:
            Tm = np.eye(L)
        else:
            Tm = solve_triangular(np.eye(L) + A, np.eye(L), lower=True, unit_diagonal=True,
                                  check_finite=False)
        w = Tm @ (beta[:, None] * (kh * gam))
        u = Tm @ (beta[:, None] * v)
        U = u - w @ S
        P = np.einsum("ic,jc,ijc->ij", qh, kh, decay)
        O = scale * ((qh * gam) @ S + P @ U)
        S_new = gam[-1][:, None] * S + (kh * last).T @ U
    return O, S_new


def kda_mutant(kind: str, q, k, v, g, beta, h0=None, cu_seqlens=None, scale=None,
               chunk: int = 64, eps: float = L2_EPS):
    """Run mutant ``kind`` (one of KINDS); same I/O as the oracle."""
    if kind not in KINDS:
        raise ValueError(kind)
    q, k, v, g, beta = (_f64(x) for x in (q, k, v, g, beta))
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    if cu_seqlens is not None:
        cu = np.asarray(cu_seqlens.cpu() if hasattr(cu_seqlens, "cpu") else cu_seqlens,
                        dtype=np.int64)
        N = len(cu) - 1
        if kind == "M3":
            cu = np.round(np.linspace(0, T, N + 1)).astype(np.int64)
        spans = [(0, int(cu[s]), int(cu[s + 1])) for s in range(N)]
    else:
        spans = [(b, 0, T) for b in range(B)]
        N = B
    h0a = _f64(h0)
    if h0a is not None and kind == "M2":
        h0a = h0a.copy()
        h0a[:, :, dk // 2:, :] = 0.0
    if scale is None:
        scale = dk ** -0.5
    if kind == "M1":
        qn, kn = q * HACK_RSQRT, k * HACK_RSQRT
    else:
        qn, kn = _l2n(q, eps), _l2n(k, eps)
    decay_fn = {"M5": _decay_naive_fp32, "M6": _decay_fp16_table}.get(kind, _decay_exact)
    piece = 32 if kind == "M4" else None
    o = np.zeros((B, T, H, dv))
    hT = np.zeros((N, H, dk, dv))
    for s, (b, bos, eos) in enumerate(spans):
        for h in range(H):
            S0 = h0a[s, h].copy() if h0a is not None else np.zeros((dk, dv))
            S = S0
            for c0 in range(bos, eos, piece or chunk):
                if piece and c0 > bos:
                    S = np.zeros((dk, dv))
                c1 = min(c0 + (piece or chunk), eos)
                O, S = _chunk(qn[b, c0:c1, h], kn[b, c0:c1, h], v[b, c0:c1, h],
                              g[b, c0:c1, h], beta[b, c0:c1, h], S, scale, decay_fn,
                              kind == "M2b")
                if kind == "M7":
                    S = _round_bf16(S)
                o[b, c0:c1, h] = O
            hT[s, h] = S
    return o, hT
