"""Pins for the fp64 oracle: checks against facts fixed by the mathematics.

Each ``pin_*`` takes a forward callable with the oracle's signature
(``fwd(q, k, v, g, beta, h0, cu_seqlens, scale, eps=...) -> (o, hT)``) and returns
the worst relative error it sees.  The oracle must keep every pin below its
tolerance; each planted mistake must push at least one pin above it.
"""
from __future__ import annotations

import math
from fractions import Fraction

import numpy as np

from oracle import brute

# Integer vectors with integer L2 norms: exact in fp64, rational after normalising.
_PYTH3 = [(1, 2, 2), (2, 3, 6), (1, 4, 8), (2, 6, 9), (4, 4, 7), (2, 10, 11), (3, 4, 12)]
_PYTH4 = [(1, 1, 1, 1), (1, 2, 2, 4), (2, 4, 5, 6), (1, 3, 3, 9), (2, 2, 4, 5), (1, 1, 3, 5)]


def _rel(a, b):
    a, b = np.asarray(a, dtype=np.float64), np.asarray(b, dtype=np.float64)
    den = np.sqrt(np.sum(b * b))
    num = np.sqrt(np.sum((a - b) ** 2))
    if not np.isfinite(num):
        return float("inf")
    return float(num / den) if den > 0 else float(num)


def _rational_vec(rng, d):
    base = _PYTH3 if d == 3 else _PYTH4
    v = list(base[rng.integers(len(base))])
    rng.shuffle(v)
    return [int(x) * (1 if rng.uniform() < 0.5 else -1) for x in v]


def brute_case(seed: int, T: int = 5, d: int = 3):
    """Tiny exact case: dk = dv = d in {3, 4}; rational alpha, beta, S0, scale."""
    rng = np.random.default_rng(seed)
    q = [_rational_vec(rng, d) for _ in range(T)]
    k = [_rational_vec(rng, d) for _ in range(T)]
    v = [[int(x) for x in rng.integers(-4, 5, size=d)] for _ in range(T)]
    alpha = [[Fraction(int(rng.integers(1, 8)), 8) for _ in range(d)] for _ in range(T)]
    beta = [Fraction(int(rng.integers(1, 5)), 4) for _ in range(T)]
    S0 = [[Fraction(int(rng.integers(-3, 4)), 4) for _ in range(d)] for _ in range(d)]
    scale = Fraction(1, 2)
    return q, k, v, alpha, beta, S0, scale


def _case_arrays(case):
    q, k, v, alpha, beta, S0, scale = case
    T, d = len(q), len(q[0])
    qa = np.array(q, dtype=np.float64).reshape(1, T, 1, d)
    ka = np.array(k, dtype=np.float64).reshape(1, T, 1, d)
    va = np.array(v, dtype=np.float64).reshape(1, T, 1, d)
    ga = np.log(np.array([[float(a) for a in row] for row in alpha])).reshape(1, T, 1, d)
    ba = np.array([float(b) for b in beta]).reshape(1, T, 1)
    h0 = np.array([[float(x) for x in row] for row in S0]).reshape(1, 1, d, d)
    return qa, ka, va, ga, ba, h0, float(scale)


def pin_brute(fwd, seeds=range(6)) -> float:
    """Oracle vs exact rational recurrence (eps = 0)."""
    worst = 0.0
    for s in seeds:
        case = brute_case(s, T=5, d=3 + (s % 2))
        o_ex, S_ex = brute.brute_recurrence(*case)
        qa, ka, va, ga, ba, h0, scale = _case_arrays(case)
        o, hT = fwd(qa, ka, va, ga, ba, h0, None, scale, eps=0.0)
        o_ref = np.array([[float(x) for x in row] for row in o_ex])
        S_ref = np.array([[float(x) for x in row] for row in S_ex])
        worst = max(worst, _rel(o[0, :, 0, :], o_ref), _rel(hT[0, 0], S_ref))
    return worst


def pin_beta_zero(fwd, seed=1) -> float:
    """beta = 0: S_t = Diag(exp(sum g)) S_0 and o_t = scale (Diag(exp(Gamma_t)) S_0)^T qh_t."""
    rng = np.random.default_rng(seed)
    B, T, H, dk, dv = 2, 40, 2, 6, 5
    q = rng.normal(size=(B, T, H, dk))
    k = rng.normal(size=(B, T, H, dk))
    v = rng.normal(size=(B, T, H, dv))
    g = -rng.uniform(0.0, 0.3, size=(B, T, H, dk))
    beta = np.zeros((B, T, H))
    h0 = rng.normal(size=(B, H, dk, dv))
    scale = 0.7
    o, hT = fwd(q, k, v, g, beta, h0, None, scale, eps=1e-6)
    Gam = np.cumsum(g, axis=1)                                     # [B, T, H, dk]
    qh = q / np.sqrt(np.sum(q * q, -1, keepdims=True) + 1e-6)
    St = np.exp(Gam)[..., None] * h0[:, None]                      # [B, T, H, dk, dv]
    o_ref = scale * np.einsum("bthkv,bthk->bthv", St, qh)
    return max(_rel(o, o_ref), _rel(hT, St[:, -1]))


def pin_delta_write(fwd, seed=2) -> float:
    """beta_t = 1 and q_t parallel to k_t (eps = 0): o_t = scale * v_t for any history."""
    rng = np.random.default_rng(seed)
    B, T, H, dk, dv = 1, 30, 3, 8, 6
    q = rng.normal(size=(B, T, H, dk))
    k = rng.normal(size=(B, T, H, dk))
    v = rng.normal(size=(B, T, H, dv))
    g = -rng.uniform(0.0, 2.0, size=(B, T, H, dk))
    beta = rng.uniform(0.0, 1.0, size=(B, T, H))
    h0 = rng.normal(size=(B, H, dk, dv))
    sel = rng.uniform(size=(B, T, H)) < 0.4
    beta[sel] = 1.0
    c = rng.uniform(0.1, 10.0, size=(B, T, H, 1))
    q = np.where(sel[..., None], c * k, q)
    scale = 1.3
    o, _ = fwd(q, k, v, g, beta, h0, None, scale, eps=0.0)
    return _rel(o[sel], scale * v[sel])


def pin_recall(fwd, seed=3) -> float:
    """alpha = 1, beta = 1, orthonormal keys, S_0 = 0: S_n = sum k_i v_i^T, and a
    later query q = k_j (beta = 0) reads back scale * v_j exactly."""
    rng = np.random.default_rng(seed)
    H, dk, dv, n = 2, 8, 5, 6
    T = 2 * n
    q = rng.normal(size=(1, T, H, dk))
    k = np.zeros((1, T, H, dk))
    v = rng.normal(size=(1, T, H, dv))
    beta = np.zeros((1, T, H))
    S_ref = np.zeros((1, H, dk, dv))
    o_idx, o_ref = [], []
    for h in range(H):
        Qm, _ = np.linalg.qr(rng.normal(size=(dk, dk)))
        keys = Qm[:, :n].T                                          # n orthonormal rows
        k[0, :n, h] = keys
        beta[0, :n, h] = 1.0
        S_ref[0, h] = keys.T @ v[0, :n, h]
        perm = rng.permutation(n)
        for t in range(n):
            j = perm[t]
            q[0, n + t, h] = keys[j] * rng.uniform(0.5, 2.0)
            k[0, n + t, h] = rng.normal(size=dk)
            o_idx.append((n + t, h))
            o_ref.append(0.5 * v[0, j, h])
    g = np.zeros((1, T, H, dk))
    o, hT = fwd(q, k, v, g, beta, None, None, 0.5, eps=0.0)
    got = np.array([o[0, t, h] for t, h in o_idx])
    return max(_rel(got, np.array(o_ref)), _rel(hT, S_ref))


def pin_varlen_split(fwd, seed=4) -> float:
    """Packed varlen equals each sequence run alone; a prefill split at any point
    and resumed from the returned state equals the whole."""
    rng = np.random.default_rng(seed)
    lens = [7, 1, 0, 19, 12]
    H, dk, dv = 2, 5, 4
    T = sum(lens)
    q = rng.normal(size=(1, T, H, dk))
    k = rng.normal(size=(1, T, H, dk))
    v = rng.normal(size=(1, T, H, dv))
    g = -rng.uniform(0.0, 1.0, size=(1, T, H, dk))
    beta = rng.uniform(size=(1, T, H))
    h0 = rng.normal(size=(len(lens), H, dk, dv))
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    o, hT = fwd(q, k, v, g, beta, h0, cu, 0.4, eps=1e-6)
    worst = 0.0
    for s, L in enumerate(lens):
        a, b = cu[s], cu[s + 1]
        o1, h1 = fwd(q[:, a:b], k[:, a:b], v[:, a:b], g[:, a:b], beta[:, a:b],
                     h0[s:s + 1], None, 0.4, eps=1e-6)
        worst = max(worst, _rel(o[:, a:b], o1) if L else 0.0, _rel(hT[s], h1[0]))
    # split the 19-token sequence at 8: resume from the returned state
    s, cut = 3, 8
    a, b = cu[s], cu[s + 1]
    sl1, sl2 = slice(a, a + cut), slice(a + cut, b)
    oA, hA = fwd(q[:, sl1], k[:, sl1], v[:, sl1], g[:, sl1], beta[:, sl1], h0[s:s + 1], None,
                 0.4, eps=1e-6)
    oB, hB = fwd(q[:, sl2], k[:, sl2], v[:, sl2], g[:, sl2], beta[:, sl2], hA, None, 0.4,
                 eps=1e-6)
    worst = max(worst, _rel(np.concatenate([oA, oB], axis=1), o[:, a:b]), _rel(hB[0], hT[s]))
    return worst


def pin_symmetries(fwd, seed=5) -> float:
    """Heads are independent (a head permutation permutes the outputs); the result is
    linear in (v, h0) jointly; permuting value channels permutes o and the state's
    columns; positive rescaling of q or k rows changes nothing (eps = 0)."""
    rng = np.random.default_rng(seed)
    B, T, H, dk, dv = 1, 25, 3, 6, 5
    q = rng.normal(size=(B, T, H, dk))
    k = rng.normal(size=(B, T, H, dk))
    v = rng.normal(size=(B, T, H, dv))
    g = -rng.uniform(0.0, 1.0, size=(B, T, H, dk))
    beta = rng.uniform(size=(B, T, H))
    h0 = rng.normal(size=(B, H, dk, dv))
    o, hT = fwd(q, k, v, g, beta, h0, None, 0.6, eps=0.0)
    worst = 0.0
    ph = [2, 0, 1]
    o2, h2 = fwd(q[:, :, ph], k[:, :, ph], v[:, :, ph], g[:, :, ph], beta[:, :, ph],
                 h0[:, ph], None, 0.6, eps=0.0)
    worst = max(worst, _rel(o2, o[:, :, ph]), _rel(h2, hT[:, ph]))
    o3, h3 = fwd(q, k, 2.5 * v, g, beta, 2.5 * h0, None, 0.6, eps=0.0)
    worst = max(worst, _rel(o3, 2.5 * o), _rel(h3, 2.5 * hT))
    pv = rng.permutation(dv)
    o4, h4 = fwd(q, k, v[..., pv], g, beta, h0[..., pv], None, 0.6, eps=0.0)
    worst = max(worst, _rel(o4, o[..., pv]), _rel(h4, hT[..., pv]))
    cq = rng.uniform(0.01, 100.0, size=(B, T, H, 1))
    ck = rng.uniform(0.01, 100.0, size=(B, T, H, 1))
    o5, h5 = fwd(cq * q, ck * k, v, g, beta, h0, None, 0.6, eps=0.0)
    worst = max(worst, _rel(o5, o), _rel(h5, hT))
    return worst


PINS = {
    "brute": (pin_brute, 1e-12),
    "beta_zero": (pin_beta_zero, 1e-12),
    "delta_write": (pin_delta_write, 1e-10),
    "recall": (pin_recall, 1e-12),
    "varlen_split": (pin_varlen_split, 1e-13),
    "symmetries": (pin_symmetries, 1e-11),
}


def expected_reciprocal_norm(d: int, sigma: float) -> float:
    """E[1/|x|] for x ~ N(0, sigma^2 I_d): Gamma((d-1)/2) / (Gamma(d/2) sqrt(2) sigma)."""
    return math.exp(math.lgamma((d - 1) / 2) - math.lgamma(d / 2)) / (math.sqrt(2) * sigma)


