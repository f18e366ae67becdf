"""TEST INFRASTRUCTURE ONLY: exact rational brute force for tiny KDA inputs.

Two independent exact forms of the gated delta rule, used to pin the fp64
oracle (``kda_oracle.c``) on inputs small enough for ``fractions.Fraction``:

* ``brute_recurrence``: the per-token update written with explicit matrices in
  the form the method is usually stated in,
  ``S_t = (I - beta_t k_t k_t^T) Diag(alpha_t) S_{t-1} + beta_t k_t v_t^T`` and
  ``o_t = scale * S_t^T q_t`` ("Autoresearch on Kimi Delta Attention", section THE
  MECHANISM: each token reads the memory's prediction and writes the correction,
  with a per-channel forget rate).
* ``brute_unrolled``: the same state unrolled as a sum over tokens of products of
  transition matrices, ``S_t = M_t...M_1 S_0 + sum_i M_t...M_{i+1} beta_i k_i v_i^T``
  with ``M_t = (I - beta_t k_t k_t^T) Diag(alpha_t)``.

Keys and queries must have rational L2 norms (for example (3/5, 4/5, 0, 0)
scaled by a rational), so that the normalisation is exact.  The
normalisation epsilon is zero here, so the fp64 oracle must be called with
``eps=0`` when compared against these forms.
"""
from __future__ import annotations

from fractions import Fraction
from math import isqrt
from typing import List, Sequence

Mat = List[List[Fraction]]


def _exact_sqrt(x: Fraction) -> Fraction:
    if x < 0:
        raise ValueError("negative")
    n, d = x.numerator, x.denominator
    rn, rd = isqrt(n), isqrt(d)
    if rn * rn != n or rd * rd != d:
        raise ValueError(f"{x} is not the square of a rational")
    return Fraction(rn, rd)


def normalise(x: Sequence[Fraction]) -> List[Fraction]:
    """x / |x| exactly; requires |x| rational and nonzero."""
    nrm = _exact_sqrt(sum((Fraction(c) * Fraction(c) for c in x), Fraction(0)))
    if nrm == 0:
        raise ValueError("zero vector")
    return [Fraction(c) / nrm for c in x]


def _zeros(r: int, c: int) -> Mat:
    return [[Fraction(0)] * c for _ in range(r)]


def _eye(n: int) -> Mat:
    m = _zeros(n, n)
    for i in range(n):
        m[i][i] = Fraction(1)
    return m


def _matmul(a: Mat, b: Mat) -> Mat:
    n, kk, m = len(a), len(b), len(b[0])
    return [[sum((a[i][p] * b[p][j] for p in range(kk)), Fraction(0)) for j in range(m)]
            for i in range(n)]


def _add(a: Mat, b: Mat) -> Mat:
    return [[a[i][j] + b[i][j] for j in range(len(a[0]))] for i in range(len(a))]


def _outer(x: Sequence[Fraction], y: Sequence[Fraction], s: Fraction = Fraction(1)) -> Mat:
    return [[s * xi * yj for yj in y] for xi in x]


def transition(kh: Sequence[Fraction], alpha: Sequence[Fraction], beta: Fraction) -> Mat:
    """M = (I - beta kh kh^T) Diag(alpha), a dense dk x dk matrix."""
    dk = len(kh)
    proj = _add(_eye(dk), _outer(kh, kh, -Fraction(beta)))
    diag = _zeros(dk, dk)
    for i in range(dk):
        diag[i][i] = Fraction(alpha[i])
    return _matmul(proj, diag)


def _readout(S: Mat, qh: Sequence[Fraction], scale: Fraction) -> List[Fraction]:
    dk, dv = len(S), len(S[0])
    return [scale * sum((S[i][j] * qh[i] for i in range(dk)), Fraction(0)) for j in range(dv)]


def brute_recurrence(q, k, v, alpha, beta, S0, scale):
    """Exact per-token form.  q, k, alpha: T lists of dk; v: T lists of dv;
    beta: T values; S0: dk x dv.  Returns (o: T lists of dv, S_T)."""
    S = [[Fraction(x) for x in row] for row in S0]
    outs = []
    for t in range(len(q)):
        kh, qh = normalise(k[t]), normalise(q[t])
        M = transition(kh, alpha[t], Fraction(beta[t]))
        S = _add(_matmul(M, S), _outer(kh, v[t], Fraction(beta[t])))
        outs.append(_readout(S, qh, Fraction(scale)))
    return outs, S


def brute_unrolled(q, k, v, alpha, beta, S0, scale):
    """Exact unrolled form: S_t = P_{t,0} S_0 + sum_i P_{t,i} beta_i k_i v_i^T with
    P_{t,i} = M_t ... M_{i+1}.  Independent of ``brute_recurrence``'s loop order."""
    T = len(q)
    dk = len(k[0]) if T else len(S0)
    khs = [normalise(k[t]) for t in range(T)]
    Ms = [transition(khs[t], alpha[t], Fraction(beta[t])) for t in range(T)]
    S0f = [[Fraction(x) for x in row] for row in S0]
    outs = []
    S_t = S0f
    for t in range(T):
        # P_{t,i} built right to left for every i <= t
        acc = _zeros(dk, len(S0[0]))
        P = _eye(dk)
        for i in range(t, -1, -1):
            acc = _add(acc, _matmul(P, _outer(khs[i], v[i], Fraction(beta[i]))))
            P = _matmul(P, Ms[i])
        S_t = _add(_matmul(P, S0f), acc)
        outs.append(_readout(S_t, normalise(q[t]), Fraction(scale)))
    return outs, S_t
