"""Pins of the backward oracle (CPU): its forward is the C oracle's, its gradients
are the C oracle's finite differences, and the beta = 0 case has a closed form."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from oracle.backward import _spans, forward_torch, kda_backward_fp64
from tests import gen
from tests.metrics import rel_rmse

pytestmark = pytest.mark.filterwarnings("ignore::UserWarning")


def _f64(x):
    return x.double() if isinstance(x, torch.Tensor) else torch.from_numpy(np.asarray(x, dtype=np.float64))


def _grads_inputs(x, seed):
    rng = np.random.default_rng(seed)
    do = rng.standard_normal(tuple(x.v.shape))
    dhT = rng.standard_normal((x.num_seqs, x.H, x.dk, x.dv))
    return do, dhT


def test_forward_equals_c_oracle():
    x = gen.make_lengths([9, 0, 17, 1], seed=1, H=2, d=8)
    t = x.tensors()
    o_c, h_c = oracle.kda_recurrence_fp64(**t)
    o_t, h_t = forward_torch(*(_f64(t[n]) for n in ("q", "k", "v", "g", "beta")), _f64(t["h0"]),
                             _spans(x.B, x.T, x.cu_seqlens), x.scale)
    assert np.abs(o_t.numpy() - o_c).max() < 1e-12 and np.abs(h_t.numpy() - h_c).max() < 1e-12


@pytest.mark.parametrize("case", ["varlen", "fixed_no_h0"])
def test_gradients_match_finite_differences(case):
    """Directional derivatives of L = sum(o do) + sum(h_T dh_T), the function taken
    from the C oracle, by central differences (step 1e-5, fp64), against the
    backward oracle's gradients, in random directions for every input."""
    if case == "varlen":
        x = gen.make_lengths([5, 0, 7], seed=2, H=2, d=4)
    else:
        x = gen.make_cfg2(seed=3, T=6, H=2, d=4, B=2)
        x.h0 = None
    do, dhT = _grads_inputs(x, 4)
    t = {n: (_f64(v) if isinstance(v, torch.Tensor) and n != "cu_seqlens" else v) for n, v in x.tensors().items()}
    grads = kda_backward_fp64(**t, do=do, dhT=dhT)
    names = ("q", "k", "v", "g", "beta", "h0")

    def loss(tt):
        o, hT = oracle.kda_recurrence_fp64(**tt)
        return float((o * do).sum() + (hT * dhT).sum())

    rng = np.random.default_rng(5)
    for name, gr in zip(names, grads):
        base = t[name] if t[name] is not None else torch.zeros(x.num_seqs, x.H, x.dk, x.dv, dtype=torch.float64)
        for _ in range(2):
            d = torch.from_numpy(rng.standard_normal(tuple(base.shape)))
            eps = 1e-5
            tp, tm = dict(t), dict(t)
            tp[name], tm[name] = base + eps * d, base - eps * d
            fd = (loss(tp) - loss(tm)) / (2 * eps)
            an = float((torch.from_numpy(gr) * d).sum())
            assert abs(fd - an) <= 1e-6 * max(1.0, abs(an)), (name, fd, an)


def test_beta_zero_closed_form():
    """beta = 0: o_t = scale (Diag(exp Gamma_t) h0)^T qh_t and h_T = Diag(exp Gamma_T) h0,
    so dL/dGamma_t[c] and dL/dh0 have closed forms; dg is the suffix sum of the former."""
    x = gen.make_lengths([11], seed=6, H=1, d=4)
    x.beta = torch.zeros_like(x.beta)
    do, dhT = _grads_inputs(x, 7)
    t = x.tensors()
    dq, dk, dv, dg, dbeta, dh0 = kda_backward_fp64(**t, do=do, dhT=dhT)
    q = x.q[0, :, 0].double().numpy()
    g = x.g[0, :, 0].double().numpy()
    h0 = x.h0[0, 0].double().numpy()
    qh = q / np.sqrt((q * q).sum(-1, keepdims=True) + oracle.L2_EPS)
    G = np.cumsum(g, axis=0)                                   # Gamma_t, [T, dk]
    T = q.shape[0]
    dGam = np.zeros_like(G)
    for t_ in range(T):
        dGam[t_] += x.scale * np.exp(G[t_]) * qh[t_] * (h0 @ do[0, t_, 0])
    dGam[T - 1] += np.exp(G[T - 1]) * (h0 * dhT[0, 0]).sum(-1)
    dg_ref = np.cumsum(dGam[::-1], axis=0)[::-1]               # dL/dg_t = sum_{t' >= t} dL/dGamma_t'
    dh0_ref = sum(x.scale * np.outer(np.exp(G[t_]) * qh[t_], do[0, t_, 0]) for t_ in range(T)) \
        + np.exp(G[T - 1])[:, None] * dhT[0, 0]
    assert np.abs(dg[0, :, 0] - dg_ref).max() < 1e-12
    assert np.abs(dh0[0, 0] - dh0_ref).max() < 1e-12
    assert np.abs(dv).max() == 0.0 and np.abs(dk).max() == 0.0  # nothing is written
