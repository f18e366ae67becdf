"""GPU parity of the backward pass (kda_bwd) against the fp64 autograd oracle
(oracle/backward.py, pinned in test_backward_oracle.py).

Every gradient (dq, dk, dv, dg, dbeta, dh0) is compared element by element through
its relative RMSE.  The kernel runs fp32 arithmetic throughout on the exact stored
inputs, so the gate is 1e-4: fp32 rounding accumulated over a few hundred dependent
steps stays near 1e-6 relative, and any wrong term (a dropped decay, a sign, a
transposed product, a missed normalisation) moves a gradient by O(1).
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

from oracle.backward import kda_backward_fp64
from tests import gen
from tests.metrics import rel_rmse
from tests.test_gpu_parity import SALT

pytestmark = pytest.mark.gpu

TOL = 1e-4
NAMES = ("dq", "dk", "dv", "dg", "dbeta", "dh0")


@pytest.fixture(scope="module")
def kda():
    import __graft_entry__
    __graft_entry__.build()
    import gated_delta_rule_25_gb300 as m
    return m


def _check(kda, x, seed=0, with_dhT=True, tol=TOL):
    rng = np.random.default_rng(seed)
    do = torch.from_numpy(rng.standard_normal(tuple(x.v.shape)).astype(np.float32)).to(x.v.dtype)
    dhT = (torch.from_numpy(rng.standard_normal((x.num_seqs, x.H, x.dk, x.dv)).astype(np.float32))
           if with_dhT else None)
    xd = x.to("cuda")
    got = kda.bwd(**xd.tensors(), do=do.to("cuda"), dhT=None if dhT is None else dhT.to("cuda"), check=True)
    torch.cuda.synchronize()
    ref = kda_backward_fp64(**x.tensors(), do=do.double(), dhT=None if dhT is None else dhT.double())
    errs = {}
    for name, a, r in zip(NAMES, got, ref):
        a = a.cpu()
        assert torch.isfinite(a).all(), name
        errs[name] = rel_rmse(a, r) if np.abs(r).max() > 0 else float(a.abs().max())
    assert all(e <= tol for e in errs.values()), f"{x.name} salt={x.salt}: {errs}"
    return errs


def test_bwd_varlen(kda):
    """Ragged sequences (partial chunks, an empty one, a one-token one)."""
    x = gen.make_lengths([70, 0, 130, 1], seed=50, salt=SALT, H=2, d=128)
    _check(kda, x)


def test_bwd_fixed_length(kda):
    x = gen.make_cfg2(seed=51, salt=SALT, T=200, H=2, B=2)
    _check(kda, x, seed=1)


def test_bwd_without_states(kda):
    """No h0 (zero initial state) and no dhT."""
    x = gen.make_cfg2(seed=52, salt=SALT, T=150, H=2, B=1)
    x.h0 = None
    _check(kda, x, seed=2, with_dhT=False)


def test_bwd_many_chunks(kda):
    """Sixteen chunks: the checkpoints and the per-chunk recompute across many chunk
    boundaries."""
    x = gen.make_cfg2(seed=53, salt=SALT, T=1000, H=1, B=1)
    _check(kda, x, seed=3)


@pytest.mark.parametrize("d", [(64, 64), (64, 128), (128, 64)])
def test_bwd_head_dims(kda, d):
    dk, dv = d
    x = gen.make_lengths([90, 40], seed=54, salt=SALT, H=2, dk=dk, dv=dv)
    _check(kda, x, seed=4)


def test_bwd_fp32_inputs(kda):
    x = gen.make_cfg1(seed=55, salt=SALT, T=120, H=2, d=128)
    _check(kda, x, seed=5)


@pytest.mark.parametrize("kind", ["deep", "saturated", "repeated_keys", "beta01", "zero_rows"])
def test_bwd_probes(kda, kind):
    x = gen.make_probe(kind, seed=56, salt=SALT, T=150, H=2, d=128)
    _check(kda, x, seed=6)


def test_bwd_many_chains(kda):
    """More (sequence, head) chains than SMs: CTAs take several chains in turn."""
    lens = [5, 0, 70, 1, 33] * 40
    x = gen.make_lengths(lens, seed=57, salt=SALT, H=1, d=64)
    assert x.num_seqs * x.H > 152
    _check(kda, x, seed=7)


@pytest.mark.parametrize("name", ["cfg2", "cfg3"])
def test_bwd_full_size_sampled_heads(kda, name):
    """The full cfg2 (8,192 tokens x 32 heads) and cfg3 (varlen) sizes through the GPU
    backward; the oracle checks two heads (the heads are independent chains)."""
    x = {"cfg2": gen.make_cfg2, "cfg3": gen.make_cfg3}[name](seed=58, salt=SALT)
    rng = np.random.default_rng(8)
    do = torch.from_numpy(rng.standard_normal(tuple(x.v.shape)).astype(np.float32)).to(x.v.dtype)
    dhT = torch.from_numpy(rng.standard_normal((x.num_seqs, x.H, x.dk, x.dv)).astype(np.float32))
    xd = x.to("cuda")
    got = kda.bwd(**xd.tensors(), do=do.to("cuda"), dhT=dhT.to("cuda"), check=True)
    torch.cuda.synchronize()
    hs = [0, x.H - 1]
    t = x.tensors()
    for key in ("q", "k", "v", "g", "beta"):
        t[key] = t[key][:, :, hs].contiguous()
    t["h0"] = t["h0"][:, hs].contiguous()
    ref = kda_backward_fp64(**t, do=do[:, :, hs].double(), dhT=dhT[:, hs].double())
    errs = {}
    for name_, a, r in zip(NAMES, got, ref):
        a = a.cpu()
        a = a[:, hs] if name_ == "dh0" else a[:, :, hs]
        errs[name_] = rel_rmse(a, r)
    assert all(e <= TOL for e in errs.values()), f"{x.name} salt={x.salt}: {errs}"
