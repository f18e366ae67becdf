"""GPU parity of the single-token decode step (kda_decode) against the fp64 oracle.

A decode step is one token of the recurrence, so the oracle is the same token-by-token
fp64 recurrence the prefill tests use, run on sequences of length 1 (or, for chained
steps, on the whole sequence).  The kernel computes in fp32 throughout, so the gates
are far tighter than the prefill's: states and fp32 outputs within 1e-4 relative RMSE;
bf16 outputs carry their own rounding (about 2^-9 relative), gate 4e-3.
"""
from __future__ import annotations

import pytest
import torch

import oracle
from tests import gen
from tests.metrics import rel_rmse

pytestmark = pytest.mark.gpu

SALT = gen.fresh_salt()
TOL_F32 = 1e-4
TOL_BF16_O = 4e-3


@pytest.fixture(scope="module")
def kda():
    import __graft_entry__
    __graft_entry__.build()
    import gated_delta_rule_25_gb300 as m
    return m


def _one_token_each(N, H, dk, dv, dtype, seed):
    """N sequences of one token each (packed), with cfg2-style inputs and states."""
    return gen.make_lengths([1] * N, seed=seed, salt=SALT, H=H, dk=dk, dv=dv, dtype=dtype,
                            name="decode")


def _decode(kda, x, state=None, **kw):
    t = {n: getattr(x, n)[0].to("cuda") for n in ("q", "k", "v", "g", "beta")}
    st = x.h0.to("cuda") if state is None else state
    o, h = kda.decode(t["q"], t["k"], t["v"], t["g"], t["beta"], st, x.scale, **kw)
    torch.cuda.synchronize()
    return o, h


@pytest.mark.parametrize("dk,dv", [(128, 128), (64, 64), (64, 128), (128, 64)])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_decode_step_matches_oracle(kda, dk, dv, dtype):
    x = _one_token_each(37, 3, dk, dv, dtype, seed=dk + dv)
    o, h = _decode(kda, x)
    o_ref, h_ref = oracle.kda_recurrence_fp64(**x.tensors())
    eo = rel_rmse(o.cpu()[None], o_ref)
    eh = rel_rmse(h.cpu(), h_ref)
    msg = f"dk={dk} dv={dv} {dtype} salt={SALT}: o {eo:.2e} h {eh:.2e}"
    assert eh <= TOL_F32, msg
    assert eo <= (TOL_F32 if dtype == torch.float32 else TOL_BF16_O), msg


def test_chained_steps_equal_the_recurrence(kda):
    """T decode steps in a row give the recurrence over the T tokens (outputs and state)."""
    x = gen.make_cfg2(seed=3, salt=SALT, T=48, H=4, d=128, B=3, dtype=torch.float32)
    state = x.h0.to("cuda")
    outs = []
    for t in range(x.T):
        step = {n: getattr(x, n)[:, t].contiguous().to("cuda") for n in ("q", "k", "v", "g", "beta")}
        o, state = kda.decode(step["q"], step["k"], step["v"], step["g"], step["beta"], state,
                              x.scale)
        outs.append(o)
    torch.cuda.synchronize()
    o = torch.stack(outs, dim=1).cpu()
    o_ref, h_ref = oracle.kda_recurrence_fp64(**x.tensors())
    assert rel_rmse(state.cpu(), h_ref) <= TOL_F32
    assert rel_rmse(o, o_ref) <= TOL_F32


def test_in_place_and_zero_state(kda):
    x = _one_token_each(20, 4, 128, 128, torch.bfloat16, seed=5)
    o1, h1 = _decode(kda, x)
    st = x.h0.to("cuda").clone()
    o2, h2 = _decode(kda, x, state=st, out_state=st)   # update in place
    assert h2.data_ptr() == st.data_ptr()
    assert torch.equal(h1, h2) and torch.equal(o1, o2)
    # no state means zeros
    t = {n: getattr(x, n)[0].to("cuda") for n in ("q", "k", "v", "g", "beta")}
    o3, h3 = kda.decode(t["q"], t["k"], t["v"], t["g"], t["beta"], None, x.scale)
    o4, h4 = kda.decode(t["q"], t["k"], t["v"], t["g"], t["beta"],
                        torch.zeros_like(x.h0, device="cuda"), x.scale)
    torch.cuda.synchronize()
    assert torch.equal(h3, h4) and torch.equal(o3, o4)


def test_deep_gates_stay_finite(kda):
    x = _one_token_each(16, 2, 128, 128, torch.bfloat16, seed=9)
    x.g = torch.full_like(x.g, -1000.0)   # every state channel forgotten at once
    o, h = _decode(kda, x)
    o_ref, h_ref = oracle.kda_recurrence_fp64(**x.tensors())
    assert torch.isfinite(h).all() and torch.isfinite(o.float()).all()
    assert rel_rmse(h.cpu(), h_ref) <= TOL_F32
