"""The shortcuts described on the kernel-design-agents page (section 03 REWARD
HACKING, and the bf16 state of section 01 RESULTS) must fail the parity gates on
at least one synthetic recipe, while the exact chunkwise form passes them all.
CPU only; two heads at the full 8,192-token length."""
from __future__ import annotations

import functools

import pytest

import oracle
from oracle.chunked import kda_chunked_fp64
from oracle.mutants import kda_mutant
from tests import gen
from tests.metrics import passes, report

# recipe that exposes each shortcut (reduced to two heads)
CATCHES = {
    "M1": "cfg3", "M2": "cfg3", "M2b": "cfg2", "M3": "cfg3", "M4": "cfg2",
    "M5": "cfg4", "M6": "cfg4", "M7": "long_memory",
}


@functools.lru_cache(maxsize=None)
def _case(name):
    if name == "cfg2":
        x = gen.make_cfg2(seed=11, H=2)
    elif name == "cfg3":
        x = gen.make_cfg3(seed=11, H=2)
    elif name == "cfg4":
        x = gen.make_cfg4(seed=11, H=2)
    else:
        x = gen.make_probe(name, seed=11, T=8192, H=2, d=128)
    o, h = oracle.kda_recurrence_fp64(**x.tensors())
    return x, o, h


@pytest.mark.parametrize("kind", sorted(CATCHES))
def test_mutant_fails_gates(kind):
    x, o, h = _case(CATCHES[kind])
    om, hm = kda_mutant(kind, **x.tensors())
    rep = report(om, hm, o, h)
    assert not passes(rep), f"{kind} passed the gates on {CATCHES[kind]}: {rep}"


@pytest.mark.parametrize("name", sorted(set(CATCHES.values())))
def test_exact_chunked_form_passes(name):
    x, o, h = _case(name)
    oc, hc = kda_chunked_fp64(**x.tensors())
    rep = report(oc, hc, o, h)
    assert passes(rep) and rep["o_rel_rmse"] < 1e-12 and rep["hT_rel_rmse"] < 1e-12, rep


def test_generators_are_not_gaussian_half():
    """The M1 constant equals E[1/|x|] only for N(0, 0.5^2) rows at d = 128; the
    recipes' mean reciprocal norm must be far from it."""
    from oracle.mutants import HACK_RSQRT
    x = gen.make_cfg2(seed=3, T=512, H=4)
    inv = 1.0 / x.q.float().norm(dim=-1)
    assert abs(float(inv.mean()) - HACK_RSQRT) > 0.05
