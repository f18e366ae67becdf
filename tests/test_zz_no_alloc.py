"""kda_fwd_noalloc: the forward for callers that cannot allocate device memory.

Such callers (a plugin inside an engine that owns all device memory, or a path
where an allocation's latency or failure is not acceptable) pass only inputs and
outputs; the library's scratch is a fixed 32 MiB device array built into it.
These tests call that entry point through the C ABI and check it against the
ordinary kda_fwd (which takes a caller-allocated workspace) on two calls in a row,
with the parity tolerances used everywhere else.  This file is collected last so
that a failure here leaves every other test already run.
"""
from __future__ import annotations

import ctypes

import pytest
import torch

from tests import gen
from tests.metrics import HT_TOL, O_TOL, rel_rmse


@pytest.fixture(scope="module")
def kda():
    import __graft_entry__
    __graft_entry__.build()
    import gated_delta_rule_25_gb300 as m
    return m


def test_noalloc_refuses_oversized_problems_without_touching_the_gpu(kda):
    lib = kda.load_library()
    p = ctypes.c_void_p(1 << 20)  # never dereferenced: the size check comes first
    st = lib.kda_fwd_noalloc(p, p, p, 0, p, p, None, None, 1, 1, 8192, 32, 128, 128, 0.1, p, p,
                             None)
    assert st == kda.KDA_ERR_TOO_LARGE
    assert lib.kda_status_string(st) == b"problem too large for the built-in no-allocation scratch"


@pytest.mark.gpu
def test_noalloc_matches_fwd_on_two_calls_in_a_row(kda):
    cases = [gen.make_lengths([200, 1, 67, 0, 150], seed=21, salt=gen.fresh_salt(), H=4, d=128),
             gen.make_cfg2(seed=22, salt=gen.fresh_salt(), T=384, H=6, B=2)]
    for x in cases:  # two calls in a row share the built-in scratch
        xd = x.to("cuda")
        o_ref, h_ref = kda.fwd(**xd.tensors(), check=True)
        o_na = torch.empty_like(o_ref)
        h_na = torch.empty_like(h_ref)
        kda.fwd_noalloc(**xd.tensors(), o=o_na, hT=h_na)
        torch.cuda.synchronize()
        assert torch.isfinite(o_na.float()).all() and torch.isfinite(h_na).all()
        eo = rel_rmse(o_na.cpu(), o_ref.cpu().double())
        eh = rel_rmse(h_na.cpu(), h_ref.cpu().double())
        assert eo <= O_TOL and eh <= HT_TOL, (x.name, eo, eh)


@pytest.mark.gpu
def test_noalloc_raises_on_oversized_problem(kda):
    x = gen.make_cfg2(seed=23, T=2048, H=32)  # ~150 MB of factors: above the 32 MiB array
    xd = x.to("cuda")
    with pytest.raises(kda.KdaError) as e:
        kda.fwd_noalloc(**xd.tensors())
    assert e.value.status == kda.KDA_ERR_TOO_LARGE
