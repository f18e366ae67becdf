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


def test_noalloc_binding_checks_arguments_before_any_launch(kda):
    """The binding checks every argument's dtype and shape before the C call (a wrong
    dtype would otherwise be read with the wrong element size on the device).  CPU
    tensors: each mistake raises before the device check is reached."""
    x = gen.make_lengths([70, 5], seed=24, salt=1, H=2, d=64)
    t = x.tensors()
    with pytest.raises(TypeError):       # this entry point takes only an fp32 gate
        kda.fwd_noalloc(**{**t, "g": t["g"].to(torch.bfloat16)})
    with pytest.raises(TypeError):       # q, k, v dtypes must agree
        kda.fwd_noalloc(**{**t, "k": t["k"].float()})
    with pytest.raises(TypeError):
        kda.fwd_noalloc(**{**t, "beta": t["beta"].double()})
    with pytest.raises(TypeError):
        kda.fwd_noalloc(**{**t, "cu_seqlens": t["cu_seqlens"].long()})
    with pytest.raises(ValueError):      # an output buffer one token short
        kda.fwd_noalloc(**t, o=torch.empty(1, x.T - 1, 2, 64, dtype=x.v.dtype))
    with pytest.raises(ValueError):      # a final-state buffer for the wrong N
        kda.fwd_noalloc(**t, hT=torch.empty(3, 2, 64, 64))
    with pytest.raises(ValueError):
        kda.fwd_noalloc(**{**t, "h0": t["h0"][:1].contiguous()})
    with pytest.raises(ValueError):      # right dtypes and shapes, but not on a GPU
        kda.fwd_noalloc(**t)


@pytest.mark.gpu
def test_noalloc_matches_fwd_on_two_calls_in_a_row(kda):
    """Both entry points run the same kernels on the same inputs, so the results are
    bit-identical; a stale or shared-scratch bug would show as any differing element."""
    cases = [gen.make_lengths([200, 1, 67, 0, 150], seed=21, salt=gen.fresh_salt(), H=4, d=128),
             gen.make_cfg2(seed=22, salt=gen.fresh_salt(), T=384, H=6, B=2),
             gen.make_cfg2(seed=26, salt=gen.fresh_salt(), T=384, H=16, B=2)]  # B*H = 32: fused
    assert kda.uses_fused(2, 384, 16, 128, 128, 2) and not kda.uses_fused(2, 384, 6, 128, 128, 2)
    for x in cases:  # two calls in a row share the built-in scratch
        xd = x.to("cuda")
        o_ref, h_ref = kda.fwd(**xd.tensors(), check=True)
        o_na = torch.empty_like(o_ref)
        h_na = torch.empty_like(h_ref)
        kda.fwd_noalloc(**xd.tensors(), o=o_na, hT=h_na, check=True)
        torch.cuda.synchronize()
        assert torch.equal(o_na, o_ref) and torch.equal(h_na, h_ref), x.name
        # and both within the parity gates of the oracle-checked path
        assert rel_rmse(o_na.cpu(), o_ref.cpu().double()) <= O_TOL
        assert rel_rmse(h_na.cpu(), h_ref.cpu().double()) <= HT_TOL


@pytest.mark.gpu
def test_noalloc_check_reports_malformed_cu_seqlens(kda):
    x = gen.make_lengths([10, 20, 34], seed=25, salt=gen.fresh_salt(), H=2, d=64)
    xd = x.to("cuda")
    xd.cu_seqlens = torch.tensor([0, 20, 10, 64], dtype=torch.int32, device="cuda")
    with pytest.raises(kda.KdaError) as e:
        kda.fwd_noalloc(**xd.tensors(), check=True)
    assert e.value.status == 6
    # the next well-formed call clears the word
    good = x.to("cuda")
    o, hT = kda.fwd_noalloc(**good.tensors(), check=True)
    o_ref, h_ref = kda.fwd(**good.tensors())
    assert torch.equal(o, o_ref) and torch.equal(hT, h_ref)


@pytest.mark.gpu
def test_noalloc_raises_on_oversized_problem(kda):
    x = gen.make_cfg2(seed=23, T=2048, H=32)  # 32 chunks x 32 heads of factors: above the array
    xd = x.to("cuda")
    with pytest.raises(kda.KdaError) as e:
        kda.fwd_noalloc(**xd.tensors())
    assert e.value.status == kda.KDA_ERR_TOO_LARGE
