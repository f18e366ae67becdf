"""Segmented chains: the exact inter-chunk split of few long (sequence, head) chains.

A chain of chunk steps S <- M_c S + D_c is cut into segments; pass A runs the first
segment from h0 and, for every middle segment, its map F (the product of its M_c)
and its state from zero Z, all at once; a scan gives each segment's start state
(F E + Z); pass C reruns the later segments from those, writing o and h_T.  The
split pipeline takes it for at most 64 chains at dk = dv = 128 where it is predicted
faster: chosen on the host for equal-length chains, on the device from the lengths
for varlen batches.  Every case is checked against the fp64 oracle with the gates of
test_gpu_parity.py, and the header words say which path ran.
"""
from __future__ import annotations

import pytest
import torch

from tests import gen
from tests.test_gpu_parity import SALT, _assert_parity, _gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def kda():
    import __graft_entry__
    __graft_entry__.build()
    import gated_delta_rule_25_gb300 as m
    return m


def _run_with_header(kda, x, **kw):
    """The forward with an explicit workspace; returns o, h_T and the header words
    {chain128, seg, tasks of pass A, tasks of pass C, scan pairs, segment length}."""
    xd = x.to("cuda")
    ws = torch.empty(kda.workspace_size(x.B, x.T, x.H, x.dk, x.dv, x.num_seqs) + 256,
                     dtype=torch.uint8, device="cuda")
    o, hT = kda.fwd(**xd.tensors(), workspace=ws, check=True, **kw)
    torch.cuda.synchronize()
    base = (-ws.data_ptr()) % 256
    words = ws[base:base + 40].cpu().numpy().view("int32").tolist()
    keys = ("chain128", "seg", "seg_na", "seg_nc", "seg_ns", "seg_len")
    return o.cpu(), (hT.cpu() if hT is not None else None), dict(zip(keys, words[4:10]))


def test_segments_fixed_length(kda):
    """One sequence of 8,192 tokens at H = 4: 128-step chains cut into segments
    (equal lengths: the host picks the segment length; five launches)."""
    x = gen.make_cfg2(seed=30, salt=SALT, T=8192, H=4, B=1)
    assert kda.launch_count(x.B, x.T, x.H, x.dk, x.dv, x.num_seqs) == 5
    o, hT, hdr = _run_with_header(kda, x)
    assert hdr["seg"] == 1 and hdr["seg_len"] >= 1 and hdr["seg_ns"] > 0
    assert hdr["seg_nc"] >= 2 * x.H
    _assert_parity(x, o, hT)


def test_segments_ragged_tail_chunk(kda):
    """A length that is not a multiple of 64 and a last segment shorter than the rest:
    the partial chunk's rows and the short tail segment through pass C."""
    x = gen.make_lengths([64 * 90 + 13], seed=31, salt=SALT, H=3, d=128)
    o, hT, hdr = _run_with_header(kda, x)
    assert hdr["seg"] == 1
    _assert_parity(x, o, hT)


def test_segments_two_batch_rows(kda):
    """B = 2 fixed-length rows: the task lists cover both sequences' chains."""
    x = gen.make_cfg2(seed=32, salt=SALT, T=6144, H=3, B=2)
    o, hT, hdr = _run_with_header(kda, x)
    assert hdr["seg"] == 1
    _assert_parity(x, o, hT)


def test_segments_varlen_decided_on_device(kda):
    """A varlen batch with few chains, one long sequence, an empty one and short ones:
    the schedule kernel chooses segments from the lengths (six launches, the tiled state
    kernel leaving at once); the short sequences run whole in pass A, the empty one
    passes h0 through."""
    x = gen.make_lengths([6000, 0, 1500, 200, 64, 1], seed=33, salt=SALT, H=4, d=128)
    assert kda.launch_count(x.B, x.T, x.H, x.dk, x.dv, x.num_seqs) == 6
    o, hT, hdr = _run_with_header(kda, x)
    assert hdr["seg"] == 1
    assert torch.equal(hT[1], x.h0[1])
    _assert_parity(x, o, hT)


def test_segments_not_chosen_for_short_chains(kda):
    """64-chunk chains: the scan's serial steps cost more than segments save, so the
    host keeps the tiled state kernel (three launches)."""
    x = gen.make_cfg2(seed=39, salt=SALT, T=4096, H=4, B=1)
    assert kda.launch_count(x.B, x.T, x.H, x.dk, x.dv, x.num_seqs) == 3
    o, hT, hdr = _run_with_header(kda, x)
    assert hdr["seg"] == 0
    _assert_parity(x, o, hT)


def test_segments_varlen_not_chosen(kda):
    """Varlen chains too short for segments to pay: the tiled state kernel runs."""
    x = gen.make_lengths([700, 900, 500], seed=34, salt=SALT, H=2, d=128)
    o, hT, hdr = _run_with_header(kda, x)
    assert hdr["seg"] == 0
    _assert_parity(x, o, hT)


def test_segments_without_initial_or_final_state(kda):
    """No h0 (zero initial state) and no h_T requested."""
    x = gen.make_cfg2(seed=35, salt=SALT, T=8192, H=2, B=1)
    x.h0 = None
    o, hT, hdr = _run_with_header(kda, x, output_final_state=False)
    assert hdr["seg"] == 1 and hT is None
    _assert_parity(x, o, None)


@pytest.mark.parametrize("kind", gen.PROBES)
def test_segments_probes(kda, kind):
    """The stress probes through segmented chains: the maps F carry the extreme
    gates (deep and abyss decay, no decay, one repeated key, beta in {0, 1}).  8,192
    tokens (128 chunks, cut into segments); beta0's gates are scaled by 1/4, since its
    pure decay would take the true final state below the fp32 range (about
    exp(-250) h0 at 8,192 tokens; exp(-62) h0 scaled)."""
    T = 8192
    assert kda.launch_count(1, T, 2, 128, 128, 1) == 5
    x = gen.make_probe(kind, seed=36, salt=SALT, T=T, H=2, d=128)
    if kind == "beta0":
        x.g = x.g * 0.25
    o, hT, hdr = _run_with_header(kda, x)
    assert hdr["seg"] == 1
    _assert_parity(x, o, hT)


def test_segments_fp32_inputs(kda):
    """fp32 q, k, v: the factor kernel writes u in the chain layout on tf32 operands."""
    x = gen.make_cfg1(seed=37, salt=SALT, T=8192, H=2, d=128)
    o, hT, hdr = _run_with_header(kda, x)
    assert hdr["seg"] == 1
    _assert_parity(x, o, hT)


def test_segments_agree_with_fused(kda):
    """The same batch segmented (split pipeline) and unsegmented (fused pipeline): each
    is within the oracle's gates; here, that they agree."""
    x = gen.make_cfg2(seed=38, salt=SALT, T=8192, H=16, B=1)
    o_s, h_s, hdr = _run_with_header(kda, x)
    assert hdr["seg"] == 1
    try:
        kda.set_pipeline("fused")
        o_f, h_f = _gpu(kda, x)
    finally:
        kda.set_pipeline("auto")
    from tests.metrics import rel_rmse
    assert rel_rmse(o_s, o_f.double()) <= 1e-2
    assert rel_rmse(h_s, h_f.double()) <= 5e-3
    _assert_parity(x, o_s, h_s, heads=[0, 7, 15])


def test_segments_one_long_sequence(kda):
    """A single 131,072-token sequence at H = 1: a 2,048-step chain cut into dozens of
    segments (the whole sequence against the oracle)."""
    x = gen.make_cfg2(seed=40, salt=SALT, T=131072, H=1, B=1)
    assert kda.launch_count(x.B, x.T, x.H, x.dk, x.dv, x.num_seqs) == 5
    o, hT, hdr = _run_with_header(kda, x)
    assert hdr["seg"] == 1 and hdr["seg_ns"] == 1
    _assert_parity(x, o, hT)
