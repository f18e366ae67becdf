"""The two pipelines of the forward: which one a call takes, and parity of each.

The fused pipeline runs factor production and the state chains in one cooperative
kernel (dk = dv = 128); the split one (a factor kernel, then a state kernel) serves
every size.  The automatic choice takes the fused one for fixed-length batches with
32 <= B * H <= 256 whose split pipeline would keep the tiled state kernel, so most of
test_gpu_parity.py runs split; the cases here force
the fused pipeline on varlen batches, edge cases and probes, and the split one on
the configs, all against the fp64 oracle with the gates of test_gpu_parity.py.
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


@pytest.fixture
def split(kda):
    kda.set_pipeline("split")
    try:
        yield kda
    finally:
        kda.set_pipeline("auto")


@pytest.fixture
def fused(kda):
    kda.set_pipeline("fused")
    try:
        yield kda
    finally:
        kda.set_pipeline("auto")


def test_pipeline_selection(kda):
    assert kda.get_pipeline() == "auto"
    assert kda.uses_fused(1, 8192, 32, 128, 128, 1)             # B * H = 32, fixed length
    assert kda.uses_fused(4, 8192, 16, 128, 128, 4)             # B * H = 64
    assert not kda.uses_fused(4, 8192, 64, 128, 128, 4)         # B * H = 256: split takes 128-column chains
    assert not kda.uses_fused(4, 8192, 32, 128, 128, 4)         # B * H = 128: the same
    assert not kda.uses_fused(1, 8192, 16, 128, 128, 1)         # B * H = 16: split is faster
    assert not kda.uses_fused(16, 8192, 32, 128, 128, 16)       # B * H = 512
    assert not kda.uses_fused(1, 8192, 32, 128, 128, 8)         # varlen
    assert not kda.uses_fused(1, 256, 32, 64, 64, 1)            # dk = dv = 64
    assert kda.launch_count(1, 8192, 32, 128, 128, 1) == 2           # schedule, fused
    assert kda.launch_count(1, 8192, 32, 128, 128, 8) == 3           # varlen, 256 chains
    assert kda.launch_count(1, 8192, 32, 128, 128, 16) == 4          # varlen, 512: both state kernels
    assert kda.launch_count(1, 256, 32, 64, 64, 1) == 3
    kda.set_pipeline("fused")
    try:
        assert kda.get_pipeline() == "fused"
        assert kda.uses_fused(1, 8192, 32, 128, 128, 2048)      # varlen, 2048 sequences
        assert kda.uses_fused(1, 8192, 16, 128, 128, 1)
        assert not kda.uses_fused(1, 8192, 32, 128, 128, 2049)  # beyond the ranking
        assert not kda.uses_fused(1, 256, 2, 64, 64, 1)         # dk = dv = 64
        assert not kda.uses_fused(1, 256, 2, 128, 64, 1)
    finally:
        kda.set_pipeline("auto")
    kda.set_pipeline("split")
    try:
        assert not kda.uses_fused(1, 8192, 32, 128, 128, 1)
        assert kda.launch_count(1, 8192, 32, 128, 128, 1) == 3           # one state kernel
    finally:
        kda.set_pipeline("auto")
    with pytest.raises(ValueError):
        kda.set_pipeline("other")


@pytest.mark.parametrize("name", ["cfg2", "cfg3", "cfg4"])
def test_split_pipeline_parity(split, name):
    x = getattr(gen, f"make_{name}")(seed=3, salt=SALT)
    heads = [0, x.H // 2, x.H - 1]
    _assert_parity(x, *_gpu(split, x), heads=heads)


def test_split_pipeline_head_dims_128(split):
    x = gen.make_lengths([70, 1, 129, 64, 0, 33] * 4, seed=8, salt=SALT, H=4, d=128)
    _assert_parity(x, *_gpu(split, x))


@pytest.mark.parametrize("name", ["cfg3", "cfg4"])
def test_fused_pipeline_varlen_configs(fused, name):
    x = getattr(gen, f"make_{name}")(seed=4, salt=SALT)
    assert fused.uses_fused(x.B, x.T, x.H, x.dk, x.dv, x.num_seqs)
    _assert_parity(x, *_gpu(fused, x), heads=[0, x.H // 2, x.H - 1])


def test_fused_pipeline_boundary_lengths(fused):
    x = gen.make_lengths([1, 63, 64, 65, 127, 128, 129, 0, 2], seed=5, salt=SALT, H=2, d=128)
    _assert_parity(x, *_gpu(fused, x))


@pytest.mark.parametrize("kind", gen.PROBES)
def test_fused_pipeline_probes(fused, kind):
    T = 8192 if kind == "long_memory" else 300
    x = gen.make_probe(kind, seed=6, salt=SALT, T=T, H=2, d=128)
    _assert_parity(x, *_gpu(fused, x))


def test_fused_pipeline_varlen_equals_independent(fused):
    x = gen.make_lengths([300, 1, 64, 129], seed=7, salt=SALT, H=4, d=128)
    o, hT = _gpu(fused, x)
    cu = x.cu_seqlens.tolist()
    for s in range(len(cu) - 1):
        a, b = cu[s], cu[s + 1]
        xs = gen.KdaInputs("one", x.q[:, a:b].contiguous(), x.k[:, a:b].contiguous(),
                           x.v[:, a:b].contiguous(), x.g[:, a:b].contiguous(),
                           x.beta[:, a:b].contiguous(), x.h0[s:s + 1].contiguous(), None,
                           x.scale)
        o1, h1 = _gpu(fused, xs)
        assert torch.equal(o1, o[:, a:b]) and torch.equal(h1[0], hT[s])


def test_fused_many_rounds_and_empty_chains(fused):
    """More chains than chain CTAs (several rounds), chains of one step, empty ones,
    and one long chain that sets the critical path."""
    lens = [0, 1, 64, 65, 3000, 0, 17, 128] * 9 + [0, 0]
    x = gen.make_lengths(lens, seed=12, salt=SALT, H=6, d=128)
    assert fused.uses_fused(x.B, x.T, x.H, x.dk, x.dv, x.num_seqs)
    _assert_parity(x, *_gpu(fused, x))


def test_fused_single_step_chains(fused):
    """Hundreds of one-chunk chains per chain CTA: every step starts a new chain."""
    lens = [64, 1, 37, 64, 50] * 40
    x = gen.make_lengths(lens, seed=13, salt=SALT, H=8, d=128)
    _assert_parity(x, *_gpu(fused, x))


def test_fused_all_sequences_empty(fused):
    """No token at all: the states pass through (h_T = h0) and nothing else runs."""
    x = gen.make_lengths([0, 0, 0], seed=14, salt=SALT, H=3, d=128)
    o, hT = _gpu(fused, x)
    assert o.numel() == 0
    assert torch.equal(hT, x.h0)


def test_fused_pipeline_bf16_gate(fused):
    """A bf16 gate through the fused pipeline: parity, and bit-identical to the fp32
    gate fed the same values."""
    x = gen.make_cfg2(seed=16, salt=SALT, T=300, H=16, B=2)
    x.g = x.g.to(torch.bfloat16)
    o16, h16 = _gpu(fused, x)
    _assert_parity(x, o16, h16)
    x32 = gen.make_cfg2(seed=16, salt=SALT, T=300, H=16, B=2)
    x32.g = x.g.float()
    o32, h32 = _gpu(fused, x32)
    assert torch.equal(o16, o32) and torch.equal(h16, h32)


def test_fused_pipeline_fp32_inputs(fused):
    """fp32 q, k, v at d = 128 through the fused pipeline (u on tf32 operands, the
    [64/4][dv][4] layout written by scalar stores)."""
    x = gen.make_cfg1(seed=17, salt=SALT, T=300, H=4, d=128)
    assert fused.uses_fused(x.B, x.T, x.H, x.dk, x.dv, x.num_seqs)
    _assert_parity(x, *_gpu(fused, x))


def _chain128_chosen(kda, x):
    """Runs the forward with an explicit workspace and reads the schedule kernel's
    choice of state kernel (the header's fifth word)."""
    xd = x.to("cuda")
    ws = torch.empty(kda.workspace_size(x.B, x.T, x.H, x.dk, x.dv, x.num_seqs) + 256,
                     dtype=torch.uint8, device="cuda")
    o, hT = kda.fwd(**xd.tensors(), workspace=ws, check=True)
    torch.cuda.synchronize()
    base = (-ws.data_ptr()) % 256
    word = int(ws[base + 16:base + 20].cpu().numpy().view("int32")[0])
    return o.cpu(), hT.cpu(), word


def test_split_pipeline_chain128_fixed(kda):
    """B * H = 512 chains of 8 chunks: the split pipeline with the 128-column chain
    kernel alone (predicted 80 us against 108 us for 64-column tiles)."""
    x = gen.make_cfg2(seed=18, salt=SALT, T=512, H=64, B=8)
    assert not kda.uses_fused(x.B, x.T, x.H, x.dk, x.dv, x.num_seqs)
    assert kda.launch_count(x.B, x.T, x.H, x.dk, x.dv, x.num_seqs) == 3
    o, hT, chosen = _chain128_chosen(kda, x)
    assert chosen == 1
    _assert_parity(x, o, hT, heads=[0, 31, 63])


def test_split_pipeline_chain128_varlen(kda):
    """Many varlen chains, empty sequences included, through the 128-column chain
    kernel when the schedule picks it; parity either way."""
    lens = [150, 0, 77, 300, 1, 64, 129, 200] * 24
    x = gen.make_lengths(lens, seed=19, salt=SALT, H=8, d=128)
    assert x.num_seqs * x.H >= 512
    o, hT, chosen = _chain128_chosen(kda, x)
    assert chosen == 1
    _assert_parity(x, o, hT)


def test_split_pipeline_tiled_state_kernel_when_few_chains(kda):
    """Few long chains: the schedule keeps the tiled state kernel."""
    x = gen.make_cfg2(seed=20, salt=SALT, T=2048, H=16, B=1)
    o, hT, chosen = _chain128_chosen(kda, x)
    assert chosen == 0
    _assert_parity(x, o, hT, heads=[0, 15])


def test_fused_and_split_agree(kda):
    """Both pipelines on the same varlen batch stay within the gates of each other's
    reference (each is checked against the oracle; here only that they agree)."""
    x = gen.make_cfg3(seed=15, salt=SALT)
    try:
        kda.set_pipeline("split")
        o_s, h_s = _gpu(kda, x)
        kda.set_pipeline("fused")
        o_f, h_f = _gpu(kda, x)
    finally:
        kda.set_pipeline("auto")
    from tests.metrics import rel_rmse
    assert rel_rmse(o_f, o_s.double()) <= 1e-2
    assert rel_rmse(h_f, h_s.double()) <= 5e-3
