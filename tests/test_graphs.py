"""CUDA-graph capture of every path: the cooperative fused kernel, the segmented
split pipeline and the backward pass are captured once, replayed on fresh inputs
swapped into the captured buffers, and compared bit for bit with eager calls on the
same inputs ("NVIDIA Kernel Design Agents optimize Kimi Delta Attention", section 04
HARDENING: CUDA Graph replay checks)."""
from __future__ import annotations

import numpy as np
import pytest
import torch

from tests import gen
from tests.test_gpu_parity import SALT

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def kda():
    import __graft_entry__
    __graft_entry__.build()
    import gated_delta_rule_25_gb300 as m
    return m


def _capture(fn):
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn()  # warm-up outside the capture (kernel attributes are set once, here)
    torch.cuda.current_stream().wait_stream(s)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        fn()
    return graph


@pytest.mark.parametrize("path", ["fused", "segments"])
def test_forward_graph_replay(kda, path):
    if path == "fused":
        mk = lambda seed, salt: gen.make_cfg2(seed=seed, salt=salt, T=384, H=16, B=2)
    else:
        mk = lambda seed, salt: gen.make_cfg2(seed=seed, salt=salt, T=8192, H=2, B=1)
    x1, x2 = mk(60, SALT), mk(61, SALT + 1)
    assert kda.uses_fused(x1.B, x1.T, x1.H, x1.dk, x1.dv, x1.num_seqs) == (path == "fused")
    if path == "segments":
        assert kda.launch_count(x1.B, x1.T, x1.H, x1.dk, x1.dv, x1.num_seqs) == 5
    d1 = x1.to("cuda")
    ws = torch.empty(kda.workspace_size(x1.B, x1.T, x1.H, 128, 128, x1.num_seqs) + 256,
                     dtype=torch.uint8, device="cuda")
    o, hT = torch.empty_like(d1.v), torch.empty_like(d1.h0)
    graph = _capture(lambda: kda.fwd(**d1.tensors(), o=o, hT=hT, workspace=ws))
    for x in (x1, x2):
        for name in ("q", "k", "v", "g", "beta", "h0"):
            getattr(d1, name).copy_(getattr(x, name).to("cuda"))
        graph.replay()
        torch.cuda.synchronize()
        o_e, h_e = kda.fwd(**x.to("cuda").tensors(), check=True)
        torch.cuda.synchronize()
        assert torch.equal(o, o_e) and torch.equal(hT, h_e)


def test_backward_graph_replay(kda):
    x1 = gen.make_lengths([150, 0, 90], seed=62, salt=SALT, H=2, d=128)
    x2 = gen.make_lengths([150, 0, 90], seed=63, salt=SALT + 1, H=2, d=128)
    rng = np.random.default_rng(0)
    do = torch.from_numpy(rng.standard_normal(tuple(x1.v.shape)).astype(np.float32)).to(x1.v.dtype).cuda()
    dhT = torch.from_numpy(rng.standard_normal((x1.num_seqs, x1.H, 128, 128)).astype(np.float32)).cuda()
    d1 = x1.to("cuda")
    ws = torch.empty(int(kda.load_library().kda_bwd_workspace_size(x1.B, x1.T, x1.H, 128, 128, x1.num_seqs))
                     + 256, dtype=torch.uint8, device="cuda")
    out = {}
    graph = _capture(lambda: out.__setitem__("g", kda.bwd(**d1.tensors(), do=do, dhT=dhT, workspace=ws)))
    for x in (x1, x2):
        for name in ("q", "k", "v", "g", "beta", "h0"):
            getattr(d1, name).copy_(getattr(x, name).to("cuda"))
        graph.replay()
        torch.cuda.synchronize()
        eager = kda.bwd(**x.to("cuda").tensors(), do=do, dhT=dhT, check=True)
        torch.cuda.synchronize()
        # dv and dh0 are written once per element (bit-equal); dq, dk, dg and dbeta
        # add the value tiles' shares in any order (equal to rounding)
        for i, (a, b) in enumerate(zip(out["g"], eager)):
            if i in (2, 5):
                assert torch.equal(a, b)
            else:
                assert torch.allclose(a, b, rtol=1e-5, atol=1e-6 * float(b.abs().max()))
