"""Input recipes: seeded reproducibility, salts, and the layouts they promise."""
import numpy as np
import torch

from tests import gen


def test_seeded_reproducible_and_salted():
    a = gen.make_cfg3(seed=5, salt=9, H=2)
    b = gen.make_cfg3(seed=5, salt=9, H=2)
    c = gen.make_cfg3(seed=5, salt=10, H=2)
    assert torch.equal(a.q, b.q) and torch.equal(a.cu_seqlens, b.cu_seqlens)
    assert not torch.equal(a.q, c.q)


def test_cfg3_layout():
    for salt in range(5):
        x = gen.make_cfg3(seed=0, salt=salt, H=1, d=16)
        lens = x.seq_lens()
        assert len(lens) == 8 and sum(lens) == 8192 and 1 in lens
        assert max(lens) <= 4000 and any(L % 64 for L in lens)
        assert x.q.dtype == torch.bfloat16 and x.h0.shape == (8, 1, 16, 16)


def test_cfg4_layout_and_probes():
    x = gen.make_cfg4(seed=0, salt=3, H=2, d=16)
    lens = x.seq_lens()
    assert len(lens) == 32 and sum(lens) == 8192 and 4750 <= max(lens) <= 5250
    g = x.g[0, 0].numpy()
    assert np.all((np.isclose(g, -1e-6)) | (np.isclose(g, np.log(1e-6))))
    assert (np.isclose(g, -1e-6).sum(-1) == 8).all()
    b = x.beta.numpy()
    assert (b == 0).mean() > 0.05 and (b == 1).mean() > 0.05
    n = x.q.float().norm(dim=-1).numpy()
    assert n.min() < 1e-2 and n.max() > 1e2


def test_cfg2_gate_range():
    x = gen.make_cfg2(seed=0, T=256, H=2, d=32)
    a = np.exp(x.g.numpy())
    assert a.min() >= 1e-4 * (1 - 1e-6) and a.max() < 1.0
    assert x.q.dtype == torch.bfloat16 and x.g.dtype == torch.float32


def test_cfg5_filled_heads_are_distinct_rolls_of_drawn_ones():
    x = gen.make_cfg5(5, 8192, False, seed=1, salt=2, drawn_heads=2)
    y = gen.make_cfg5(2, 8192, False, seed=1, salt=2)  # the same draws, two heads
    assert torch.equal(x.q[:, :, :2], y.q) and torch.equal(x.g[:, :, :2], y.g)
    for h in range(2, 5):
        shift = 37 * (h // 2)
        assert torch.equal(x.q[:, :, h], torch.roll(x.q[:, :, h % 2], shift, dims=1))
        assert torch.equal(x.beta[:, :, h], torch.roll(x.beta[:, :, h % 2], shift, dims=1))
        assert torch.equal(x.h0[:, h], torch.roll(x.h0[:, h % 2], shift, dims=1))
    for a in range(5):
        for b in range(a):
            assert not torch.equal(x.k[:, :, a], x.k[:, :, b])
    z = gen.make_cfg5(3, 8192, True, seed=1, salt=2, drawn_heads=2)
    assert z.cu_seqlens is not None and z.q.shape == (1, 8192, 3, 128)
