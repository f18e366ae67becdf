"""The fp64 oracle against what the mathematics fixes (CPU only)."""
from __future__ import annotations

import functools
import math
import os

import numpy as np
import pytest

import oracle
from oracle import brute
from oracle.chunked import kda_chunked_fp64, kda_segmented_fp64
from tests import gen
from tests.metrics import rel_rmse
from tests.oracle_pins import PINS, brute_case, expected_reciprocal_norm

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _fwd(mutant=0):
    def f(q, k, v, g, beta, h0, cu, scale, eps):
        return oracle.kda_recurrence_fp64(q, k, v, g, beta, h0, cu, scale, eps=eps,
                                          _mutant=mutant)
    return f


@pytest.mark.parametrize("name", sorted(PINS))
def test_oracle_pin(name):
    fn, tol = PINS[name]
    err = fn(_fwd(0))
    assert err <= tol, f"pin {name}: {err:.3e} > {tol:.1e}"


@pytest.mark.parametrize("seed", range(4))
def test_brute_forms_agree_exactly(seed):
    case = brute_case(100 + seed, T=4, d=3 + seed % 2)
    o1, S1 = brute.brute_recurrence(*case)
    o2, S2 = brute.brute_unrolled(*case)
    assert o1 == o2 and S1 == S2


def test_golden_brute_fixture():
    """The stored exact case (written by tests/golden/make_golden.py from oracle.brute)."""
    import json
    from fractions import Fraction
    with open(os.path.join(GOLDEN, "brute_tiny.json")) as f:
        fx = json.load(f)
    case = brute_case(fx["seed"], T=fx["T"], d=fx["d"])
    o, S = brute.brute_recurrence(*case)
    assert [[str(x) for x in r] for r in o] == fx["o"]
    assert [[str(x) for x in r] for r in S] == fx["S"]
    from tests.oracle_pins import _case_arrays
    qa, ka, va, ga, ba, h0, scale = _case_arrays(case)
    oo, hh = oracle.kda_recurrence_fp64(qa, ka, va, ga, ba, h0, None, scale, eps=0.0)
    ref_o = np.array([[float(Fraction(x)) for x in r] for r in fx["o"]])
    assert rel_rmse(oo[0, :, 0], ref_o) < 1e-13


def test_hack_constant_is_expected_reciprocal_norm():
    """The constant the kernel-design-agents page quotes (section 03 REWARD HACKING)
    is E[1/|x|] for x ~ N(0, 0.5^2) at d = 128 (tests/golden/hack_constant.txt)."""
    with open(os.path.join(GOLDEN, "hack_constant.txt")) as f:
        vals = dict(line.split("=", 1) for line in f if "=" in line and not line.startswith("#"))
    c = float(vals["constant"])
    assert abs(expected_reciprocal_norm(int(vals["d"]), float(vals["sigma"])) - c) < 5e-11


@pytest.mark.parametrize("chunk", [1, 2, 7, 16, 64])
def test_chunked_equals_recurrence(chunk):
    x = gen.make_lengths([70, 1, 0, 129, 64], seed=3, H=2, d=16)
    o, h = oracle.kda_recurrence_fp64(**x.tensors())
    oc, hc = kda_chunked_fp64(**x.tensors(), chunk=chunk)
    assert rel_rmse(oc, o) < 1e-11 and rel_rmse(hc, h) < 1e-11


@pytest.mark.parametrize("kind", ["deep", "abyss", "saturated", "repeated_keys", "zero_rows"])
def test_chunked_equals_recurrence_probes(kind):
    x = gen.make_probe(kind, seed=1, T=150, H=2, d=16)
    o, h = oracle.kda_recurrence_fp64(**x.tensors())
    oc, hc = kda_chunked_fp64(**x.tensors(), chunk=64)
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(h))
    assert rel_rmse(oc, o) < 1e-10 and rel_rmse(hc, h) < 1e-10


@pytest.mark.parametrize("seg_chunks,chunk", [(1, 4), (2, 4), (3, 8), (5, 4), (4, 64)])
def test_segmented_equals_recurrence(seg_chunks, chunk):
    """The exact inter-chunk split (segment maps, a scan of start states, the later
    segments rerun) equals the token recurrence: chains of 0 to 10 segments, ragged
    last chunks and segments, an empty sequence."""
    x = gen.make_lengths([70, 1, 0, 129, 64, 300], seed=5, H=2, d=8)
    o, h = oracle.kda_recurrence_fp64(**x.tensors())
    os_, hs = kda_segmented_fp64(**x.tensors(), seg_chunks=seg_chunks, chunk=chunk)
    assert rel_rmse(os_, o) < 1e-11 and rel_rmse(hs, h) < 1e-11


@pytest.mark.parametrize("kind", ["deep", "abyss", "saturated", "repeated_keys", "beta01"])
def test_segmented_equals_recurrence_probes(kind):
    x = gen.make_probe(kind, seed=2, T=200, H=2, d=8)
    o, h = oracle.kda_recurrence_fp64(**x.tensors())
    os_, hs = kda_segmented_fp64(**x.tensors(), seg_chunks=2, chunk=16)
    assert np.all(np.isfinite(os_)) and np.all(np.isfinite(hs))
    assert rel_rmse(os_, o) < 1e-10 and rel_rmse(hs, h) < 1e-10


def test_zero_length_sequence_returns_h0():
    x = gen.make_lengths([5, 0, 3], seed=0, H=2, d=8)
    _, h = oracle.kda_recurrence_fp64(**x.tensors())
    assert np.array_equal(h[1], x.h0[1].double().numpy())


def test_zero_rows_normalise_to_zero():
    x = gen.make_probe("zero_rows", seed=2, T=40, H=2, d=16)
    o, h = oracle.kda_recurrence_fp64(**x.tensors())
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(h))
    zq = (x.q.float().abs().sum(-1) == 0).numpy()
    assert zq.any() and np.all(o[zq] == 0.0)


def test_rejects_bad_arguments():
    x = gen.make_lengths([3, 4], seed=0, H=1, d=4)
    t = x.tensors()
    t["cu_seqlens"] = np.array([0, 5, 4], dtype=np.int64)
    with pytest.raises(ValueError):
        oracle.kda_recurrence_fp64(**t)


@pytest.mark.parametrize("mutant", range(1, 11))
def test_planted_mistake_fails_a_pin(mutant):
    """Each planted mistake in the oracle's C source is caught by at least one pin."""
    f = _fwd(mutant)
    failed = []
    for name, (fn, tol) in PINS.items():
        try:
            err = fn(f)
        except Exception:
            err = float("inf")
        if not (err <= tol):
            failed.append(name)
    assert failed, f"mutant {mutant} passed every pin"


def test_threads_do_not_change_results():
    x = gen.make_cfg3(seed=1, total=1024, n=5, H=3, d=16, max_len=800)
    o1, h1 = oracle.kda_recurrence_fp64(**x.tensors(), nthreads=1)
    o2, h2 = oracle.kda_recurrence_fp64(**x.tensors(), nthreads=4)
    assert np.array_equal(o1, o2) and np.array_equal(h1, h2)
