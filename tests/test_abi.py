"""The C-ABI library: it loads, exports every declared entry point, and rejects bad
arguments on the host before touching the GPU (CPU only: no CUDA call is made on
these paths)."""
from __future__ import annotations

import ctypes
import os
import re

import pytest

import __graft_entry__  # noqa: F401  (puts the repo root on sys.path)
from gated_delta_rule_25_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    _build.build()
    import gated_delta_rule_25_gb300 as kda
    return kda.load_library()


def _declared():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            src = open(os.path.join(ROOT, "include", fn)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names |= set(re.findall(r"\b(kda_\w+)\s*\(", src))
    return names


def test_exports_every_declared_symbol(lib):
    names = _declared()
    assert {"kda_fwd", "kda_fwd_workspace_size", "kda_fwd_check", "kda_status_string"} <= names
    for n in names:
        assert hasattr(lib, n), f"{n} declared in include/ but not exported"


def test_workspace_size(lib):
    ws = lib.kda_fwd_workspace_size
    a = ws(1, 8192, 32, 128, 128, 1)
    b = ws(1, 8192, 32, 128, 128, 8)
    assert 0 < a < b
    assert ws(1, 8192, 32, 96, 128, 1) == 0          # unsupported dk
    assert ws(2, 100, 4, 64, 64, 3) == 0             # fixed length needs N == B
    assert ws(4, 8192, 16, 128, 128, 4) > 0


def _call(lib, **kw):
    p = ctypes.c_void_p(1 << 20)  # never dereferenced: every case fails host checks
    args = dict(q=p, k=p, v=p, dt=0, g=p, beta=p, h0=None, cu=None, N=1, B=1, T=64, H=2,
                dk=64, dv=64, scale=0.125, o=p, hT=None, ws=ctypes.c_void_p(1 << 20),
                wsb=1 << 40, stream=None)
    args.update(kw)
    return lib.kda_fwd(args["q"], args["k"], args["v"], args["dt"], args["g"], args["beta"],
                       args["h0"], args["cu"], args["N"], args["B"], args["T"], args["H"],
                       args["dk"], args["dv"], args["scale"], args["o"], args["hT"], args["ws"],
                       args["wsb"], args["stream"])


def test_host_validation(lib):
    assert _call(lib, dk=96) == 2                     # unsupported head dim
    assert _call(lib, dv=32) == 2
    assert _call(lib, dt=7) == 2                      # unknown dtype
    assert _call(lib, scale=float("nan")) == 1
    assert _call(lib, B=2, N=1) == 1                  # fixed length needs N == B
    assert _call(lib, cu=ctypes.c_void_p(1 << 20), B=2, N=2) == 1  # varlen needs B == 1
    assert _call(lib, q=None) == 1
    assert _call(lib, g=ctypes.c_void_p((1 << 20) + 4)) == 3       # misaligned
    assert _call(lib, wsb=16) == 4                    # workspace too small
    assert _call(lib, ws=ctypes.c_void_p((1 << 20) + 128)) == 4    # workspace misaligned
    assert _call(lib, ws=None) == 4
    assert _call(lib, N=0, B=0, T=0) == 0             # nothing to do: no launch


def test_status_strings(lib):
    for s in range(7):
        assert lib.kda_status_string(s)
    assert lib.kda_status_string(99) == b"unknown status"


def test_python_binding_fails_loudly_without_cuda():
    import torch

    import gated_delta_rule_25_gb300 as kda
    x = torch.zeros(1, 4, 1, 64)
    with pytest.raises(ValueError):
        kda.fwd(x, x, x, x.float(), torch.zeros(1, 4, 1))


def _decode(lib, **kw):
    p = ctypes.c_void_p(1 << 20)  # never dereferenced: every case fails host checks
    args = dict(q=p, k=p, v=p, dt=0, g=p, beta=p, h_in=p, h_out=ctypes.c_void_p(1 << 30), N=2,
                H=2, dk=64, dv=64, scale=0.125, o=p, stream=None)
    args.update(kw)
    return lib.kda_decode(args["q"], args["k"], args["v"], args["dt"], args["g"], args["beta"],
                          args["h_in"], args["h_out"], args["N"], args["H"], args["dk"],
                          args["dv"], args["scale"], args["o"], args["stream"])


def test_decode_host_validation(lib):
    assert _decode(lib, dk=96) == 2
    assert _decode(lib, dv=256) == 2
    assert _decode(lib, dt=3) == 2
    assert _decode(lib, scale=float("inf")) == 1
    assert _decode(lib, H=0) == 1
    assert _decode(lib, N=-1) == 1
    assert _decode(lib, q=None) == 1
    assert _decode(lib, h_out=None) == 1
    assert _decode(lib, o=ctypes.c_void_p((1 << 20) + 2)) == 3      # misaligned
    # overlapping (but not identical) state buffers
    assert _decode(lib, h_in=ctypes.c_void_p(1 << 30), h_out=ctypes.c_void_p((1 << 30) + 256)) == 1
    assert _decode(lib, N=0) == 0                                   # nothing to do: no launch


def test_python_decode_fails_loudly_without_cuda():
    import torch

    import gated_delta_rule_25_gb300 as kda
    x = torch.zeros(2, 1, 64)
    with pytest.raises(ValueError):
        kda.decode(x, x, x, x.float(), torch.zeros(2, 1))


def test_fwd_ex_gate_dtypes(lib):
    p = ctypes.c_void_p(1 << 20)  # never dereferenced: every case fails host checks

    def call(dt, gdt, **kw):
        a = dict(ws=ctypes.c_void_p(1 << 20), wsb=1 << 40)
        a.update(kw)
        return lib.kda_fwd_ex(p, p, p, dt, p, gdt, p, None, None, 1, 1, 64, 2, 64, 64, 0.125, p,
                              None, a["ws"], a["wsb"], None)
    assert call(1, 0) == 2      # bf16 gate with fp32 q/k/v
    assert call(0, 5) == 2      # unknown gate dtype
    assert call(0, 0, wsb=16) == 4   # valid dtypes reach the workspace check
    assert call(0, 1, wsb=16) == 4


def _bwd(lib, **kw):
    p = ctypes.c_void_p(1 << 20)  # never dereferenced: every case fails host checks
    args = dict(q=p, k=p, v=p, dt=0, g=p, beta=p, h0=None, cu=None, N=1, B=1, T=64, H=2, dk=64,
                dv=64, scale=0.125, do=p, dhT=None, dq=p, dk_=p, dv_=p, dg=p, db=p, dh0=None,
                ws=ctypes.c_void_p(1 << 20), wsb=1 << 40, stream=None)
    args.update(kw)
    a = args
    return lib.kda_bwd(a["q"], a["k"], a["v"], a["dt"], a["g"], a["beta"], a["h0"], a["cu"], a["N"],
                       a["B"], a["T"], a["H"], a["dk"], a["dv"], a["scale"], a["do"], a["dhT"], a["dq"],
                       a["dk_"], a["dv_"], a["dg"], a["db"], a["dh0"], a["ws"], a["wsb"], a["stream"])


def test_bwd_host_validation(lib):
    assert lib.kda_bwd_workspace_size(1, 8192, 32, 128, 128, 1) > 0
    assert lib.kda_bwd_workspace_size(1, 8192, 32, 96, 128, 1) == 0
    assert _bwd(lib, dk=96) == 2                      # unsupported head dim
    assert _bwd(lib, dt=7) == 2                       # unknown dtype
    assert _bwd(lib, scale=float("nan")) == 1
    assert _bwd(lib, B=2, N=1) == 1                   # fixed length needs N == B
    assert _bwd(lib, do=None) == 1                    # an input gradient is missing
    assert _bwd(lib, dq=None) == 1                    # an output is missing
    assert _bwd(lib, dg=ctypes.c_void_p((1 << 20) + 4)) == 3       # misaligned
    assert _bwd(lib, wsb=16) == 4                     # workspace too small
    assert _bwd(lib, ws=ctypes.c_void_p((1 << 20) + 128)) == 4     # workspace misaligned
    assert _bwd(lib, N=0, B=0, T=0) == 0              # nothing to do: no launch


def test_python_bwd_fails_loudly_without_cuda():
    import torch

    import gated_delta_rule_25_gb300 as kda
    x = torch.zeros(1, 4, 1, 64)
    with pytest.raises(ValueError):
        kda.bwd(x, x, x, x.float(), torch.zeros(1, 4, 1), do=x)
