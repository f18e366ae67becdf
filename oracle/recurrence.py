"""TEST INFRASTRUCTURE ONLY: build, load and call the fp64 C oracle.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this module.  The CUDA library never calls it.

The oracle is the token-by-token fp64 recurrence of the Kimi Delta Attention
forward ("NVIDIA Kernel Design Agents optimize Kimi Delta Attention", section 01
RESULTS: every kernel is checked against a token-by-token fp64 recurrence).  The
arithmetic lives in ``kda_oracle.c``; this file only marshals arrays.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kda_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB = os.path.join(_OUT_DIR, "libkda_oracle.so")
_lock = threading.Lock()
_handles = {}

# L2-norm epsilon: x / sqrt(sum(x^2) + eps).  The pages name the normalisation but
# not its epsilon; 1e-6 is the reading taken (stated with the other readings in
# the design notes).  The CUDA library fixes the same number independently.
L2_EPS = 1e-6


def _lib_path(mutant: int) -> str:
    return _LIB if mutant == 0 else os.path.join(_OUT_DIR, f"libkda_oracle_mut{mutant}.so")


def build(force: bool = False, mutant: int = 0) -> str:
    """Compile kda_oracle.c into a shared library (gcc, OpenMP, no fast-math).

    ``mutant`` > 0 builds a copy with one planted mistake (tests only)."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    lib = _lib_path(mutant)
    if (not force and os.path.exists(lib)
            and os.path.getmtime(lib) >= os.path.getmtime(_SRC)):
        return lib
    tmp = lib + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
           "-std=c11", f"-DKDA_ORACLE_MUTANT={int(mutant)}", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, lib)
    return lib


def _lib(mutant: int = 0):
    with _lock:
        if mutant not in _handles:
            path = build(mutant=mutant)
            lib = ctypes.CDLL(path)
            dp = ctypes.POINTER(ctypes.c_double)
            lib.kda_oracle_fwd.argtypes = [
                dp, dp, dp, dp, dp, dp, ctypes.POINTER(ctypes.c_int64), ctypes.c_int64,
                ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                ctypes.c_double, ctypes.c_double, dp, dp, ctypes.c_int]
            lib.kda_oracle_fwd.restype = ctypes.c_int
            lib.kda_oracle_max_threads.restype = ctypes.c_int
            _handles[mutant] = lib
    return _handles[mutant]


def max_threads() -> int:
    return int(_lib().kda_oracle_max_threads())


def _f64(x) -> np.ndarray:
    """Exact conversion of the stored values (bf16 / fp32 / fp64) to fp64."""
    if x is None:
        return None
    if hasattr(x, "detach"):  # torch tensor: widen on the CPU, exactly
        x = x.detach().to("cpu").double().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def kda_recurrence_fp64(q, k, v, g, beta, h0=None, cu_seqlens=None, scale=None,
                        eps: float = L2_EPS, nthreads: int = 0, _mutant: int = 0):
    """Run the fp64 oracle.

    Shapes: q, k, g ``[B, T, H, dk]``; v ``[B, T, H, dv]``; beta ``[B, T, H]``;
    h0 ``[N, H, dk, dv]`` or None; cu_seqlens ``[N+1]`` (varlen, B == 1) or None.
    Returns ``(o [B,T,H,dv], hT [N,H,dk,dv])`` as fp64 numpy arrays.
    """
    q, k, v, g, beta = (_f64(x) for x in (q, k, v, g, beta))
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    if k.shape != q.shape or g.shape != q.shape or v.shape[:3] != q.shape[:3] \
            or beta.shape != q.shape[:3]:
        raise ValueError("inconsistent input shapes")
    if cu_seqlens is not None:
        cu = np.ascontiguousarray(np.asarray(
            cu_seqlens.cpu() if hasattr(cu_seqlens, "cpu") else cu_seqlens, dtype=np.int64))
        N = cu.shape[0] - 1
        cu_ptr = cu.ctypes.data_as(ctypes.POINTER(ctypes.c_int64))
    else:
        cu, N, cu_ptr = None, B, None
    h0a = _f64(h0)
    if h0a is not None and h0a.shape != (N, H, dk, dv):
        raise ValueError(f"h0 shape {h0a.shape} != {(N, H, dk, dv)}")
    if scale is None:
        scale = dk ** -0.5
    o = np.zeros((B, T, H, dv), dtype=np.float64)
    hT = np.zeros((N, H, dk, dv), dtype=np.float64)
    rc = _lib(_mutant).kda_oracle_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(h0a),
                               cu_ptr, N, B, T, H, dk, dv, float(scale), float(eps),
                               _ptr(o), _ptr(hT), int(nthreads))
    if rc != 0:
        raise ValueError(f"kda_oracle_fwd rejected its arguments (rc={rc})")
    return o, hT
