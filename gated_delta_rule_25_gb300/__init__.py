"""Kimi Delta Attention prefill forward (and its backward) for GB300 (sm_103a).

A thin binding over the C ABI in ``include/kda.h`` (``_lib/libkda.so``).  This
module only checks and marshals arguments; every step of the computation runs in
the library's CUDA kernels.  PyTorch provides device memory and the current
stream.  There is no CPU path: without the built library every call raises.

    o, hT = fwd(q, k, v, g, beta, h0=None, cu_seqlens=None, scale=None)
    dq, dk, dv, dg, dbeta, dh0 = bwd(q, k, v, g, beta, h0, cu_seqlens, scale, do=do, dhT=dhT)
    o, h  = decode(q, k, v, g, beta, state=None, scale=None)   # one token per sequence
    set_pipeline("auto" | "fused" | "split" | "split-whole")  # the forward's kernels

q, k: [B, T, H, dk]; v: [B, T, H, dv] (bf16 or fp32, same dtype); g: [B, T, H, dk]
fp32, or bf16 with bf16 q/k/v (log of the per-channel decay, <= 0); beta: [B, T, H] fp32 in [0, 1];
h0: [N, H, dk, dv] fp32 or None; cu_seqlens: int32 [N + 1] (packed varlen, B == 1)
or None.  Returns o [B, T, H, dv] in q's dtype and hT [N, H, dk, dv] fp32.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional, Tuple

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_lib", "libkda.so")

KDA_OK, KDA_ERR_DEVICE = 0, 6
KDA_BF16, KDA_FP32 = 0, 1
_STATUS = {0: "ok", 1: "invalid argument", 2: "unsupported size or dtype",
           3: "tensor pointer not 16-byte aligned", 4: "workspace missing, too small or misaligned",
           5: "CUDA runtime error", 6: "device reported malformed input",
           7: "problem too large for the built-in no-allocation scratch"}
KDA_ERR_TOO_LARGE = 7

_lock = threading.Lock()
_lib = None


class KdaError(RuntimeError):
    def __init__(self, status: int, what: str = "kda_fwd"):
        self.status = status
        super().__init__(f"{what}: {_STATUS.get(status, 'unknown')} (status {status})")


def load_library():
    """Load libkda.so; raises if it has not been built (no fallback exists)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: build it first "
                "(python -c 'import __graft_entry__ as g; g.build()')")
        lib = ctypes.CDLL(LIB_PATH)
        vp, i32, f32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
        lib.kda_fwd_workspace_size.argtypes = [i32] * 6
        lib.kda_fwd_workspace_size.restype = sz
        lib.kda_fwd_launch_count.argtypes = [i32] * 6
        lib.kda_fwd_launch_count.restype = i32
        lib.kda_fwd.argtypes = [vp, vp, vp, i32, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32,
                                f32, vp, vp, vp, sz, vp]
        lib.kda_fwd.restype = i32
        lib.kda_fwd_ex.argtypes = [vp, vp, vp, i32, vp, i32, vp, vp, vp, i32, i32, i32, i32, i32,
                                   i32, f32, vp, vp, vp, sz, vp]
        lib.kda_fwd_ex.restype = i32
        lib.kda_fwd_profiled.argtypes = lib.kda_fwd_ex.argtypes + [ctypes.POINTER(vp)]
        lib.kda_fwd_profiled.restype = i32
        lib.kda_fwd_noalloc.argtypes = [vp, vp, vp, i32, vp, vp, vp, vp, i32, i32, i32, i32,
                                        i32, i32, f32, vp, vp, vp]
        lib.kda_fwd_noalloc.restype = i32
        lib.kda_fwd_check.argtypes = [vp, vp, ctypes.POINTER(ctypes.c_uint32)]
        lib.kda_fwd_check.restype = i32
        lib.kda_fwd_noalloc_check.argtypes = [vp, ctypes.POINTER(ctypes.c_uint32)]
        lib.kda_fwd_noalloc_check.restype = i32
        lib.kda_decode.argtypes = [vp, vp, vp, i32, vp, vp, vp, vp, i32, i32, i32, i32, f32, vp, vp]
        lib.kda_decode.restype = i32
        lib.kda_status_string.argtypes = [i32]
        lib.kda_status_string.restype = ctypes.c_char_p
        lib.kda_set_pipeline.argtypes = [i32]
        lib.kda_set_pipeline.restype = None
        lib.kda_get_pipeline.argtypes = []
        lib.kda_get_pipeline.restype = i32
        lib.kda_fwd_uses_fused.argtypes = [i32] * 6
        lib.kda_fwd_uses_fused.restype = i32
        lib.kda_bwd_workspace_size.argtypes = [i32] * 6
        lib.kda_bwd_workspace_size.restype = sz
        lib.kda_bwd.argtypes = [vp, vp, vp, i32, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, f32,
                                vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
        lib.kda_bwd.restype = i32
        _lib = lib
        return lib


def workspace_size(B: int, T: int, H: int, dk: int, dv: int, num_seqs: int) -> int:
    return int(load_library().kda_fwd_workspace_size(B, T, H, dk, dv, num_seqs))


def launch_count(B: int, T: int, H: int, dk: int, dv: int, num_seqs: int) -> int:
    return int(load_library().kda_fwd_launch_count(B, T, H, dk, dv, num_seqs))


PIPELINES = {"auto": 0, "fused": 1, "split": 2, "split-whole": 3}


def set_pipeline(name: str) -> None:
    """Selects the forward's pipeline, process-wide: "auto" (default: the fused one
    where it applies and was measured faster, else split), "fused" (one cooperative
    kernel producing factors and running the state chains at once, wherever the
    sizes allow), "split" (a factor kernel, then the state kernels; few long chains
    cut into segments where predicted faster) or "split-whole" (split, chains never
    cut)."""
    if name not in PIPELINES:
        raise ValueError(f"pipeline must be one of {sorted(PIPELINES)}, got {name!r}")
    load_library().kda_set_pipeline(PIPELINES[name])


def get_pipeline() -> str:
    v = int(load_library().kda_get_pipeline())
    return next(k for k, x in PIPELINES.items() if x == v)


def uses_fused(B: int, T: int, H: int, dk: int, dv: int, num_seqs: int) -> bool:
    """True if fwd takes the fused pipeline for these sizes (current setting, device)."""
    return bool(load_library().kda_fwd_uses_fused(B, T, H, dk, dv, num_seqs))


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _check(t, name, dtype, shape, device):
    if t.dtype != dtype:
        raise TypeError(f"{name}: dtype {t.dtype}, expected {dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: shape {tuple(t.shape)}, expected {tuple(shape)}")
    if t.device != device:
        raise ValueError(f"{name}: on {t.device}, expected {device}")
    if not t.is_contiguous():
        raise ValueError(f"{name}: must be contiguous")


def _validate(q, k, v, g, beta, h0, cu_seqlens, o, hT, gate_bf16_ok: bool):
    """Every dtype and shape check of the forward, before anything is launched.

    Returns (B, T, H, dk, dv, N, device).  Dtypes and shapes are checked before the
    device, so a wrong argument raises the same error with or without a GPU."""
    if q.dim() != 4:
        raise ValueError("q must be [B, T, H, dk]")
    if v.dim() != 4:
        raise ValueError("v must be [B, T, H, dv]")
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    dev = q.device
    if q.dtype not in (torch.bfloat16, torch.float32):
        raise TypeError("q, k, v must be bfloat16 or float32")
    _check(q, "q", q.dtype, (B, T, H, dk), dev)
    _check(k, "k", q.dtype, (B, T, H, dk), dev)
    _check(v, "v", q.dtype, (B, T, H, dv), dev)
    if g.dtype == torch.bfloat16:
        if not gate_bf16_ok:
            raise TypeError("g: this entry point takes an fp32 gate")
        if q.dtype != torch.bfloat16:
            raise TypeError("a bf16 gate needs bf16 q, k, v")
    _check(g, "g", g.dtype if g.dtype == torch.bfloat16 else torch.float32, (B, T, H, dk), dev)
    _check(beta, "beta", torch.float32, (B, T, H), dev)
    if cu_seqlens is not None:
        if B != 1:
            raise ValueError("varlen (cu_seqlens) needs B == 1")
        if cu_seqlens.dim() != 1 or cu_seqlens.numel() < 1:
            raise ValueError("cu_seqlens must be a 1-D tensor of num_seqs + 1 offsets")
        _check(cu_seqlens, "cu_seqlens", torch.int32, (cu_seqlens.numel(),), dev)
        N = cu_seqlens.numel() - 1
    else:
        N = B
    if h0 is not None:
        _check(h0, "h0", torch.float32, (N, H, dk, dv), dev)
    if o is not None:
        _check(o, "o", q.dtype, (B, T, H, dv), dev)
    if hT is not None:
        _check(hT, "hT", torch.float32, (N, H, dk, dv), dev)
    if dev.type != "cuda":
        raise ValueError("inputs must be CUDA tensors")
    return B, T, H, dk, dv, N, dev


def fwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, g: torch.Tensor,
        beta: torch.Tensor, h0: Optional[torch.Tensor] = None,
        cu_seqlens: Optional[torch.Tensor] = None, scale: Optional[float] = None, *,
        output_final_state: bool = True, o: Optional[torch.Tensor] = None,
        hT: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
        check: bool = False, events=None) -> Tuple[torch.Tensor, Optional[torch.Tensor]]:
    """KDA prefill forward on the current CUDA stream.  See the module docstring.

    ``o``, ``hT``, ``workspace``: optional preallocated buffers (needed for CUDA-graph
    capture with stable addresses).  ``check``: synchronise and raise on a device-side
    error.  ``events``: launch_count + 1 recorded torch.cuda.Event objects; each kernel
    launch is bracketed by two of them (per-kernel timing)."""
    B, T, H, dk, dv, N, dev = _validate(q, k, v, g, beta, h0, cu_seqlens, o,
                                        hT if output_final_state else None, True)
    lib = load_library()
    if scale is None:
        scale = dk ** -0.5
    if o is None:
        o = torch.empty((B, T, H, dv), dtype=q.dtype, device=dev)
    if output_final_state:
        if hT is None:
            hT = torch.empty((N, H, dk, dv), dtype=torch.float32, device=dev)
    else:
        hT = None
    ws_bytes = int(lib.kda_fwd_workspace_size(B, T, H, dk, dv, N))
    if ws_bytes == 0:
        raise KdaError(2, "kda_fwd_workspace_size")
    if workspace is None or workspace.numel() - (-workspace.data_ptr()) % 256 < ws_bytes:
        workspace = torch.empty(ws_bytes + 256, dtype=torch.uint8, device=dev)
    ws_ptr = (workspace.data_ptr() + 255) & ~255  # the library wants 256-byte alignment
    avail = workspace.numel() - (ws_ptr - workspace.data_ptr())
    stream = torch.cuda.current_stream(dev).cuda_stream
    dt = KDA_BF16 if q.dtype == torch.bfloat16 else KDA_FP32
    gdt = KDA_BF16 if g.dtype == torch.bfloat16 else KDA_FP32
    args = (_ptr(q), _ptr(k), _ptr(v), dt, _ptr(g), gdt, _ptr(beta), _ptr(h0), _ptr(cu_seqlens),
            N, B, T, H, dk, dv, float(scale), _ptr(o), _ptr(hT), ctypes.c_void_p(ws_ptr), avail,
            ctypes.c_void_p(stream))
    if events is None:
        st = lib.kda_fwd_ex(*args)
    else:
        # one torch.cuda.Event per launch boundary (kda_fwd_launch_count + 1), already
        # recorded once so that its CUDA event exists
        arr = (ctypes.c_void_p * len(events))(*[e.cuda_event for e in events])
        st = lib.kda_fwd_profiled(*args, arr)
    if st != KDA_OK:
        raise KdaError(st)
    if check:
        err = ctypes.c_uint32(0)
        st = lib.kda_fwd_check(ctypes.c_void_p(ws_ptr), ctypes.c_void_p(stream), ctypes.byref(err))
        if st != KDA_OK:
            raise KdaError(st, f"kda_fwd_check (device error bits {err.value:#x})")
    return o, hT


def fwd_noalloc(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, g: torch.Tensor,
                beta: torch.Tensor, h0: Optional[torch.Tensor] = None,
                cu_seqlens: Optional[torch.Tensor] = None, scale: Optional[float] = None, *,
                o: Optional[torch.Tensor] = None, hT: Optional[torch.Tensor] = None,
                check: bool = False) -> Tuple[torch.Tensor, torch.Tensor]:
    """The forward through ``kda_fwd_noalloc``: no workspace is passed, the library
    uses the device scratch array built into it (KDA_NOALLOC_SCRATCH_BYTES, 32 MiB).

    For callers that cannot allocate device memory where they run the forward
    (a plugin inside an engine that owns all device memory, a path where an
    allocation's latency or failure is not acceptable): pass preallocated ``o``
    and ``hT``; the call then allocates nothing.  The arguments get the same dtype
    and shape checks as ``fwd``, except that the gate must be fp32.  Problems too
    large for the array raise KdaError with status KDA_ERR_TOO_LARGE.  Calls share
    the array, so their work must not overlap on the GPU (order them on one
    stream).  ``check``: synchronise and raise if the device reported an error
    (``kda_fwd_noalloc_check``)."""
    B, T, H, dk, dv, N, dev = _validate(q, k, v, g, beta, h0, cu_seqlens, o, hT, False)
    lib = load_library()
    if o is None:
        o = torch.empty((B, T, H, dv), dtype=q.dtype, device=dev)
    if hT is None:
        hT = torch.empty((N, H, dk, dv), dtype=torch.float32, device=dev)
    if scale is None:
        scale = dk ** -0.5
    dt = KDA_BF16 if q.dtype == torch.bfloat16 else KDA_FP32
    stream = torch.cuda.current_stream(dev).cuda_stream
    st = lib.kda_fwd_noalloc(_ptr(q), _ptr(k), _ptr(v), dt, _ptr(g), _ptr(beta), _ptr(h0),
                             _ptr(cu_seqlens), N, B, T, H, dk, dv, float(scale), _ptr(o),
                             _ptr(hT), ctypes.c_void_p(stream))
    if st != KDA_OK:
        raise KdaError(st, "kda_fwd_noalloc")
    if check:
        err = ctypes.c_uint32(0)
        st = lib.kda_fwd_noalloc_check(ctypes.c_void_p(stream), ctypes.byref(err))
        if st != KDA_OK:
            raise KdaError(st, f"kda_fwd_noalloc_check (device error bits {err.value:#x})")
    return o, hT


def bwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, g: torch.Tensor,
        beta: torch.Tensor, h0: Optional[torch.Tensor] = None,
        cu_seqlens: Optional[torch.Tensor] = None, scale: Optional[float] = None, *,
        do: torch.Tensor, dhT: Optional[torch.Tensor] = None, want_dh0: bool = True,
        workspace: Optional[torch.Tensor] = None, check: bool = False):
    """Backward pass through ``kda_bwd``: the gradients of sum(o * do) + sum(h_T * dhT)
    of the forward on the same inputs, with respect to q, k, v, g, beta and h0.

    Returns (dq, dk, dv, dg, dbeta, dh0), fp32 tensors shaped like the inputs (dh0
    [N, H, dk, dv], or None when ``want_dh0`` is False).  ``do`` has v's dtype and
    shape; ``dhT`` (fp32 [N, H, dk, dv]) may be None.  The gate must be fp32."""
    B, T, H, dk, dv, N, dev = _validate(q, k, v, g, beta, h0, cu_seqlens, None, None, False)
    _check(do, "do", q.dtype, (B, T, H, dv), dev)
    if dhT is not None:
        _check(dhT, "dhT", torch.float32, (N, H, dk, dv), dev)
    lib = load_library()
    if scale is None:
        scale = dk ** -0.5
    f32 = dict(dtype=torch.float32, device=dev)
    dq = torch.empty((B, T, H, dk), **f32)
    dk_ = torch.empty((B, T, H, dk), **f32)
    dv_ = torch.empty((B, T, H, dv), **f32)
    dg = torch.empty((B, T, H, dk), **f32)
    dbeta = torch.empty((B, T, H), **f32)
    dh0 = torch.empty((N, H, dk, dv), **f32) if want_dh0 else None
    ws_bytes = int(lib.kda_bwd_workspace_size(B, T, H, dk, dv, N))
    if ws_bytes == 0:
        raise KdaError(2, "kda_bwd_workspace_size")
    if workspace is None or workspace.numel() - (-workspace.data_ptr()) % 256 < ws_bytes:
        workspace = torch.empty(ws_bytes + 256, dtype=torch.uint8, device=dev)
    ws_ptr = (workspace.data_ptr() + 255) & ~255
    avail = workspace.numel() - (ws_ptr - workspace.data_ptr())
    stream = torch.cuda.current_stream(dev).cuda_stream
    dt = KDA_BF16 if q.dtype == torch.bfloat16 else KDA_FP32
    st = lib.kda_bwd(_ptr(q), _ptr(k), _ptr(v), dt, _ptr(g), _ptr(beta), _ptr(h0), _ptr(cu_seqlens),
                     N, B, T, H, dk, dv, float(scale), _ptr(do), _ptr(dhT), _ptr(dq), _ptr(dk_),
                     _ptr(dv_), _ptr(dg), _ptr(dbeta), _ptr(dh0), ctypes.c_void_p(ws_ptr), avail,
                     ctypes.c_void_p(stream))
    if st != KDA_OK:
        raise KdaError(st, "kda_bwd")
    if check:
        err = ctypes.c_uint32(0)
        st = lib.kda_fwd_check(ctypes.c_void_p(ws_ptr), ctypes.c_void_p(stream), ctypes.byref(err))
        if st != KDA_OK:
            raise KdaError(st, f"kda_bwd (device error bits {err.value:#x})")
    return dq, dk_, dv_, dg, dbeta, dh0


__all__ = ["fwd", "bwd", "fwd_noalloc", "workspace_size", "launch_count", "load_library", "KdaError",
           "LIB_PATH", "set_pipeline", "get_pipeline", "uses_fused"]


def decode(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, g: torch.Tensor,
           beta: torch.Tensor, state: Optional[torch.Tensor] = None,
           scale: Optional[float] = None, *, out_state: Optional[torch.Tensor] = None,
           o: Optional[torch.Tensor] = None) -> Tuple[torch.Tensor, torch.Tensor]:
    """One recurrence step per sequence (single-token decode), via ``kda_decode``.

    q, k: [N, H, dk]; v: [N, H, dv] (bf16 or fp32); g: [N, H, dk] fp32; beta: [N, H]
    fp32; state: [N, H, dk, dv] fp32 or None (zeros).  Returns (o [N, H, dv] in q's
    dtype, new state).  ``out_state`` may be ``state`` itself (update in place);
    by default a new tensor is returned."""
    lib = load_library()
    if q.dim() != 3:
        raise ValueError("q must be [N, H, dk]")
    N, H, dk = q.shape
    dv = v.shape[-1]
    dev = q.device
    if dev.type != "cuda":
        raise ValueError("inputs must be CUDA tensors")
    if q.dtype not in (torch.bfloat16, torch.float32):
        raise TypeError("q, k, v must be bfloat16 or float32")
    _check(q, "q", q.dtype, (N, H, dk), dev)
    _check(k, "k", q.dtype, (N, H, dk), dev)
    _check(v, "v", q.dtype, (N, H, dv), dev)
    _check(g, "g", torch.float32, (N, H, dk), dev)
    _check(beta, "beta", torch.float32, (N, H), dev)
    if state is not None:
        _check(state, "state", torch.float32, (N, H, dk, dv), dev)
    if out_state is None:
        out_state = torch.empty((N, H, dk, dv), dtype=torch.float32, device=dev)
    else:
        _check(out_state, "out_state", torch.float32, (N, H, dk, dv), dev)
    if o is None:
        o = torch.empty((N, H, dv), dtype=q.dtype, device=dev)
    else:
        _check(o, "o", q.dtype, (N, H, dv), dev)
    if scale is None:
        scale = dk ** -0.5
    stream = torch.cuda.current_stream(dev).cuda_stream
    dt = KDA_BF16 if q.dtype == torch.bfloat16 else KDA_FP32
    st = lib.kda_decode(_ptr(q), _ptr(k), _ptr(v), dt, _ptr(g), _ptr(beta), _ptr(state),
                        _ptr(out_state), N, H, dk, dv, float(scale), _ptr(o),
                        ctypes.c_void_p(stream))
    if st != KDA_OK:
        raise KdaError(st, "kda_decode")
    return o, out_state
