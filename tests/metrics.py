"""Error metrics used by the parity gates (fp64 throughout).

The pages name relative RMSE for outputs and final states ("NVIDIA Kernel Design
Agents optimize Kimi Delta Attention", section 01 RESULTS, the two accuracy
charts) without a formula; the reading taken is the Frobenius ratio over the
whole tensor.  Element-wise maxima (section 04 HARDENING, strict element-wise
tolerances) are reported as diagnostics.
"""
from __future__ import annotations

import numpy as np

# Gates: output relative RMSE <= 1e-2, final-state relative RMSE <= 5e-3.
O_TOL = 1e-2
HT_TOL = 5e-3


def _np(x) -> np.ndarray:
    if hasattr(x, "detach"):
        x = x.detach().to("cpu").double().numpy()
    return np.asarray(x, dtype=np.float64)


def rel_rmse(x, ref) -> float:
    """||x - ref||_F / ||ref||_F over the whole tensor (0 when both vanish)."""
    x, ref = _np(x), _np(ref)
    num = np.sqrt(np.sum((x - ref) ** 2))
    den = np.sqrt(np.sum(ref ** 2))
    if den == 0.0:
        return 0.0 if num == 0.0 else float("inf")
    return float(num / den)


def max_abs(x, ref) -> float:
    x, ref = _np(x), _np(ref)
    return float(np.max(np.abs(x - ref))) if x.size else 0.0


def per_sequence_rel_rmse(o, ref, lens):
    """Output relative RMSE of each packed sequence (o, ref: [1, T, H, dv])."""
    o, ref = _np(o), _np(ref)
    out, pos = [], 0
    for L in lens:
        out.append(rel_rmse(o[:, pos:pos + L], ref[:, pos:pos + L]) if L else 0.0)
        pos += L
    return out


def report(o, hT, o_ref, hT_ref) -> dict:
    return {"o_rel_rmse": rel_rmse(o, o_ref), "hT_rel_rmse": rel_rmse(hT, hT_ref),
            "o_max_abs": max_abs(o, o_ref), "hT_max_abs": max_abs(hT, hT_ref)}


def passes(rep: dict) -> bool:
    """Both gates met, and every value finite."""
    ok = rep["o_rel_rmse"] <= O_TOL and rep["hT_rel_rmse"] <= HT_TOL
    return bool(ok and np.isfinite(rep["o_max_abs"]) and np.isfinite(rep["hT_max_abs"]))
