"""Comparison rules shared by the parity tests.

The floating-point bar for a GEMM output Y (bf16) against the fp64 oracle Yref:
  |y - yref| <= 8e-3 * |yref| + 2e-3 * max|Yref|   element-wise, and
  cosine(Y, Yref) >= 0.99999 over the whole output,
both evaluated in fp64.
"""
from __future__ import annotations

import numpy as np

REL_TOL = 8e-3
ABS_TOL_FRAC = 2e-3
COS_MIN = 0.99999


def bf16_bits_to_f64(bits) -> np.ndarray:
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def compare(y, yref, mask=None):
    """Return (ok, report) for y (fp64 values) against yref (fp64)."""
    y = np.asarray(y, dtype=np.float64)
    yref = np.asarray(yref, dtype=np.float64)
    if mask is not None:
        y, yref = y[mask], yref[mask]
    y = y.ravel()
    yref = yref.ravel()
    if yref.size == 0:
        return True, {"n": 0}
    scale = float(np.max(np.abs(yref)))
    err = np.abs(y - yref)
    bound = REL_TOL * np.abs(yref) + ABS_TOL_FRAC * scale
    finite = bool(np.all(np.isfinite(y)))
    within = bool(np.all(err <= bound)) and finite
    denom = float(np.linalg.norm(y) * np.linalg.norm(yref))
    if denom == 0.0:
        cos = 1.0 if float(np.linalg.norm(y - yref)) == 0.0 else 0.0
    else:
        cos = float(np.dot(y, yref) / denom)
    ok = within and cos >= COS_MIN
    worst = int(np.argmax(err - bound)) if y.size else 0
    return ok, {
        "n": int(y.size), "max_abs_ref": scale, "max_err": float(err.max()),
        "worst_excess": float((err - bound)[worst]), "cos": cos, "finite": finite,
    }


def assert_close(y, yref, mask=None, what=""):
    ok, rep = compare(y, yref, mask)
    assert ok, f"{what} parity failed: {rep}"
    return rep
