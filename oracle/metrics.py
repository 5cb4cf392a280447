"""Error metric of the parity tests (test infrastructure only).

rel_err = max_i |g_i - o_i| / max(|o_i|, rms(o)): element-wise relative
error with a floor at the RMS of the oracle's output, so that elements near
zero do not dominate.  The Frobenius-norm relative error is reported beside
it.  Bars: 1e-2 for bf16 paths (fp32 accumulate), 1e-4 for fp32.
"""
from __future__ import annotations

import numpy as np


def rel_err(got, want) -> float:
    g = np.asarray(got, np.float64).ravel()
    o = np.asarray(want, np.float64).ravel()
    if o.size == 0:
        return 0.0
    rms = float(np.sqrt(np.mean(o * o)))
    den = np.maximum(np.abs(o), rms)
    den[den == 0] = 1.0
    return float(np.max(np.abs(g - o) / den))


def fro_err(got, want) -> float:
    g = np.asarray(got, np.float64).ravel()
    o = np.asarray(want, np.float64).ravel()
    n = float(np.linalg.norm(o))
    return float(np.linalg.norm(g - o) / (n if n > 0 else 1.0))


BF16_TOL = 1e-2
F32_TOL = 1e-4
