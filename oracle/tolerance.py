"""Acceptance bound for a GPU GEMM result against the FP64 oracle: test
infrastructure only.

An element passes when

    |C_gpu - C_ref| <= 2e-3 * C_abs + 1e-6 + ulp_out(|C_ref|)

with C_abs = sum_k |a_ik * b_kj| and ulp_out(x) the spacing of the output
format at x. The pages give no tolerance; this is the bound the build sets for
FP32 accumulation (rounding error at most about K * 2^-24 * C_abs, which is
4.9e-4 * C_abs at K = 8192 and 9.8e-4 * C_abs at K = 16384, below 2e-3),
plus one rounding of the cast on store.

ulp_out(x) = 2^(floor(log2 x) - p) for x at or above the smallest normal
2^emin, and 2^(emin - p) below it, with (p, emin) = (10, -14) for FP16,
(7, -126) for BF16 and (23, -126) for FP32.
"""
from __future__ import annotations

import numpy as np

FORMATS = {"f16": (10, -14), "bf16": (7, -126), "f32": (23, -126)}
REL = 2e-3
ABS = 1e-6


def ulp_out(x, dtype_out: str) -> np.ndarray:
    p, emin = FORMATS[dtype_out]
    ax = np.abs(np.asarray(x, dtype=np.float64))
    # frexp: ax = m * 2^e with m in [0.5, 1), so floor(log2 ax) = e - 1
    _, e = np.frexp(ax)
    expo = np.where(ax >= np.ldexp(1.0, emin), e - 1, emin)
    return np.ldexp(1.0, expo - p)


def bound(C_ref, C_abs, dtype_out: str) -> np.ndarray:
    return REL * np.asarray(C_abs) + ABS + ulp_out(C_ref, dtype_out)


def check(C_gpu, C_ref, C_abs, dtype_out: str):
    """Return (ok, worst error/bound ratio, number of failing elements, first failing index)."""
    C_gpu = np.asarray(C_gpu, dtype=np.float64)
    C_ref = np.asarray(C_ref, dtype=np.float64)
    err = np.abs(C_gpu - C_ref)
    lim = bound(C_ref, C_abs, dtype_out)
    bad = ~(err <= lim)          # NaN in the result counts as a failure
    n_bad = int(bad.sum())
    ratio = float(np.nanmax(err / lim)) if err.size else 0.0
    first = tuple(int(v) for v in np.argwhere(bad)[0]) if n_bad else None
    return n_bad == 0, ratio, n_bad, first
