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


# Attention forward ("Two Waves, One Stage Apart", section "Beyond GEMM:
# FlashAttention"). The probabilities enter the PV product rounded to the
# operand type (relative error <= 2^-9 for BF16, 2^-12 for FP16) while the
# row sum l is taken before the rounding, so the output error is at most about
# 2^-9 * O_abs from the numerator plus 2^-9 * |O| from the normalisation,
# <= 2^-8 * O_abs with O_abs = sum_k p_k |v_k| / l; the FP32 score and output
# sums add far less. The bound below doubles that.
#
# The row log-sum-exp LSE = log sum_j exp(t_j), t_j = scale * q.k_j, sees no
# rounding to the operand type. An error d_j in each score moves it by
# sum_j p_j d_j <= max_j |d_j|, and the FP32 dot product of d = 128 exact
# products errs by at most gamma_d * scale * sum_i |q_i k_ji| with
# gamma_d ~ d * 2^-24 = 2^-17: twice that, times S_abs = scale * max_j
# sum_i |q_i k_ji|, bounds the score term. The FP32 row sum of about 160
# sequential additions of probabilities (each from one 2^-22-accurate ex2)
# errs by under 160 * 2^-24 < 2^-16 relative, which moves the logarithm by
# the same amount; and the final FP32 value carries a few ulps of |LSE|.
ATT_REL = 2.0 ** -7
ATT_LSE_SCORE = 2.0 ** -16
ATT_LSE_ABS = 2.0 ** -16
ATT_LSE_ULPS = 4.0


def attention_lse_bound(L_ref, S_abs):
    """|LSE - LSE_ref| bound for rows with finite LSE_ref (see above)."""
    L_ref = np.asarray(L_ref, dtype=np.float64)
    return (ATT_LSE_SCORE * np.asarray(S_abs, dtype=np.float64) + ATT_LSE_ABS
            + ATT_LSE_ULPS * ulp_out(L_ref, "f32"))


def check_lse(lse_gpu, L_ref, S_abs):
    """Rows with a visible key must be finite and within attention_lse_bound; rows
    without one must be -inf on both sides. Returns (ok, worst ratio, n_bad)."""
    lse_gpu = np.asarray(lse_gpu, dtype=np.float64)
    L_ref = np.asarray(L_ref, dtype=np.float64)
    fin = np.isfinite(L_ref)
    same_inf = np.array_equal(np.isfinite(lse_gpu), fin) and np.all(lse_gpu[~fin] == L_ref[~fin])
    err = np.abs(lse_gpu[fin] - L_ref[fin])
    lim = attention_lse_bound(L_ref[fin], np.asarray(S_abs, dtype=np.float64)[fin])
    bad = ~(err <= lim)
    ratio = float(np.max(err / lim)) if err.size else 0.0
    return bool(same_inf and not bad.any()), ratio, int(bad.sum())


def attention_bound(O_ref, O_abs, dtype_out: str):
    return ATT_REL * O_abs + 1e-6 + ulp_out(O_ref, dtype_out)


def check_attention(O_gpu, O_ref, O_abs, dtype_out: str):
    """Elementwise |O_gpu - O_ref| <= attention_bound. Returns (ok, worst ratio, n_bad, first bad)."""
    O_gpu = np.asarray(O_gpu, dtype=np.float64)
    err = np.abs(O_gpu - O_ref)
    lim = attention_bound(O_ref, O_abs, dtype_out)
    bad = ~(err <= lim)
    ratio = float(np.max(err / lim)) if err.size else 0.0
    idx = np.argwhere(bad)
    return (not bad.any(), ratio, int(bad.sum()), tuple(int(i) for i in idx[0]) if idx.size else None)
