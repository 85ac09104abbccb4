"""Pins for the CPU FP64 attention oracle (no GPU).

The oracle (oracle/attention_oracle.c) computes softmax(scale * Q K^T) V
directly. It is checked against things other than itself: torch's float64
scaled_dot_product_attention (a library routine), torch's logsumexp for the
LSE, and closed forms: uniform scores average V, a single key returns its
value row, the first causal row sees only key 0, a common score shift leaves
O unchanged and moves LSE by the shift, permuting keys with their values
leaves O unchanged, and one dominant key returns its value row. Planted
mistakes compiled from the source must each fail one of these pins.
"""
from __future__ import annotations

import math
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

import oracle

TDT = {"f16": torch.float16, "bf16": torch.bfloat16}


def bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def operands(B, H, Lq, Lk, d, dtype, seed, q_scale=1.0):
    g = torch.Generator().manual_seed(seed)
    q = (q_scale * torch.randn(B, H, Lq, d, generator=g)).to(TDT[dtype])
    k = torch.randn(B, H, Lk, d, generator=g).to(TDT[dtype])
    v = torch.randn(B, H, Lk, d, generator=g).to(TDT[dtype])
    return q, k, v


def run(lib, q, k, v, dtype, causal=False, scale=None, rows=None):
    B, H, Lq, d = q.shape
    Lk = k.shape[2]
    return oracle.attention_ref(bits(q), bits(k), bits(v), B, H, Lq, Lk, d, dtype, causal, scale,
                                rows=rows, lib=lib)


def _pin_sdpa(lib):
    out = []
    for (B, H, Lq, Lk, d) in ((1, 1, 1, 1, 8), (2, 3, 5, 7, 16), (1, 2, 9, 4, 32), (1, 1, 33, 33, 64)):
        for dtype in ("f16", "bf16"):
            for causal in (False, True):
                # q_scale 8 gives scores in the hundreds: exp overflows without the max shift
                for q_scale in (1.0, 8.0):
                    q, k, v = operands(B, H, Lq, Lk, d, dtype, B + H + Lq + Lk + d, q_scale)
                    O, _, LSE = run(lib, q, k, v, dtype, causal)
                    mask = torch.ones(Lq, Lk, dtype=torch.bool).tril(diagonal=Lk - Lq) if causal else None
                    if causal and Lk - Lq < 0:
                        continue
                    ref = torch.nn.functional.scaled_dot_product_attention(
                        q.double(), k.double(), v.double(), attn_mask=mask).reshape(-1, d).numpy()
                    s = (q.double() @ k.double().transpose(-1, -2)) / math.sqrt(d)
                    if mask is not None:
                        s = s.masked_fill(~mask, float("-inf"))
                    lse = torch.logsumexp(s, dim=-1).reshape(-1).numpy()
                    if not (np.all(np.isfinite(O)) and np.allclose(O, ref, rtol=1e-12, atol=1e-12)
                            and np.allclose(LSE, lse, rtol=1e-12, atol=1e-12)):
                        out.append(f"sdpa_{B}x{H}x{Lq}x{Lk}x{d}_{dtype}_{causal}_{q_scale}")
    return out


def _pin_closed_forms(lib):
    out = []
    g = torch.Generator().manual_seed(3)
    d = 16
    # uniform scores: K = 0 -> every p = 1 -> O = mean of V, LSE = log(Lk)
    q = torch.randn(1, 1, 4, d, generator=g).half()
    k = torch.zeros(1, 1, 9, d).half()
    v = torch.randn(1, 1, 9, d, generator=g).half()
    O, _, LSE = run(lib, q, k, v, "f16")
    mean = np.array([math.fsum(v[0, 0, :, c].double().tolist()) / 9 for c in range(d)])
    if not (np.allclose(O, mean[None, :], rtol=1e-15, atol=1e-15) and np.allclose(LSE, math.log(9))):
        out.append("uniform")
    # a single key returns its value row exactly
    k1 = torch.randn(1, 1, 1, d, generator=g).half()
    v1 = torch.randn(1, 1, 1, d, generator=g).half()
    O, _, LSE = run(lib, q, k1, v1, "f16")
    s0 = (q.double()[0, 0] @ k1.double()[0, 0, 0]) / math.sqrt(d)
    if not (np.array_equal(O, np.repeat(v1.double().reshape(1, d).numpy(), 4, 0))
            and np.allclose(LSE, s0.numpy(), rtol=1e-15, atol=1e-15)):
        out.append("single_key")
    # causal, Lq == Lk: row 0 sees key 0 only
    q, k, v = operands(1, 1, 6, 6, d, "bf16", 5)
    O, _, _ = run(lib, q, k, v, "bf16", causal=True)
    if not np.array_equal(O[0], v.double()[0, 0, 0].numpy()):
        out.append("causal_row0")
    # a common score shift: extra feature q = 4, k = 1 shifts every score by 4 * scale
    q, k, v = operands(1, 2, 5, 7, d, "f16", 6)
    qx = torch.cat([q, torch.full((1, 2, 5, 1), 4.0).half()], dim=-1)
    kx = torch.cat([k, torch.ones(1, 2, 7, 1).half()], dim=-1)
    vx = torch.cat([v, torch.zeros(1, 2, 7, 1).half()], dim=-1)
    scale = 0.25
    O0, _, L0 = run(lib, q, k, v, "f16", scale=scale)
    O1, _, L1 = run(lib, qx, kx, vx, "f16", scale=scale)
    if not (np.allclose(O1[:, :d], O0, rtol=1e-13, atol=1e-14) and np.allclose(L1, L0 + 4 * scale, rtol=1e-14)):
        out.append("shift")
    # permuting keys together with their values leaves O unchanged
    perm = torch.randperm(7, generator=g)
    O2, _, L2 = run(lib, q, k[:, :, perm], v[:, :, perm], "f16", scale=scale)
    if not (np.allclose(O2, O0, rtol=1e-13, atol=1e-14) and np.allclose(L2, L0, rtol=1e-14)):
        out.append("permutation")
    # one dominant key (score 60 above the rest) returns its value row
    k3 = torch.zeros(1, 1, 5, d).half()
    k3[0, 0, 2, 0] = 15.0
    q3 = torch.zeros(1, 1, 1, d).half()
    q3[0, 0, 0, 0] = 4.0
    v3 = torch.randn(1, 1, 5, d, generator=g).half()
    O3, _, L3 = run(lib, q3, k3, v3, "f16", scale=1.0)
    if not (np.allclose(O3[0], v3.double()[0, 0, 2].numpy(), rtol=1e-20, atol=1e-20 + 4 * math.exp(-60) * 8)
            and abs(L3[0] - 60.0) < 1e-20 + 5 * math.exp(-60)):
        out.append("dominant")
    return out


def _pin_abs_and_rows(lib):
    out = []
    q, k, v = operands(2, 2, 6, 9, 16, "bf16", 8)
    O, Oa, L = run(lib, q, k, v, "bf16")
    s = torch.softmax((q.double() @ k.double().transpose(-1, -2)) / 4.0, dim=-1)
    oa = (s @ v.double().abs()).reshape(-1, 16).numpy()
    if not np.allclose(Oa, oa, rtol=1e-12, atol=1e-13):
        out.append("o_abs")
    rows = [23, 0, 5, 5, 12]
    Or, Oar, Lr = run(lib, q, k, v, "bf16", rows=rows)
    if not (np.array_equal(Or, O[rows]) and np.array_equal(Oar, Oa[rows]) and np.array_equal(Lr, L[rows])):
        out.append("rows")
    return out


PINS = [_pin_sdpa, _pin_closed_forms, _pin_abs_and_rows]


def pin_battery(lib):
    failed = []
    for pin in PINS:
        try:
            failed += pin(lib)
        except Exception as exc:  # a crash in a mutant counts as a caught mistake
            failed.append(f"{pin.__name__}: {type(exc).__name__}")
    return failed


@pytest.fixture(scope="module")
def lib():
    return oracle._load()


@pytest.mark.parametrize("pin", PINS, ids=lambda p: p.__name__[5:])
def test_pin(lib, pin):
    assert pin(lib) == []


def test_argument_errors(lib):
    q = np.zeros(8, np.uint16)
    with pytest.raises(ValueError):
        oracle.attention_ref(q, q, q, 1, 1, 2, 2, 3, "f16")
    with pytest.raises(RuntimeError):                  # flat row 4 of 2 x 2 rows does not exist
        oracle.attention_ref(q[:4], q[:4], q[:4], 1, 1, 2, 2, 2, "f16", rows=[4])


MUTANTS = {
    "no_max_shift": ("s[k] = exp(s[k] - m);", "s[k] = exp(s[k]);"),
    "scale_dropped": ("s[k] = j->scale * acc;", "s[k] = acc;"),
    "causal_offset": ("n_keys = i + (Lk - j->Lq) + 1;", "n_keys = i + 1;"),
    "not_normalised": ("o[c] = n_keys ? o[c] / l : 0.0;", "o[c] = n_keys ? o[c] : 0.0;"),
    "lse_without_log": ("j->LSE[r] = n_keys ? m + log(l) : -INFINITY;", "j->LSE[r] = n_keys ? m + l : -INFINITY;"),
    "first_key_skipped": ("        for (int64_t k = 0; k < n_keys; ++k) {\n            double acc",
                          "        for (int64_t k = 1; k < n_keys; ++k) {\n            double acc"),
    "v_row_swapped": ("dec(vmat[k * d + c], j->dtype)", "dec(vmat[(n_keys - 1 - k) * d + c], j->dtype)"),
    "abs_dropped": ("oa[c] += fabs(pv);", "oa[c] += pv;"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistakes(name, tmp_path):
    src = open(oracle._ATT_SRC).read()
    old, new = MUTANTS[name]
    assert src.count(old) == 1, f"mutation anchor for {name} not unique"
    path = tmp_path / "attention_mutant.c"
    path.write_text(src.replace(old, new))
    so = tmp_path / "libmutant.so"
    subprocess.run(oracle.compile_cmd(str(so), (oracle._SRC, str(path))), check=True)
    here = os.path.dirname(os.path.abspath(__file__))
    code = ("import sys; sys.path[:0] = [%r, %r]; import oracle, test_attention_oracle as t; "
            "failed = t.pin_battery(oracle.load_library(%r)); sys.exit(0 if failed else 3)"
            ) % (here, os.path.dirname(here), str(so))
    res = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=600)
    assert res.returncode != 3, f"no pin caught the planted mistake {name}"
