"""Parity of the attention forward pass (attention_fwd) against the FP64 oracle.

Bound (oracle/tolerance.py): |O - O_ref| <= 2^-7 * sum_k p_k |v_k| / l + 1e-6
+ one output ulp, and |LSE - LSE_ref| <= 2^-7, from the rounding of the
probabilities to the operand type before the PV product. Closed forms are
checked exactly: with Q = 0 every visible key has probability 1, so O is the
mean of the visible value rows; causal row 0 sees only key 0, so it returns
V[0]; a row with no visible key returns zeros and LSE = -inf.
"""
from __future__ import annotations

import math

import numpy as np
import pytest
import torch

import oracle
from oracle import tolerance
import workloads

pytestmark = pytest.mark.gpu

TDT = {"f16": torch.float16, "bf16": torch.bfloat16}


@pytest.fixture(scope="module")
def dtg():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import dense_tiled_gemm_gb300 as mod
    torch.cuda.set_device(0)
    mod.gemm_last_device_status()
    return mod


def bits(t):
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def run(dtg, Q, K, V, causal=False, scale=None, max_ctas=0):
    O, lse = dtg.attention(Q.cuda(), K.cuda(), V.cuda(), causal=causal, scale=scale, return_lse=True,
                           max_ctas=max_ctas)
    status, detail = dtg.gemm_last_device_status()
    assert status == dtg.GEMM_OK, f"device status {dtg.gemm_status_string(status)} site {detail:#x}"
    return O.cpu(), lse.cpu()


def case(dtg, B, H, Lq, Lk, dtype="bf16", causal=False, seed=0, q_scale=1.0, rows=None, scale=None,
         max_ctas=0):
    Q, K, V = workloads.make_attention_operands(B, H, Lq, Lk, 128, dtype, ("normal", 1.0), seed)
    Q = (Q.float() * q_scale).to(TDT[dtype])
    O, lse = run(dtg, Q, K, V, causal, scale, max_ctas)
    O_ref, O_abs, L_ref = oracle.attention_ref(bits(Q), bits(K), bits(V), B, H, Lq, Lk, 128, dtype, causal,
                                               scale, rows=rows)
    got = O.float().numpy().astype(np.float64).reshape(-1, 128)
    lse = lse.numpy().astype(np.float64).reshape(-1)
    if rows is not None:
        got, lse = got[rows], lse[rows]
    ok, ratio, n_bad, first = tolerance.check_attention(got, O_ref, O_abs, dtype)
    assert ok, f"{n_bad} out of bound (worst {ratio:.3g}) first {first}: gpu {got[first]} ref {O_ref[first]}"
    fin = np.isfinite(L_ref)
    assert np.array_equal(np.isfinite(lse), fin)
    assert np.all(np.abs(lse[fin] - L_ref[fin]) <= tolerance.ATT_LSE_ABS)


# ---------------------------------------------------------------- one tile, one block
@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_single_block(dtg, dtype):
    case(dtg, 1, 1, 128, 128, dtype)


def test_zero_q_gives_mean_of_values(dtg):
    """Q = 0: every probability is exactly 1, O = mean of V (integers keep the sum exact)."""
    B, H, Lq, Lk = 1, 2, 128, 384
    g = torch.Generator().manual_seed(1)
    Q = torch.zeros(B, H, Lq, 128, dtype=torch.bfloat16)
    K = torch.randn(B, H, Lk, 128, generator=g).to(torch.bfloat16)
    V = torch.randint(-4, 5, (B, H, Lk, 128), generator=g).to(torch.bfloat16)
    O, lse = run(dtg, Q, K, V)
    mean = V.double().mean(dim=2, keepdim=True).expand(B, H, Lq, 128)
    assert torch.equal(O, mean.to(torch.bfloat16))
    assert torch.allclose(lse.double(), torch.full((B, H, Lq), math.log(Lk), dtype=torch.float64), atol=1e-6)


def test_causal_first_row_returns_first_value(dtg):
    Q, K, V = workloads.make_attention_operands(1, 1, 256, 256, 128, "bf16", ("normal", 1.0), 2)
    O, _ = run(dtg, Q, K, V, causal=True)
    assert torch.equal(O[0, 0, 0], V[0, 0, 0])


def test_rows_without_visible_keys(dtg):
    """Causal with Lq > Lk: the first Lq - Lk rows see no key at all."""
    Q, K, V = workloads.make_attention_operands(1, 1, 300, 100, 128, "bf16", ("normal", 1.0), 3)
    O, lse = run(dtg, Q, K, V, causal=True)
    assert torch.count_nonzero(O[0, 0, :200]) == 0
    assert torch.all(torch.isinf(lse[0, 0, :200])) and torch.all(lse[0, 0, :200] < 0)
    case(dtg, 1, 1, 300, 100, causal=True, seed=3)


# ---------------------------------------------------------------- many blocks, masks, tails
@pytest.mark.parametrize("causal", [False, True], ids=["full", "causal"])
@pytest.mark.parametrize("shape", [(1, 2, 256, 1024), (2, 3, 200, 300), (1, 1, 128, 1), (1, 1, 1, 129),
                                   (1, 2, 384, 384), (1, 1, 1000, 777)], ids=lambda s: "x".join(map(str, s)))
def test_shapes(dtg, shape, causal):
    B, H, Lq, Lk = shape
    case(dtg, B, H, Lq, Lk, "bf16", causal, seed=sum(shape))


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_large_scores_rescale(dtg, dtype):
    """Scores in the tens: the running maximum grows across blocks and O is rescaled."""
    case(dtg, 1, 2, 256, 1024, dtype, seed=4, q_scale=6.0)


def test_custom_scale(dtg):
    case(dtg, 1, 1, 256, 512, "bf16", seed=5, scale=0.3)


# ---------------------------------------------------------------- the workloads, sampled
@pytest.mark.parametrize("name", sorted(workloads.ATTENTION_WORKLOADS))
def test_workload_sampled(dtg, name):
    w = workloads.ATTENTION_WORKLOADS[name]
    total = w.B * w.H * w.Lq
    rows = sorted(set(workloads.sample_rows(total, 64, w.seed)) | {0, w.Lq - 1, total - 1})
    case(dtg, w.B, w.H, w.Lq, w.Lk, w.dtype, w.causal, w.seed, rows=rows)


# ---------------------------------------------------------------- persistent CTAs, many row blocks each
@pytest.mark.parametrize("causal", [False, True], ids=["full", "causal"])
@pytest.mark.parametrize("shape,cap", [((2, 3, 1000, 777), 1), ((1, 5, 600, 1100), 2), ((3, 2, 513, 300), 3),
                                       ((1, 2, 300, 100), 2)], ids=lambda v: "x".join(map(str, v))
                         if isinstance(v, tuple) else f"cap{v}")
def test_capped_grid(dtg, shape, cap, causal):
    """A capped grid makes every CTA walk several row blocks (different key-block
    counts under the causal mask, rows with no visible key when Lk < Lq): the ring
    and barrier phases carried from one block to the next must give the oracle's
    result, and the same bits as the uncapped launch."""
    B, H, Lq, Lk = shape
    case(dtg, B, H, Lq, Lk, "bf16", causal, seed=sum(shape) + cap, max_ctas=cap)
    Q, K, V = workloads.make_attention_operands(B, H, Lq, Lk, 128, "f16", ("normal", 1.0), 7)
    O1, l1 = run(dtg, Q, K, V, causal, None, 0)
    O2, l2 = run(dtg, Q, K, V, causal, None, cap)
    assert torch.equal(O1, O2) and torch.equal(l1, l2)


def test_many_heads(dtg):
    """70,007 heads of 3 query rows and 5 keys: more (batch, head) pairs than a 2-D
    grid's y extent, so each persistent CTA walks hundreds of row blocks."""
    case(dtg, 7, 10001, 3, 5, "bf16", False, seed=31)
    case(dtg, 7, 10001, 3, 5, "bf16", True, seed=32)
