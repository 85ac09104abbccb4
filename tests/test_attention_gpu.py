"""Parity of the attention forward pass (attention_fwd) against the FP64 oracle.

Bound (oracle/tolerance.py): |O - O_ref| <= 2^-7 * sum_k p_k |v_k| / l + 1e-6
+ one output ulp, from the rounding of the probabilities to the operand type
before the PV product; and |LSE - LSE_ref| <= 2^-16 * S_abs + 2^-16 + 4 ulps,
from the FP32 scores (S_abs = scale * max_j sum_i |q_i k_ji|) and the FP32
row sum. Closed forms are
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


def score_abs_max(Q, K, scale, rows=None):
    """scale * max_j sum_i |q_i k_ji| for each query row (over every key of its head):
    the size of the FP32 score error, for the log-sum-exp bound."""
    B, H, Lq, d = Q.shape
    Lk = K.shape[2]
    scale = d ** -0.5 if scale is None else scale
    Qa = Q.double().abs().reshape(B * H, Lq, d)
    Ka = K.double().abs().reshape(B * H, Lk, d)
    if rows is None:
        return (torch.bmm(Qa, Ka.transpose(1, 2)).amax(dim=2).reshape(-1) * scale).numpy()
    rows = np.asarray(rows)
    head, qi = rows // Lq, rows % Lq
    out = np.empty(len(rows))
    for h in np.unique(head):
        sel = np.nonzero(head == h)[0]
        out[sel] = (Qa[h, qi[sel]] @ Ka[h].T).amax(dim=1).numpy() * scale
    return out


def check(Q, K, V, O, lse, B, H, Lq, Lk, dtype, causal, scale=None, rows=None):
    O_ref, O_abs, L_ref = oracle.attention_ref(bits(Q), bits(K), bits(V), B, H, Lq, Lk, 128, dtype, causal,
                                               scale, rows=rows)
    got = O.float().numpy().astype(np.float64).reshape(-1, 128)
    lse = lse.numpy().astype(np.float64).reshape(-1)
    if rows is not None:
        got, lse = got[rows], lse[rows]
    ok, ratio, n_bad, first = tolerance.check_attention(got, O_ref, O_abs, dtype)
    assert ok, f"{n_bad} out of bound (worst {ratio:.3g}) first {first}: gpu {got[first]} ref {O_ref[first]}"
    ok, lratio, n_bad = tolerance.check_lse(lse, L_ref, score_abs_max(Q, K, scale, rows))
    assert ok, f"log-sum-exp: {n_bad} rows out of bound (worst error/bound {lratio:.3g})"
    return ratio, lratio


def case(dtg, B, H, Lq, Lk, dtype="bf16", causal=False, seed=0, q_scale=1.0, rows=None, scale=None,
         max_ctas=0):
    Q, K, V = workloads.make_attention_operands(B, H, Lq, Lk, 128, dtype, ("normal", 1.0), seed)
    Q = (Q.float() * q_scale).to(TDT[dtype])
    O, lse = run(dtg, Q, K, V, causal, scale, max_ctas)
    return check(Q, K, V, O, lse, B, H, Lq, Lk, dtype, causal, scale, rows)


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


@pytest.mark.parametrize("causal", [False, True], ids=["full", "causal"])
@pytest.mark.parametrize("profile", ["jump", "ramp", "fall"])
def test_row_maximum_moves_mid_row(dtg, profile, causal):
    """Key blocks scaled so that the row maxima (in log2 units of the scaled scores)
    jump by far more than the lazy-rescale threshold of 2^8 mid-row ("jump": blocks 3
    and later x12), climb past it in steps each below it ("ramp": block j x (1 + j/2)),
    or fall after the first blocks ("fall": x8 then x1). O and the log-sum-exp must
    match the oracle in every case."""
    B, H, Lq, Lk = 1, 2, 256, 1024
    Q, K, V = workloads.make_attention_operands(B, H, Lq, Lk, 128, "bf16", ("normal", 1.0), 40)
    blk = torch.arange(Lk) // 128
    if profile == "jump":
        f = torch.where(blk >= 3, 12.0, 1.0)
    elif profile == "ramp":
        f = 1.0 + blk.double() / 2
    else:
        f = torch.where(blk < 2, 8.0, 1.0)
    K = (K.double() * f[None, None, :, None]).to(torch.bfloat16)
    O, lse = run(dtg, Q, K, V, causal)
    check(Q, K, V, O, lse, B, H, Lq, Lk, "bf16", causal)
    # the scaled scores' row maxima (log2 units) do what the profile says: grow by more
    # than 2^8 past the first block, or never rise after the first two blocks
    t = (Q.double() @ K.double().transpose(-1, -2)) * 128 ** -0.5 / math.log(2)
    if profile in ("jump", "ramp"):
        grew = (t.amax(-1) - t[..., :128].amax(-1) > 8).double().mean().item()
        assert grew > 0.9, grew
    else:
        assert bool((t[..., 256:].amax(-1) < t[..., :256].amax(-1)).all())


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
