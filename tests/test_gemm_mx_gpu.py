"""Parity of the block-scaled (MX) GEMM against the FP64 CPU oracle.

The MXFP8 and MXFP4 GEMMs of "Two Waves, One Stage Apart" (section "MI450",
Table 1), in the OCP Microscaling reading: E4M3/E5M2 or packed E2M1
elements, one E8M0 scale per 32 K of every row of A and column of B.

Bit-exact cases use small-integer elements and scales 2^-3 .. 2^0: every
scaled product is a multiple of 2^-6 of magnitude <= 9, so every FP32
partial sum is exact (for K < 29,000) and the GPU must equal the oracle bit
for bit whatever the accumulation order. Scales that differ per row, per
column and per 32-block make a misplaced scale show up as a wrong value.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from oracle import tolerance
import workloads

pytestmark = pytest.mark.gpu

ELEM = {"mxfp8": "e4m3", "mxfp8_e5m2": "e5m2", "mxfp4": "e2m1"}
OUT = {"f16": torch.float16, "bf16": torch.bfloat16, "f32": torch.float32}


@pytest.fixture(scope="module")
def dtg():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import dense_tiled_gemm_gb300 as mod
    torch.cuda.set_device(0)
    mod.gemm_last_device_status()
    return mod


def run_mx(dtg, A, B, SFA, SFB, K, dtype_out, options=None):
    C = dtg.gemm_mx(A.cuda(), B.cuda(), SFA.cuda(), SFB.cuda(), K=K, out_dtype=OUT[dtype_out],
                    options=options)
    status, detail = dtg.gemm_last_device_status()
    assert status == dtg.GEMM_OK, f"device status {dtg.gemm_status_string(status)} site {detail:#x}"
    return C


def reference(A, B, SFA, SFB, M, N, K, mx, rows=None):
    return oracle.gemm_ref_mx(workloads.as_bits(A), workloads.as_bits(B), SFA.numpy(), SFB.numpy(),
                              M, N, K, ELEM[mx], rows=rows)


def exact_case(dtg, M, N, K, mx, options=None, seed=0, rows=None):
    A, B, SFA, SFB = workloads.make_mx_operands(M, N, K, mx, ("int", -3, 3), seed, scale_range=0)
    g = torch.Generator().manual_seed(1000 + seed)
    SFA = torch.randint(124, 128, SFA.shape, generator=g).to(torch.uint8)
    SFB = torch.randint(124, 128, SFB.shape, generator=g).to(torch.uint8)
    C = run_mx(dtg, A, B, SFA, SFB, K, "f32", options)
    C_ref, _ = reference(A, B, SFA, SFB, M, N, K, mx, rows)
    got = C.cpu().numpy().astype(np.float64)
    if rows is not None:
        got = got[rows]
    bad = np.argwhere(got != C_ref)
    assert bad.size == 0, (f"{len(bad)} inexact elements, first {tuple(bad[0])}: gpu {got[tuple(bad[0])]} "
                           f"ref {C_ref[tuple(bad[0])]}")


def bound_case(dtg, M, N, K, mx, dtype_out="bf16", options=None, seed=0, dist=("normal", 1.0)):
    A, B, SFA, SFB = workloads.make_mx_operands(M, N, K, mx, dist, seed)
    C = run_mx(dtg, A, B, SFA, SFB, K, dtype_out, options)
    C_ref, C_abs = reference(A, B, SFA, SFB, M, N, K, mx)
    ok, ratio, n_bad, first = tolerance.check(C.float().cpu().numpy().astype(np.float64), C_ref, C_abs,
                                              dtype_out)
    assert ok, f"{n_bad} out of bound (worst {ratio:.3g}) first {first}"


MX = ["mxfp8", "mxfp4"]


# ---------------------------------------------------------------- one tile, one stage
@pytest.mark.parametrize("mx", MX)
def test_unit_scales_single_stage(dtg, mx):
    A, B, SFA, SFB = workloads.make_mx_operands(256, 224, 256, mx, ("int", -3, 3), 1, scale_range=0)
    C = run_mx(dtg, A, B, SFA, SFB, 256, "f32")
    C_ref, _ = reference(A, B, SFA, SFB, 256, 224, 256, mx)
    assert np.array_equal(C.cpu().numpy().astype(np.float64), C_ref)


@pytest.mark.parametrize("mx", MX)
def test_scales_single_tile(dtg, mx):
    exact_case(dtg, 256, 224, 512, mx, seed=2)


@pytest.mark.parametrize("mx", MX + ["mxfp8_e5m2"])
def test_multi_stage_integer_exact(dtg, mx):
    exact_case(dtg, 512, 448, 2048, mx, seed=3)


# ---------------------------------------------------------------- tails and schedules
@pytest.mark.parametrize("mx", MX)
@pytest.mark.parametrize("shape", [(300, 500, 700), (129, 97, 33), (1, 1, 1), (257, 225, 100), (64, 640, 1000)],
                         ids=lambda s: "x".join(map(str, s)))
def test_ragged_integer_exact(dtg, mx, shape):
    exact_case(dtg, *shape, mx, seed=sum(shape))


@pytest.mark.parametrize("mx", MX)
@pytest.mark.parametrize("opts", [{"stream_k": 2, "max_clusters": 3}, {"stream_k": 2, "max_clusters": 8},
                                  {"stream_k": 1, "max_clusters": 1}],
                         ids=["sk3", "sk8", "one_pair"])
def test_schedules_integer_exact(dtg, mx, opts):
    exact_case(dtg, 700, 900, 3000, mx, options=opts, seed=4)


# ---------------------------------------------------------------- rounding bound, output types
@pytest.mark.parametrize("mx", MX)
@pytest.mark.parametrize("dtype_out", ["bf16", "f16", "f32"])
def test_normal_data_bound(dtg, mx, dtype_out):
    bound_case(dtg, 384, 640, 1536, mx, dtype_out, seed=5, dist=("normal", 2.0 if mx == "mxfp4" else 1.0))


# ---------------------------------------------------------------- the pages' shape, sampled
@pytest.mark.parametrize("name", ["gemm_4096x4096x65536_mxfp8", "gemm_4096x4096x65536_mxfp4"])
def test_workload_sampled(dtg, name):
    w = workloads.WORKLOADS[name]
    A, B, SFA, SFB = workloads.workload_operands(w)
    C = run_mx(dtg, A, B, SFA, SFB, w.K, w.dtype_out)
    rows = workloads.sample_rows(w.M, 12, w.seed)
    C_ref, C_abs = reference(A, B, SFA, SFB, w.M, w.N, w.K, w.dtype_in, rows=rows)
    ok, ratio, n_bad, first = tolerance.check(C.float().cpu().numpy().astype(np.float64)[rows], C_ref, C_abs,
                                              w.dtype_out)
    assert ok, f"{n_bad} out of bound (worst {ratio:.3g}) first {first}"


# ---------------------------------------------------------------- both MXFP4 stage depths
@pytest.mark.parametrize("shape", [(512, 448, 2048), (300, 500, 700), (257, 225, 100)],
                         ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("k_stage", [256, 512], ids=["one_slab", "two_slabs"])
def test_mxfp4_stage_depths_integer_exact(dtg, shape, k_stage):
    """Packed FP4 runs one-slab (256 K) stages by default and two-slab stages on
    request; each slab's scales go to the next of two TMEM buffers beside the
    accumulators. Both must match the oracle bit for bit."""
    plan = dtg.gemm_plan(*shape, dtype_in=torch.uint8, dtype_out=torch.float32, block_scaled=True,
                         options={"k_stage": k_stage})
    assert plan["block_n"] == 224 and plan["block_k"] == k_stage
    exact_case(dtg, *shape, "mxfp4", options={"k_stage": k_stage}, seed=sum(shape) + k_stage)


@pytest.mark.parametrize("shape", [(512, 448, 1024), (300, 500, 700), (257, 225, 100)],
                         ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("k_stage", [128, 256], ids=["one_slab", "two_slabs"])
def test_mxfp8_stage_depths_integer_exact(dtg, shape, k_stage):
    """MXFP8 stages hold one 128-K slab (one scale group per stage) or two; both
    must match the oracle bit for bit, ragged K included."""
    plan = dtg.gemm_plan(*shape, dtype_in=torch.float8_e4m3fn, dtype_out=torch.float32, block_scaled=True,
                         options={"k_stage": k_stage})
    assert plan["block_n"] == 224 and plan["block_k"] == k_stage
    exact_case(dtg, *shape, "mxfp8", options={"k_stage": k_stage}, seed=sum(shape) + k_stage)
