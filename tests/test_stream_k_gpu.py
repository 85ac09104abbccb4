"""Parity of stream-K tail scheduling against the FP64 CPU oracle.

`stream_k = 2` forces the last tiles to be split along K; `max_clusters`
shrinks the grid so that the splits fall in many places: two-way splits
(at least one full wave of stream-K tiles) and many-way splits (fewer
tiles than units, so a tile's owner adds several writers' partial sums).
Small-integer inputs make every FP32 partial sum exact, so the split result
must equal the oracle bit for bit however the K range was cut.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from oracle import tolerance
import workloads

pytestmark = pytest.mark.gpu

TORCH_DT = {"f16": torch.float16, "bf16": torch.bfloat16, "f32": torch.float32,
            "e4m3": torch.float8_e4m3fn, "e5m2": torch.float8_e5m2}


@pytest.fixture(scope="module")
def dtg():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import dense_tiled_gemm_gb300 as mod
    torch.cuda.set_device(0)
    mod.gemm_last_device_status()
    return mod


def run_gpu(dtg, A, B, layout_b, dtype_out, options):
    C = dtg.gemm(A.cuda(), B.cuda(), layout_b=layout_b, out_dtype=TORCH_DT[dtype_out], options=options)
    status, detail = dtg.gemm_last_device_status()
    assert status == dtg.GEMM_OK, f"device status {dtg.gemm_status_string(status)} site {detail:#x}"
    return C


def exact_case(dtg, M, N, K, dtype_in, layout_b, options, seed):
    A, B = workloads.make_operands(M, N, K, dtype_in, layout_b, ("int", -3, 3), seed)
    C = run_gpu(dtg, A, B, layout_b, "f32", options)
    C_ref, _ = oracle.gemm_ref(workloads.as_bits(A), workloads.as_bits(B), M, N, K, dtype_in, layout_b)
    bad = np.argwhere(C.cpu().numpy().astype(np.float64) != C_ref)
    assert bad.size == 0, f"{len(bad)} inexact elements, first {tuple(bad[0])}"


def bound_case(dtg, M, N, K, dtype_in, dtype_out, layout_b, options, seed, dist=("normal", 1.0)):
    A, B = workloads.make_operands(M, N, K, dtype_in, layout_b, dist, seed)
    C = run_gpu(dtg, A, B, layout_b, dtype_out, options)
    C_ref, C_abs = oracle.gemm_ref(workloads.as_bits(A), workloads.as_bits(B), M, N, K, dtype_in, layout_b)
    ok, ratio, n_bad, first = tolerance.check(C.float().cpu().numpy().astype(np.float64), C_ref, C_abs,
                                              dtype_out)
    assert ok, f"{n_bad} out of bound (worst {ratio:.3g}) first {first}"
    return C


def sk(cg, units, **kw):
    return {"cta_group": cg, "stream_k": 2, "max_clusters": units, **kw}


# 640 x 512 in 256 x 256 pair tiles = 6 tiles; in 128 x 256 single tiles = 10 tiles
@pytest.mark.parametrize("units", [2, 4, 5, 8, 13])
@pytest.mark.parametrize("K", [2048, 1000, 130, 64])
def test_pairs_integer_exact(dtg, units, K):
    exact_case(dtg, 640, 512, K, "f16", "k", sk(2, units), seed=units * 7 + K)


@pytest.mark.parametrize("units", [3, 4, 7, 16, 25])
@pytest.mark.parametrize("K", [2048, 777])
def test_single_cta_integer_exact(dtg, units, K):
    exact_case(dtg, 640, 512, K, "bf16", "k", sk(1, units), seed=units + K)


@pytest.mark.parametrize("units", [4, 9])
def test_n224_and_mn_layout(dtg, units):
    exact_case(dtg, 700, 900, 1500, "bf16", "k", sk(2, units, block_n=224), seed=units)
    exact_case(dtg, 700, 900, 1500, "f16", "mn", sk(2, units), seed=units + 1)


@pytest.mark.parametrize("dtype_in", ["e4m3", "e5m2"])
@pytest.mark.parametrize("units", [3, 8])
def test_fp8_integer_exact(dtg, dtype_in, units):
    exact_case(dtg, 640, 512, 3000, dtype_in, "k", sk(2, units), seed=units)


@pytest.mark.parametrize("dtype_out", ["f16", "bf16", "f32"])
def test_output_types_and_direct_store(dtg, dtype_out):
    # N = 333 is odd: C rows are not 16-byte multiples, so the owner stores directly
    din = "bf16" if dtype_out == "bf16" else "f16"
    bound_case(dtg, 520, 333, 2050, din, dtype_out, "k", sk(2, 5), seed=3)
    bound_case(dtg, 520, 512, 2050, din, dtype_out, "k", sk(2, 5), seed=4)


def test_repeatable_bits(dtg):
    A, B = workloads.make_operands(900, 1100, 3000, "f16", "k", ("normal", 1.0), 21)
    opts = sk(2, 7)
    C1 = run_gpu(dtg, A, B, "k", "f32", opts)
    C2 = run_gpu(dtg, A, B, "k", "f32", opts)
    assert torch.equal(C1, C2)


def test_planner_picks_stream_k_for_ragged_workload(dtg):
    w = workloads.WORKLOADS["gemm_3000x5000x2050_bf16_f32_bmn"]
    p = dtg.gemm_plan(w.M, w.N, w.K, dtype_in=torch.bfloat16, dtype_out=torch.float32, layout_b="mn")
    assert p["sk_tiles"] > 0 and p["workspace_bytes"] > 0
    off = dtg.gemm_plan(w.M, w.N, w.K, dtype_in=torch.bfloat16, dtype_out=torch.float32, layout_b="mn",
                        options={"stream_k": 1})
    assert off["sk_tiles"] == 0 and off["workspace_bytes"] == 0
    # forced stream-K on 304 tiles: the data-parallel part is whole waves of the units
    on = dtg.gemm_plan(4096, 4096, 8192, options={"stream_k": 2, "block_n": 224})
    units = on["grid_ctas"] // 2
    assert on["sk_tiles"] > 0 and (on["num_tiles"] - on["sk_tiles"]) % units == 0


def test_ragged_workload_both_schedules(dtg):
    """The 3000 x 5000 x 2050 workload (automatic plan: stream-K) and the same
    problem kept data-parallel: both within the bound, sampled rows."""
    w = workloads.WORKLOADS["gemm_3000x5000x2050_bf16_f32_bmn"]
    A, B = workloads.workload_operands(w)
    rows = workloads.sample_rows(w.M, 64, w.seed)
    C_ref, C_abs = oracle.gemm_ref(workloads.as_bits(A), workloads.as_bits(B), w.M, w.N, w.K, w.dtype_in,
                                   w.layout_b, rows=rows)
    for opts in (None, {"stream_k": 1}):
        C = dtg.gemm(A.cuda(), B.cuda(), layout_b=w.layout_b, out_dtype=torch.float32, options=opts)
        assert dtg.gemm_last_device_status() == (dtg.GEMM_OK, 0)
        ok, ratio, n_bad, first = tolerance.check(C.cpu().numpy().astype(np.float64)[rows], C_ref, C_abs,
                                                  "f32")
        assert ok, f"{opts}: {n_bad} out of bound (worst {ratio:.3g}) first {first}"


def test_ragged_workload_integer_exact_auto_plan(dtg):
    exact_case(dtg, 3000, 5000, 2050, "bf16", "mn", None, seed=31)


def test_large_split_k(dtg):
    """Few tiles and a long K (1024 x 1024 x 16384): the planner splits each tile
    several ways; sampled rows against the oracle."""
    p = dtg.gemm_plan(1024, 1024, 16384)
    assert p["sk_tiles"] > 0
    bound_case(dtg, 1024, 1024, 16384, "f16", "f32", "k", None, seed=5)
