"""Parity of the FP8 (E4M3 / E5M2) GEMM against the FP64 CPU oracle.

The FP8 form follows "Porting High-Performance HIP Kernels to FlyDSL"
(section "A More Complex Kernel"): E4M3 operands, identity block scales and
FP32 accumulation, so the oracle's plain definition applies unchanged with
its FP8 decoders. The same bar as the 16-bit path holds:
|C - C_ref| <= 2e-3 * sum_k |a*b| + 1e-6 + ulp_out(|C_ref|), and bit-exact
FP32 output on small-integer inputs (every FP32 partial sum is exact).

A slab of FP8 K is 128 elements (one 128-byte swizzle row), so the K tails
here sit at multiples of 128 and 256 rather than 64 and 128.
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
FP8 = ["e4m3", "e5m2"]


@pytest.fixture(scope="module")
def dtg():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import dense_tiled_gemm_gb300 as mod
    torch.cuda.set_device(0)
    mod.gemm_last_device_status()
    return mod


def run_gpu(dtg, A, B, dtype_out, options=None):
    C = dtg.gemm(A.cuda(), B.cuda(), layout_b="k", out_dtype=TORCH_DT[dtype_out], options=options)
    status, detail = dtg.gemm_last_device_status()
    assert status == dtg.GEMM_OK, f"device status {dtg.gemm_status_string(status)} site {detail:#x}"
    return C


def compare(C, A, B, M, N, K, dtype_in, dtype_out, rows=None):
    C_ref, C_abs = oracle.gemm_ref(workloads.as_bits(A), workloads.as_bits(B), M, N, K, dtype_in,
                                   "k", rows=rows)
    got = C.float().cpu().numpy().astype(np.float64)
    if rows is not None:
        got = got[rows]
    ok, ratio, n_bad, first = tolerance.check(got, C_ref, C_abs, dtype_out)
    assert ok, (f"{n_bad} elements out of bound (worst error/bound {ratio:.3g}); first {first}: "
                f"gpu {got[first]} ref {C_ref[first]}")


def case(dtg, M, N, K, dtype_in="e4m3", dtype_out="bf16", dist=("normal", 1.0), seed=0,
         options=None):
    A, B = workloads.make_operands(M, N, K, dtype_in, "k", dist, seed)
    C = run_gpu(dtg, A, B, dtype_out, options)
    compare(C, A, B, M, N, K, dtype_in, dtype_out)


def exact_case(dtg, M, N, K, dtype_in, options=None, seed=0, rows=None):
    A, B = workloads.make_operands(M, N, K, dtype_in, "k", ("int", -3, 3), seed)
    C = run_gpu(dtg, A, B, "f32", options)
    C_ref, _ = oracle.gemm_ref(workloads.as_bits(A), workloads.as_bits(B), M, N, K, dtype_in, "k",
                               rows=rows)
    got = C.cpu().numpy().astype(np.float64)
    if rows is not None:
        got = got[rows]
    bad = np.argwhere(got != C_ref)
    assert bad.size == 0, f"{len(bad)} inexact elements, first {tuple(bad[0])}"


CG1 = {"cta_group": 1}
CG2 = {"cta_group": 2}


# ---------------------------------------------------------------- one tile
@pytest.mark.parametrize("dtype_in", FP8)
@pytest.mark.parametrize("opts,M", [(CG1, 128), (CG2, 256)], ids=["cta1", "cta2"])
def test_single_tile_integer(dtg, dtype_in, opts, M):
    exact_case(dtg, M, 256, 128, dtype_in, options=opts)


@pytest.mark.parametrize("dtype_in", FP8)
@pytest.mark.parametrize("opts,M", [(CG1, 128), (CG2, 256)], ids=["cta1", "cta2"])
def test_multi_kblock_integer(dtg, dtype_in, opts, M):
    exact_case(dtg, M, 256, 1280, dtype_in, options=opts, seed=1)


@pytest.mark.parametrize("opts", [CG1, CG2], ids=["cta1", "cta2"])
def test_single_tile_normal(dtg, opts):
    case(dtg, 128 * opts["cta_group"], 256, 128, options=opts)


# ---------------------------------------------------------------- ring depths and K tails
STAGES = [{"cta_group": 2, "k_stage": 128}, {"cta_group": 2, "k_stage": 256},
          {"cta_group": 2, "block_n": 224, "k_stage": 256}, {"cta_group": 1, "k_stage": 128},
          {"cta_group": 1, "k_stage": 256}, {"cta_group": 2, "k_stage": 256, "max_clusters": 2}]


@pytest.mark.parametrize("opts", STAGES, ids=["cta2_k128", "cta2_k256", "cta2_n224_k256",
                                              "cta1_k128", "cta1_k256", "cta2_k256_two_pairs"])
@pytest.mark.parametrize("K", [1920, 2000, 128, 96, 16])
def test_k_stage_integer_exact(dtg, opts, K):
    """K = 1920 leaves the last 256-deep stage's second slab wholly past K (its
    MMAs are skipped); 2000 leaves it partly filled; 96 and 16 are single
    partial slabs (96 bytes per row is not a multiple of 16: A and B are
    re-pitched first)."""
    exact_case(dtg, 640, 512, K, "e4m3", options=opts, seed=K)


# ---------------------------------------------------------------- output types, many tiles
@pytest.mark.parametrize("dtype_out", ["f16", "bf16", "f32"])
@pytest.mark.parametrize("dtype_in", FP8)
@pytest.mark.parametrize("opts", [CG1, CG2, {"cta_group": 2, "block_n": 224}],
                         ids=["cta1", "cta2", "cta2_n224"])
def test_output_types(dtg, dtype_out, dtype_in, opts):
    case(dtg, 384, 640, 640, dtype_in, dtype_out, ("normal", 1.0), 5, options=opts)


@pytest.mark.parametrize("dtype_in", FP8)
@pytest.mark.parametrize("opts", [{"cta_group": 1, "block_n": 128}, {"cta_group": 1, "block_n": 64},
                                  {"cta_group": 1, "block_n": 64, "stream_k": 2}],
                         ids=["cta1_n128", "cta1_n64", "cta1_n64_sk"])
def test_narrow_integer_exact(dtg, dtype_in, opts):
    """Narrow single-CTA tiles, with K ragged at the 128-byte slab."""
    exact_case(dtg, 384, 448, 1000, dtype_in, options=opts, seed=7)


@pytest.mark.parametrize("opts", [{"cta_group": 1, "max_clusters": 1},
                                  {"cta_group": 2, "max_clusters": 1},
                                  {"cta_group": 2, "max_clusters": 3, "group_m": 2},
                                  {"cta_group": 2, "block_n": 224, "max_clusters": 2}],
                         ids=["cta1_one", "cta2_one", "cta2_three", "cta2_n224_two"])
def test_many_tiles_per_cta(dtg, opts):
    exact_case(dtg, 1024, 1024, 896, "e4m3", options=opts, seed=4)


# ---------------------------------------------------------------- ragged shapes
RAGGED = [(1, 1, 1), (7, 9, 3), (127, 129, 65), (129, 127, 200), (255, 257, 300),
          (300, 500, 130), (1, 300, 128), (300, 1, 128), (64, 64, 1), (513, 1000, 77)]


@pytest.mark.parametrize("shape", RAGGED, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("dtype_in", FP8)
def test_ragged(dtg, shape, dtype_in):
    M, N, K = shape
    case(dtg, M, N, K, dtype_in, "f32", ("uniform", -2.0, 2.0), seed=M + N + K)


def test_ragged_integer_all_paths(dtg):
    """K bytes not a multiple of 16 (operand re-pitch) and N odd (direct stores), exact."""
    exact_case(dtg, 300, 333, 2050, "e4m3", seed=6)
    exact_case(dtg, 300, 333, 2050, "e5m2", seed=7)


# ---------------------------------------------------------------- closed forms
@pytest.mark.parametrize("dtype_in", FP8)
def test_identity_returns_a(dtg, dtype_in):
    """FP8 values have at most 4 significant bits, so A·I = A is exact in BF16 and FP16."""
    M, K = 300, 512
    A, _ = workloads.make_operands(M, K, K, dtype_in, "k", ("normal", 1.0), 8)
    eye = torch.eye(K, dtype=torch.float32).to(TORCH_DT[dtype_in])
    for out in ("bf16", "f16", "f32"):
        C = run_gpu(dtg, A, eye, out)
        assert torch.equal(C.cpu(), A.to(TORCH_DT[out])), out


def test_rank_one(dtg):
    # u_i and v_j are E4M3 values with at most 4 significant bits, so every partial sum
    # m*u_i*v_j (m <= K = 1024) is exact in FP32: C = K*u_i*v_j.
    M, N, K = 200, 300, 1024
    u = torch.tensor([((i % 15) - 7) / 4 for i in range(M)]).to(torch.float8_e4m3fn)
    v = torch.tensor([((j % 31) - 15) / 8 for j in range(N)]).to(torch.float8_e4m3fn)
    A = u[:, None].expand(M, K).contiguous()
    B = v[:, None].expand(N, K).contiguous()
    C = run_gpu(dtg, A, B, "f32")
    expect = K * np.outer(u.double().numpy(), v.double().numpy())
    assert np.array_equal(C.cpu().double().numpy(), expect)


# ---------------------------------------------------------------- the FP8 workloads at full size
def test_workload_full(dtg):
    """Every element of the 8192^3 FP8 workload, at the benchmark's launch."""
    w = workloads.WORKLOADS["gemm_8192_e4m3"]
    A, B = workloads.workload_operands(w)
    C = run_gpu(dtg, A, B, w.dtype_out)      # the benchmark's launch (automatic plan)
    compare(C, A, B, w.M, w.N, w.K, w.dtype_in, w.dtype_out)


@pytest.mark.parametrize("name,n_rows", [("gemm_12288_e4m3", 16)])
def test_workload_sampled(dtg, name, n_rows):
    """Sampled: 12288^3 (3.7e12 flop) on sampled whole rows."""
    w = workloads.WORKLOADS[name]
    A, B = workloads.workload_operands(w)
    C = run_gpu(dtg, A, B, w.dtype_out)      # the benchmark's launch (automatic plan)
    rows = workloads.sample_rows(w.M, n_rows, w.seed)
    compare(C, A, B, w.M, w.N, w.K, w.dtype_in, w.dtype_out, rows=rows)


def test_fp8_workload_integer_exact(dtg):
    """The 8192^3 FP8 launch on small integers: every element bit-exact."""
    exact_case(dtg, 8192, 8192, 8192, "e4m3", seed=12)


# ---------------------------------------------------------------- entry points and limits
def test_mn_major_fp8_is_unsupported(dtg):
    A = torch.zeros(256, 256, dtype=torch.float8_e4m3fn, device="cuda")
    B = torch.zeros(256, 256, dtype=torch.float8_e4m3fn, device="cuda")
    with pytest.raises(dtg.GemmError) as exc:
        dtg.gemm(A, B, layout_b="mn")
    assert exc.value.status == dtg.binding.GEMM_ERR_UNSUPPORTED


def test_plan_fp8(dtg):
    p = dtg.gemm_plan(8192, 8192, 8192, dtype_in=torch.float8_e4m3fn, dtype_out=torch.bfloat16)
    assert p["cta_group"] == 2 and p["block_k"] == 256
    q = dtg.gemm_plan(256, 256, 100, dtype_in=torch.float8_e5m2, dtype_out=torch.float32)
    assert q["realign_a"] == 1 and q["realign_b"] == 1
    r = dtg.gemm_plan(256, 256, 112, dtype_in=torch.float8_e4m3fn, dtype_out=torch.float32)
    assert r["realign_a"] == 0 and r["realign_b"] == 0


def test_from_host_fp8(dtg):
    A, B = workloads.make_operands(700, 900, 600, "e4m3", "k", ("normal", 1.0), 13)
    C_dev = run_gpu(dtg, A, B, "bf16")
    C_host = dtg.gemm_from_host(A, B)
    assert C_host.dtype == torch.bfloat16
    assert torch.equal(C_host.view(torch.int16), C_dev.cpu().view(torch.int16))
    dtg.gemm_release_workspace()
