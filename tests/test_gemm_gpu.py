"""Parity of the CUDA GEMM against the FP64 CPU oracle, through the C ABI.

Every comparison is element by element. Floating-point inputs must meet
|C - C_ref| <= 2e-3 * sum_k |a*b| + 1e-6 + ulp_out(|C_ref|). Small-integer
inputs make every FP32 partial sum exact, so the GPU must match the oracle
bit for bit there. The workloads are checked whole at the exact launch
configuration the benchmark uses, except 16384^3, which is checked on sampled
whole rows.

Tests run in order from a single tile upwards, so a run that stops at the
first failure stops on the simplest failing case.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from oracle import tolerance
import workloads

pytestmark = pytest.mark.gpu

TORCH_DT = {"f16": torch.float16, "bf16": torch.bfloat16, "f32": torch.float32}


@pytest.fixture(scope="module")
def dtg():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import dense_tiled_gemm_gb300 as mod
    torch.cuda.set_device(0)
    mod.gemm_last_device_status()   # clear anything left by an earlier process
    return mod


def run_gpu(dtg, A, B, layout_b, dtype_out, options=None):
    C = dtg.gemm(A.cuda(), B.cuda(), layout_b=layout_b, out_dtype=TORCH_DT[dtype_out],
                 options=options)
    status, detail = dtg.gemm_last_device_status()
    assert status == dtg.GEMM_OK, f"device status {dtg.gemm_status_string(status)} site {detail:#x}"
    return C


def compare(C, A, B, M, N, K, dtype_in, dtype_out, layout_b, rows=None):
    C_ref, C_abs = oracle.gemm_ref(workloads.as_bits(A), workloads.as_bits(B), M, N, K, dtype_in,
                                   layout_b, rows=rows)
    got = C.float().cpu().numpy().astype(np.float64)
    if rows is not None:
        got = got[rows]
    ok, ratio, n_bad, first = tolerance.check(got, C_ref, C_abs, dtype_out)
    assert ok, (f"{n_bad} elements out of bound (worst error/bound {ratio:.3g}); first {first}: "
                f"gpu {got[first]} ref {C_ref[first]}")
    return ratio


def case(dtg, M, N, K, dtype_in="f16", dtype_out="f32", layout_b="k", dist=("uniform", -1.0, 1.0),
         seed=0, options=None, rows=None):
    A, B = workloads.make_operands(M, N, K, dtype_in, layout_b, dist, seed)
    C = run_gpu(dtg, A, B, layout_b, dtype_out, options)
    return compare(C, A, B, M, N, K, dtype_in, dtype_out, layout_b, rows)


def exact_case(dtg, M, N, K, dtype_in, layout_b, options=None, seed=0, rows=None):
    """Small integers in [-3, 3]: FP32 output must equal the oracle bit for bit."""
    A, B = workloads.make_operands(M, N, K, dtype_in, layout_b, ("int", -3, 3), seed)
    C = run_gpu(dtg, A, B, layout_b, "f32", options)
    C_ref, _ = oracle.gemm_ref(workloads.as_bits(A), workloads.as_bits(B), M, N, K, dtype_in,
                               layout_b, rows=rows)
    got = C.cpu().numpy().astype(np.float64)
    if rows is not None:
        got = got[rows]
    bad = np.argwhere(got != C_ref)
    assert bad.size == 0, f"{len(bad)} inexact elements, first {tuple(bad[0])}"


CG1 = {"cta_group": 1}
CG2 = {"cta_group": 2}


# ---------------------------------------------------------------- one tile
def test_single_tile_cta1(dtg):
    case(dtg, 128, 256, 64, options=CG1)


def test_single_tile_cta1_integer(dtg):
    exact_case(dtg, 128, 256, 64, "f16", "k", options=CG1)


def test_multi_kblock_cta1(dtg):
    exact_case(dtg, 128, 256, 640, "f16", "k", options=CG1)


def test_single_tile_cta2(dtg):
    case(dtg, 256, 256, 64, options=CG2)


def test_multi_kblock_cta2_integer(dtg):
    exact_case(dtg, 256, 256, 640, "f16", "k", options=CG2)


# ---------------------------------------------------------------- layouts and types
@pytest.mark.parametrize("opts", [CG1, CG2], ids=["cta1", "cta2"])
@pytest.mark.parametrize("dtype_in", ["f16", "bf16"])
@pytest.mark.parametrize("layout_b", ["k", "mn"])
def test_integer_exact(dtg, opts, dtype_in, layout_b):
    exact_case(dtg, 512, 512, 1024, dtype_in, layout_b, options=opts, seed=3)


@pytest.mark.parametrize("dtype_out", ["f16", "bf16", "f32"])
@pytest.mark.parametrize("opts", [CG1, CG2, {"cta_group": 2, "block_n": 224}],
                         ids=["cta1", "cta2", "cta2_n224"])
def test_output_types(dtg, dtype_out, opts):
    case(dtg, 384, 640, 320, "bf16" if dtype_out == "bf16" else "f16", dtype_out, "k",
         ("normal", 1.0), 5, options=opts)


# ---------------------------------------------------------------- persistent loop
@pytest.mark.parametrize("opts", [{"cta_group": 1, "max_clusters": 1},
                                  {"cta_group": 2, "max_clusters": 1},
                                  {"cta_group": 2, "max_clusters": 3, "group_m": 2},
                                  {"cta_group": 2, "block_n": 224, "max_clusters": 2}],
                         ids=["cta1_one", "cta2_one", "cta2_three", "cta2_n224_two"])
def test_many_tiles_per_cta(dtg, opts):
    """A handful of CTAs walk many tiles: ring and accumulator phases wrap many times."""
    exact_case(dtg, 1024, 1024, 448, "f16", "k", options=opts, seed=4)


# ---------------------------------------------------------------- narrow single-CTA tiles
NARROW = [{"cta_group": 1, "block_n": 128}, {"cta_group": 1, "block_n": 64}]
NARROW_IDS = ["cta1_n128", "cta1_n64"]


@pytest.mark.parametrize("opts", NARROW, ids=NARROW_IDS)
@pytest.mark.parametrize("dtype_in", ["f16", "bf16"])
@pytest.mark.parametrize("layout_b", ["k", "mn"])
def test_narrow_integer_exact(dtg, opts, dtype_in, layout_b):
    exact_case(dtg, 512, 512, 1024, dtype_in, layout_b, options=opts, seed=3)


@pytest.mark.parametrize("opts", NARROW, ids=NARROW_IDS)
@pytest.mark.parametrize("shape", [(1, 1, 1), (129, 130, 65), (300, 70, 1000), (1000, 999, 257)],
                         ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("layout_b", ["k", "mn"])
def test_narrow_ragged(dtg, opts, shape, layout_b):
    M, N, K = shape
    case(dtg, M, N, K, "bf16", "f32", layout_b, ("uniform", -2.0, 2.0), seed=M + N + K, options=opts)


@pytest.mark.parametrize("dtype_out", ["f16", "bf16"])
@pytest.mark.parametrize("opts", NARROW, ids=NARROW_IDS)
def test_narrow_16bit_out(dtg, dtype_out, opts):
    case(dtg, 384, 640, 320, "bf16" if dtype_out == "bf16" else "f16", dtype_out, "k",
         ("normal", 1.0), 5, options=opts)


@pytest.mark.parametrize("opts", [dict(NARROW[0], stream_k=2), dict(NARROW[1], stream_k=2),
                                  dict(NARROW[0], max_clusters=3), dict(NARROW[1], max_clusters=5, group_m=2)],
                         ids=["cta1_n128_sk", "cta1_n64_sk", "cta1_n128_three", "cta1_n64_five"])
def test_narrow_stream_k_and_many_tiles(dtg, opts):
    """Stream-K splits and a handful of CTAs walking many narrow tiles."""
    exact_case(dtg, 1024, 1024, 448, "f16", "k", options=opts, seed=4)


# ---------------------------------------------------------------- epilogue warps
EPI = [({"epilogue_warps": 8, "stream_k": 2}, "k"), ({"epilogue_warps": 4, "stream_k": 2}, "k"),
       ({"epilogue_warps": 8, "block_n": 224, "stream_k": 2}, "k"),
       ({"epilogue_warps": 8, "cta_group": 1, "block_n": 64, "stream_k": 2}, "k"),
       ({"epilogue_warps": 8, "cta_group": 1, "block_n": 256, "max_clusters": 3}, "mn"),
       ({"epilogue_warps": 8, "max_clusters": 3, "group_m": 2}, "mn"),
       ({"epilogue_warps": 4, "cta_group": 1, "block_n": 128}, "k")]


@pytest.mark.parametrize("opts,layout_b", EPI, ids=["cta2_8_sk", "cta2_4_sk", "n224_8_sk", "cta1_n64_8_sk",
                                                    "cta1_8_three", "cta2_8_three", "cta1_n128_4"])
def test_epilogue_warps_integer_exact(dtg, opts, layout_b):
    """Four and eight epilogue warps: stream-K flags and partial chunks per warp,
    an odd chunk count split 4/3, and accumulator phases wrapping over many tiles."""
    exact_case(dtg, 1024, 1024, 448, "f16", layout_b, options=opts, seed=6)


@pytest.mark.parametrize("dtype_out", ["f16", "bf16", "f32"])
@pytest.mark.parametrize("warps", [4, 8])
def test_epilogue_warps_output_types(dtg, dtype_out, warps):
    """One (FP32) or two (16-bit) staging buffers per warp with eight warps, and a
    ragged tile edge."""
    case(dtg, 300, 700, 320, "bf16" if dtype_out == "bf16" else "f16", dtype_out, "k",
         ("normal", 1.0), 8, options={"epilogue_warps": warps})


def test_planner_epilogue_warps(dtg):
    """Eight warps where a CTA's work is at most two tiles, or four with a 16-bit C;
    four where main loops dominate or C is FP32."""
    assert dtg.gemm_plan(2048, 2048, 2048)["epilogue_warps"] == 8
    assert dtg.gemm_plan(1024, 1024, 1024)["epilogue_warps"] == 8
    assert dtg.gemm_plan(4096, 4096, 8192)["epilogue_warps"] == 8
    assert dtg.gemm_plan(8192, 8192, 8192)["epilogue_warps"] == 4
    assert dtg.gemm_plan(3000, 5000, 2050, dtype_in=torch.bfloat16, dtype_out=torch.float32,
                         layout_b="mn")["epilogue_warps"] == 4
    assert dtg.gemm_plan(2048, 2048, 2048, options={"epilogue_warps": 4})["epilogue_warps"] == 4


# ---------------------------------------------------------------- 128-deep ring stages
K128 = [{"cta_group": 2, "k_stage": 128}, {"cta_group": 2, "block_n": 224, "k_stage": 128},
        {"cta_group": 1, "k_stage": 128}, {"cta_group": 2, "k_stage": 128, "max_clusters": 2}]


@pytest.mark.parametrize("opts", K128, ids=["cta2", "cta2_n224", "cta1", "cta2_two_pairs"])
@pytest.mark.parametrize("layout_b", ["k", "mn"])
@pytest.mark.parametrize("K", [960, 1000, 64])
def test_k_stage_128_integer_exact(dtg, opts, layout_b, K):
    """Two 64-wide K slabs per stage. K = 960 leaves the last stage's second slab
    wholly past K (its MMAs are skipped); K = 1000 leaves it partly filled."""
    if layout_b == "mn" and opts.get("block_n") == 224:
        pytest.skip("224-wide tiles need a K-major B")
    exact_case(dtg, 640, 512, K, "f16", layout_b, options=opts, seed=K)


def test_k_stage_128_workload(dtg):
    w = workloads.WORKLOADS["gemm_4096x4096x8192_f16"]
    A, B = workloads.workload_operands(w)
    C = run_gpu(dtg, A, B, w.layout_b, w.dtype_out, options={"k_stage": 128})
    compare(C, A, B, w.M, w.N, w.K, w.dtype_in, w.dtype_out, w.layout_b,
            rows=workloads.sample_rows(w.M, 32, w.seed))


# ---------------------------------------------------------------- ragged shapes
RAGGED = [
    (1, 1, 1), (7, 9, 3), (127, 129, 65), (129, 127, 63), (255, 257, 200), (300, 500, 130),
    (1, 300, 64), (300, 1, 64), (64, 64, 1), (130, 70, 1000), (513, 1000, 77),
]


@pytest.mark.parametrize("shape", RAGGED, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("layout_b", ["k", "mn"])
def test_ragged(dtg, shape, layout_b):
    M, N, K = shape
    case(dtg, M, N, K, "bf16", "f32", layout_b, ("uniform", -2.0, 2.0), seed=M + N + K)


@pytest.mark.parametrize("shape", [(257, 300, 131), (1000, 999, 257)], ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("dtype_out", ["f16", "bf16"])
def test_ragged_16bit_out(dtg, shape, dtype_out):
    M, N, K = shape
    case(dtg, M, N, K, "f16" if dtype_out == "f16" else "bf16", dtype_out, "k", ("normal", 1.0), seed=K)


def test_ragged_integer_all_paths(dtg):
    """K not a multiple of 8 (operand re-pitch) and N odd (direct stores), exact."""
    exact_case(dtg, 300, 333, 2050, "bf16", "mn", seed=6)
    exact_case(dtg, 300, 333, 2050, "f16", "k", seed=7)


# ---------------------------------------------------------------- closed forms
@pytest.mark.parametrize("dtype_in", ["f16", "bf16"])
def test_identity_returns_a(dtg, dtype_in):
    M, K = 300, 512
    A, _ = workloads.make_operands(M, K, K, dtype_in, "k", ("normal", 1.0), 8)
    eye = torch.eye(K, dtype=TORCH_DT[dtype_in])
    C16 = run_gpu(dtg, A, eye, "k", dtype_in)
    assert torch.equal(C16.cpu().view(torch.int16), A.view(torch.int16))
    C32 = run_gpu(dtg, A, eye, "mn", "f32")
    assert torch.equal(C32.cpu(), A.float())


def test_all_ones_gives_column_sums(dtg):
    M, N, K = 256, 384, 1000
    _, B = workloads.make_operands(M, N, K, "f16", "mn", ("uniform", -1.0, 1.0), 9)
    A = torch.ones(M, K, dtype=torch.float16)
    C = run_gpu(dtg, A, B, "mn", "f32")
    colsum = B.double().sum(0).numpy()
    err = np.abs(C.cpu().double().numpy() - colsum[None, :])
    assert np.all(err <= 2e-3 * B.double().abs().sum(0).numpy()[None, :] + 1e-6)


def test_rank_one(dtg):
    # u_i and v_j have at most 5 significant bits, so every partial sum m*u_i*v_j
    # (m <= K = 512) needs at most 19 bits and is exact in FP32: C = K*u_i*v_j.
    M, N, K = 200, 300, 512
    u = torch.tensor([((i % 17) - 8) / 8 for i in range(M)], dtype=torch.float16)
    v = torch.tensor([((j % 33) - 16) / 4 for j in range(N)], dtype=torch.float16)
    A = u[:, None].expand(M, K).contiguous()
    B = v[:, None].expand(N, K).contiguous()       # K-major B: b[k][j] = v_j
    C = run_gpu(dtg, A, B, "k", "f32")
    expect = K * np.outer(u.double().numpy(), v.double().numpy())
    assert np.array_equal(C.cpu().double().numpy(), expect)


# ---------------------------------------------------------------- the workloads at full size
def _full_size(dtg, name, n_rows):
    w = workloads.WORKLOADS[name]
    A, B = workloads.workload_operands(w)
    C = run_gpu(dtg, A, B, w.layout_b, w.dtype_out)      # the benchmark's launch (automatic plan)
    rows = workloads.sample_rows(w.M, n_rows, w.seed)
    return compare(C, A, B, w.M, w.N, w.K, w.dtype_in, w.dtype_out, w.layout_b, rows=rows)


def test_workload_256_full(dtg):
    w = workloads.WORKLOADS["gemm_256_f16_f32"]
    A, B = workloads.workload_operands(w)
    C = run_gpu(dtg, A, B, w.layout_b, w.dtype_out)
    compare(C, A, B, w.M, w.N, w.K, w.dtype_in, w.dtype_out, w.layout_b)


def test_workload_ragged_full(dtg):
    w = workloads.WORKLOADS["gemm_3000x5000x2050_bf16_f32_bmn"]
    A, B = workloads.workload_operands(w)
    C = run_gpu(dtg, A, B, w.layout_b, w.dtype_out)
    compare(C, A, B, w.M, w.N, w.K, w.dtype_in, w.dtype_out, w.layout_b)


@pytest.mark.parametrize("name", ["gemm_4096x4096x8192_f16", "gemm_8192_bf16", "square_f16_1024",
                                  "square_f16_2048", "square_f16_4096", "square_f16_8192"])
def test_workload_full(dtg, name):
    """Every element of the workload, at the benchmark's launch, against the oracle
    (the 8192^3 cases take the oracle about 25 s on 16 host cores)."""
    w = workloads.WORKLOADS[name]
    A, B = workloads.workload_operands(w)
    C = run_gpu(dtg, A, B, w.layout_b, w.dtype_out)
    compare(C, A, B, w.M, w.N, w.K, w.dtype_in, w.dtype_out, w.layout_b)


@pytest.mark.parametrize("name,n_rows", [("square_f16_16384", 16)])
def test_workload_sampled(dtg, name, n_rows):
    """Sampled: 16384^3 (8.8e12 flop) would take the oracle minutes; whole rows at
    every 128-row tile edge plus seeded random rows are checked."""
    _full_size(dtg, name, n_rows)


def test_headline_shape_integer_exact(dtg):
    """The 4096 x 4096 x 8192 launch on small integers: every element bit-exact."""
    exact_case(dtg, 4096, 4096, 8192, "f16", "k", seed=12)


@pytest.mark.parametrize("N", [32776, 32769], ids=["tma_store", "direct_store"])
def test_output_beyond_int32_elements(dtg, N):
    """C with more than 2^31 elements (4.3 GB of FP16): row offsets past the
    32-bit range, through the TMA store (pitch a multiple of 16 bytes) and
    through the direct store (odd N). Sampled rows, first and last included,
    are bit-exact on small integers."""
    M, K = 65573, 72
    assert M * N > 2**31
    A, B = workloads.make_operands(M, N, K, "f16", "k", ("int", -3, 3), 21)
    C = run_gpu(dtg, A, B, "k", "f16")
    plan = dtg.gemm_plan(M, N, K, dtype_in=torch.float16, dtype_out=torch.float16)
    assert plan["direct_store"] == (1 if N % 8 else 0)
    rows = sorted(set([0, 1, M // 2, M - 2, M - 1] + list(workloads.sample_rows(M, 8, 21))))
    got = C[torch.tensor(rows, device=C.device)].float().cpu().numpy().astype(np.float64)
    del C
    C_ref, _ = oracle.gemm_ref(workloads.as_bits(A), workloads.as_bits(B), M, N, K, "f16", "k", rows=rows)
    bad = np.argwhere(got != C_ref)
    assert bad.size == 0, f"{len(bad)} inexact elements, first {tuple(bad[0])}"


# ---------------------------------------------------------------- other entry points
def test_from_host_matches_device(dtg):
    A, B = workloads.make_operands(700, 900, 600, "f16", "k", ("normal", 1.0), 13)
    C_dev = run_gpu(dtg, A, B, "k", "f16")
    C_host = dtg.gemm_from_host(A, B, out_dtype=torch.float16)
    assert torch.equal(C_host.view(torch.int16), C_dev.cpu().view(torch.int16))
    dtg.gemm_release_workspace()


def test_from_host_async_overlapping_calls(dtg):
    """Five asynchronous host calls in flight at once, of three sizes (the two staging
    slots grow while the other slot is still busy), each with its own pinned inputs and
    output: after one synchronisation every C equals the device-side gemm bit for bit."""
    shapes = [(300, 400, 500), (700, 900, 600), (300, 400, 500), (1000, 520, 777), (64, 64, 64)]
    cases = []
    for i, (M, N, K) in enumerate(shapes):
        A, B = workloads.make_operands(M, N, K, "bf16", "k", ("normal", 1.0), 40 + i)
        Ah, Bh = A.pin_memory(), B.pin_memory()
        Ch = torch.full((M, N), float("nan"), dtype=torch.float32).pin_memory()
        dtg.gemm_from_host_async(Ah, Bh, Ch, out_dtype=torch.float32)
        cases.append((A, B, Ch))
    torch.cuda.synchronize()
    for A, B, Ch in cases:
        C_dev = run_gpu(dtg, A, B, "k", "f32")
        assert torch.equal(Ch, C_dev.cpu())
    status, detail = dtg.gemm_last_device_status()
    assert status == dtg.GEMM_OK
    dtg.gemm_release_workspace()


def test_plan_reports_launch(dtg):
    p = dtg.gemm_plan(4096, 4096, 8192)
    assert p["cta_group"] == 2 and p["block_k"] == 128 and p["num_sms"] > 0
    assert p["grid_ctas"] % 2 == 0 and p["realign_a"] == 0 and p["direct_store"] == 0
    q = dtg.gemm_plan(3000, 5000, 2050, dtype_in=torch.bfloat16, dtype_out=torch.float32,
                      layout_b="mn")
    assert q["realign_a"] == 1 and q["realign_b"] == 0 and q["direct_store"] == 0


def test_launch_count_counts_kernels(dtg):
    before = dtg.gemm_launch_count()
    A, B = workloads.make_operands(256, 256, 256, "f16", "k", ("normal", 1.0), 14)
    run_gpu(dtg, A, B, "k", "f16")
    assert dtg.gemm_launch_count() == before + 1
    A2, B2 = workloads.make_operands(256, 256, 250, "f16", "k", ("normal", 1.0), 15)
    run_gpu(dtg, A2, B2, "k", "f16")       # K*2 bytes not a multiple of 16: two copies + GEMM
    assert dtg.gemm_launch_count() == before + 4


def test_wait_timeout_is_reported_not_hung(dtg):
    """A bounded wait on a barrier nothing arrives at ends and is reported."""
    dtg.gemm_selftest_wait_timeout(50)
    status, detail = dtg.gemm_last_device_status()
    assert status == dtg.GEMM_ERR_TIMEOUT and detail == 0x307
    assert dtg.gemm_last_device_status() == (dtg.GEMM_OK, 0)     # read clears it
    case(dtg, 256, 256, 256)                                      # the context is still usable
