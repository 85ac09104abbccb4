"""Two CTA pairs per cluster sharing their A tiles (gemm_options_t.cluster_pairs = 2).

Each cluster of four CTAs computes two tiles side by side in N; each CTA
loads half of its 128 A rows and multicasts them to the CTA with the same
row half in the other pair. Small-integer inputs make every FP32 partial sum
exact, so the result must equal the oracle bit for bit, and equal the
one-pair-per-cluster launch. The cases cover an odd number of tile columns
(the second pair of the last cluster column has no tile), ragged M/N/K with
re-pitched operands, forced stream-K, a grid small enough that every cluster
walks many tile pairs, MN-major B, FP8, and guard bytes around C.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from oracle import tolerance
import workloads

pytestmark = pytest.mark.gpu

TWO = {"cluster_pairs": 2}


@pytest.fixture(scope="module")
def dtg():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import dense_tiled_gemm_gb300 as mod
    torch.cuda.set_device(0)
    mod.gemm_last_device_status()
    return mod


def _exact(dtg, M, N, K, dtype_in="f16", layout_b="k", options=TWO, seed=0):
    A, B = workloads.make_operands(M, N, K, dtype_in, layout_b, ("int", -3, 3), seed)
    Ad, Bd = A.cuda(), B.cuda()
    C = dtg.gemm(Ad, Bd, layout_b=layout_b, out_dtype=torch.float32, options=options)
    assert dtg.gemm_last_device_status() == (dtg.GEMM_OK, 0)
    plan = dtg.gemm_plan(M, N, K, dtype_in=Ad.dtype, dtype_out=torch.float32, layout_b=layout_b,
                         a_ptr=Ad.data_ptr(), b_ptr=Bd.data_ptr(), options=options)
    assert plan["cluster_pairs"] == 2 and plan["block_n"] == 256 and plan["grid_ctas"] % 4 == 0
    C_ref, _ = oracle.gemm_ref(workloads.as_bits(A), workloads.as_bits(B), M, N, K, dtype_in, layout_b)
    got = C.cpu().numpy().astype(np.float64)
    bad = np.argwhere(got != C_ref)
    assert bad.size == 0, f"{len(bad)} inexact elements, first {tuple(bad[0])}"
    C1 = dtg.gemm(Ad, Bd, layout_b=layout_b, out_dtype=torch.float32, options={"cluster_pairs": 1})
    assert torch.equal(C, C1)
    return plan


@pytest.mark.parametrize("shape", [(256, 512, 64), (512, 512, 640), (1024, 1024, 1024), (512, 768, 512),
                                   (300, 700, 200), (1000, 999, 257), (257, 130, 1001), (1, 1, 1)],
                         ids=lambda s: "x".join(map(str, s)))
def test_shared_a_integer_exact(dtg, shape):
    """768 and 700 wide: an odd tile count in N (a phantom second tile); 130 wide:
    one tile column; 1001 and 257 K: re-pitched operands."""
    _exact(dtg, *shape, seed=sum(shape))


@pytest.mark.parametrize("opts", [{"stream_k": 2}, {"stream_k": 1}, {"max_clusters": 1}, {"max_clusters": 3},
                                  {"k_stage": 64}, {"k_stage": 64, "stream_k": 2, "max_clusters": 5}],
                         ids=["sk", "dp", "one_cluster", "three_clusters", "one_slab", "one_slab_sk5"])
def test_shared_a_schedules(dtg, opts):
    _exact(dtg, 1280, 1792, 1088, options={**TWO, **opts}, seed=11)


@pytest.mark.parametrize("layout_b", ["k", "mn"])
@pytest.mark.parametrize("dtype_in", ["f16", "bf16"])
def test_shared_a_layouts(dtg, layout_b, dtype_in):
    _exact(dtg, 768, 1280, 960, dtype_in, layout_b, seed=12)


@pytest.mark.parametrize("dtype_in", ["e4m3", "e5m2"])
def test_shared_a_fp8(dtg, dtype_in):
    _exact(dtg, 768, 1280, 1024, dtype_in, seed=13)
    _exact(dtg, 300, 700, 130, dtype_in, seed=14)


def test_shared_a_headline_tolerance(dtg):
    """The 4096 x 4096 x 8192 FP16 workload with shared A, every element against the oracle."""
    w = workloads.WORKLOADS["gemm_4096x4096x8192_f16"]
    A, B = workloads.workload_operands(w)
    C = dtg.gemm(A.cuda(), B.cuda(), options=TWO)
    assert dtg.gemm_last_device_status() == (dtg.GEMM_OK, 0)
    C_ref, C_abs = oracle.gemm_ref(workloads.as_bits(A), workloads.as_bits(B), w.M, w.N, w.K, w.dtype_in, "k")
    ok, ratio, n_bad, first = tolerance.check(C.float().cpu().numpy().astype(np.float64), C_ref, C_abs, "f16")
    assert ok, f"{n_bad} out of bound, first {first}"


def test_shared_a_writes_only_c(dtg):
    M, N, K = 1000, 999, 257
    A, B = workloads.make_operands(M, N, K, "f16", "k", ("int", -3, 3), 15)
    Ad, Bd = A.cuda(), B.cuda()
    guard = 4096
    buf = torch.full((2 * guard + M * N * 4,), 0xA5, dtype=torch.uint8, device="cuda")
    C = buf[guard:guard + M * N * 4].view(torch.float32).view(M, N)
    for opts in (TWO, {**TWO, "stream_k": 2}):
        dtg.gemm(Ad, Bd, C, options=opts)
        torch.cuda.synchronize()
        assert bool((buf[:guard] == 0xA5).all() and (buf[guard + M * N * 4:] == 0xA5).all())
        assert torch.equal(C, dtg.gemm(Ad, Bd, out_dtype=torch.float32))
