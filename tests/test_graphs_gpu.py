"""CUDA-graph capture of the library's calls.

A graph captured from gemm, gemm_mx, attention or gemm_no_alloc calls replays
them with the kernel parameters, launch ids and workspaces of the capture. The
tests change the inputs in place between replays and require, after every
replay, the bits of an eager call on the same inputs (the same plan runs both
ways, so the results are identical, stream-K partial sums included). Stream-K
owners clear the flags they consumed, so a replay never reads the previous
replay's partial sums.
"""
from __future__ import annotations

import ctypes

import pytest
import torch

import workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dtg():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import dense_tiled_gemm_gb300 as mod
    torch.cuda.set_device(0)
    mod.gemm_last_device_status()
    return mod


def status_ok(dtg):
    status, detail = dtg.gemm_last_device_status()
    assert status == dtg.GEMM_OK, f"device status {dtg.gemm_status_string(status)} site {detail:#x}"


def refill(tensors, seed):
    """New values in place (same addresses), drawn on the host from a seeded generator."""
    g = torch.Generator().manual_seed(seed)
    for t in tensors:
        if t.dtype == torch.uint8:
            t.copy_(torch.randint(0, 256, t.shape, generator=g, dtype=torch.uint8))
        else:
            t.copy_(torch.randn(t.shape, generator=g).to(t.dtype))


def capture(fn):
    fn()                       # first call outside the capture: per-device setup
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        fn()
    torch.cuda.synchronize()
    return graph


@pytest.mark.parametrize("shape,opts", [((4096, 4096, 2048), {"stream_k": 2}),
                                        ((4096, 4096, 8192), None),
                                        ((1000, 3000, 700), {"stream_k": 2, "max_clusters": 5})],
                         ids=["stream_k", "headline_plan", "ragged_stream_k"])
def test_gemm_replays_match_eager(dtg, shape, opts):
    M, N, K = shape
    plan = dtg.gemm_plan(M, N, K, options=opts)
    assert plan["sk_tiles"] > 0
    A = torch.empty(M, K, dtype=torch.float16, device="cuda")
    B = torch.empty(N, K, dtype=torch.float16, device="cuda")
    C = torch.empty(M, N, dtype=torch.float16, device="cuda")
    refill([A, B], 1)
    graph = capture(lambda: dtg.gemm(A, B, C, options=opts))
    for trial in range(3):
        refill([A, B], 10 + trial)
        C.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        status_ok(dtg)
        eager = dtg.gemm(A, B, options=opts)
        torch.cuda.synchronize()
        assert torch.equal(C.view(torch.int16), eager.view(torch.int16)), f"replay {trial}"


def test_gemm_realigned_operands_replay(dtg):
    """The ragged 3000 x 5000 x 2050 workload (A re-pitched into stream-ordered scratch,
    B N-major, FP32 out, stream-K): the scratch allocation is captured with the launch."""
    M, N, K = 3000, 5000, 2050
    assert dtg.gemm_plan(M, N, K, dtype_in=torch.bfloat16, dtype_out=torch.float32,
                         layout_b="mn")["realign_a"] == 1
    A = torch.empty(M, K, dtype=torch.bfloat16, device="cuda")
    B = torch.empty(K, N, dtype=torch.bfloat16, device="cuda")
    C = torch.empty(M, N, dtype=torch.float32, device="cuda")
    refill([A, B], 2)
    graph = capture(lambda: dtg.gemm(A, B, C, layout_b="mn", out_dtype=torch.float32))
    for trial in range(2):
        refill([A, B], 20 + trial)
        C.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        status_ok(dtg)
        eager = dtg.gemm(A, B, layout_b="mn", out_dtype=torch.float32)
        assert torch.equal(C, eager), f"replay {trial}"


@pytest.mark.parametrize("mx", ["mxfp8", "mxfp4"])
def test_gemm_mx_replays_match_eager(dtg, mx):
    M, N, K = 512, 448, 2048
    A, B, SFA, SFB = [t.cuda() for t in workloads.make_mx_operands(M, N, K, mx, ("normal", 1.0), 3)]
    C = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    graph = capture(lambda: dtg.gemm_mx(A, B, SFA, SFB, C, K=K))
    for trial in range(2):
        A2, B2, SFA2, SFB2 = workloads.make_mx_operands(M, N, K, mx, ("normal", 1.0), 30 + trial)
        for dst, src in ((A, A2), (B, B2), (SFA, SFA2), (SFB, SFB2)):
            dst.copy_(src)
        C.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        status_ok(dtg)
        eager = dtg.gemm_mx(A, B, SFA, SFB, K=K)
        assert torch.equal(C.view(torch.int16), eager.view(torch.int16)), f"replay {trial}"


@pytest.mark.parametrize("causal", [False, True], ids=["full", "causal"])
def test_attention_replays_match_eager(dtg, causal):
    Bt, H, L, d = 2, 3, 1000, 128
    Q, K, V = [torch.empty(Bt, H, L, d, dtype=torch.bfloat16, device="cuda") for _ in range(3)]
    O = torch.empty_like(Q)
    refill([Q, K, V], 4)
    graph = capture(lambda: dtg.attention(Q, K, V, causal=causal, O=O))
    for trial in range(2):
        refill([Q, K, V], 40 + trial)
        O.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        status_ok(dtg)
        eager = dtg.attention(Q, K, V, causal=causal)
        assert torch.equal(O.view(torch.int16), eager.view(torch.int16)), f"replay {trial}"


def test_no_alloc_stream_k_replays(dtg):
    """gemm_no_alloc keeps its re-pitched operands and stream-K partials in one fixed
    device array: a graph of it allocates nothing, and its replays reuse that array."""
    from dense_tiled_gemm_gb300 import binding
    M, N, K = 3000, 5000, 2050
    A = torch.empty(M, K, dtype=torch.bfloat16, device="cuda")
    B = torch.empty(K, N, dtype=torch.bfloat16, device="cuda")
    C = torch.empty(M, N, dtype=torch.float32, device="cuda")
    refill([A, B], 5)

    def call():
        rc = binding.lib.gemm_no_alloc(A.data_ptr(), B.data_ptr(), C.data_ptr(), M, N, K, 1, 2, 0, 1,
                                       torch.cuda.current_stream().cuda_stream)
        assert rc == 0

    graph = capture(call)
    for trial in range(2):
        refill([A, B], 50 + trial)
        C.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        detail = ctypes.c_uint32(0)
        assert binding.lib.gemm_last_device_status(None, ctypes.byref(detail)) == 0
        eager = dtg.gemm(A, B, layout_b="mn", out_dtype=torch.float32)
        assert torch.equal(C, eager), f"replay {trial}"
