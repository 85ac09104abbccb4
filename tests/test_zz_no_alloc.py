"""gemm_no_alloc: the allocation-free entry point, checked through the C ABI.

Some callers cannot allocate device memory: a serving runtime whose own pool
already owns the GPU's memory, or a latency-critical loop in which cudaMalloc
or cudaFree could stall the device or fail. gemm_no_alloc serves them by
putting re-pitched operands into a fixed device array instead of newly
allocated scratch. These tests give it inputs that need that scratch and
require the same result as gemm, within the parity tolerance, on two
different calls in a row. The second call runs while the array still holds
the first call's data. The file is named so that pytest collects it last.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from oracle import tolerance
import workloads

pytestmark = pytest.mark.gpu

OUT = {"f16": (torch.float16, 0), "bf16": (torch.bfloat16, 1), "f32": (torch.float32, 2)}
IN = {"f16": 0, "bf16": 1}
LAYOUT = {"k": 0, "mn": 1}


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(0)
    from dense_tiled_gemm_gb300 import binding
    return binding.lib


def _call(fn, A, B, C, M, N, K, din, dout, layout_b):
    stream = torch.cuda.current_stream().cuda_stream
    return fn(A.data_ptr(), B.data_ptr(), C.data_ptr(), M, N, K, IN[din], OUT[dout][1], 0,
              LAYOUT[layout_b], stream)


def test_no_alloc_matches_gemm_on_two_calls_in_a_row(lib):
    # Both shapes need re-pitched operands (K*2 or N*2 bytes not a multiple of 16).
    cases = [(300, 333, 2050, "bf16", "f32", "k", 21),
             (257, 129, 1001, "f16", "f16", "mn", 22)]
    for M, N, K, din, dout, layout_b, seed in cases:
        A, B = workloads.make_operands(M, N, K, din, layout_b, ("uniform", -2.0, 2.0), seed)
        Ad, Bd = A.cuda(), B.cuda()
        C_gemm = torch.empty((M, N), dtype=OUT[dout][0], device="cuda")
        C_new = torch.full((M, N), float("nan"), dtype=OUT[dout][0], device="cuda")
        assert _call(lib.gemm, Ad, Bd, C_gemm, M, N, K, din, dout, layout_b) == 0
        assert _call(lib.gemm_no_alloc, Ad, Bd, C_new, M, N, K, din, dout, layout_b) == 0
        torch.cuda.synchronize()
        import ctypes
        detail = ctypes.c_uint32(0)
        assert lib.gemm_last_device_status(None, ctypes.byref(detail)) == 0
        Bkn = B.double() if layout_b == "mn" else B.double().T
        C_abs = (A.double().abs() @ Bkn.abs()).numpy()
        ref = C_gemm.double().cpu().numpy()
        ok, ratio, n_bad, first = tolerance.check(C_new.double().cpu().numpy(), ref, C_abs, dout)
        assert ok, f"{n_bad} elements differ beyond the bound, first {first}"
        # and directly against the FP64 oracle, so that a fault in the re-pitch copy
        # that both entry points share cannot pass unnoticed
        C_ref, C_ref_abs = oracle.gemm_ref(workloads.as_bits(A), workloads.as_bits(B), M, N, K, din, layout_b)
        ok, ratio, n_bad, first = tolerance.check(C_new.double().cpu().numpy(), C_ref, C_ref_abs, dout)
        assert ok, f"{n_bad} elements out of the oracle's bound, first {first}"


def test_no_alloc_rejects_operands_beyond_its_array(lib):
    # Padded A alone needs 8200 x 2112 x 2 bytes (rows padded to 128-byte multiples)
    # > 32 MiB: refused before any launch.
    M, N, K = 8200, 64, 2050
    A = torch.zeros((M, K), dtype=torch.bfloat16, device="cuda")
    B = torch.zeros((N, K), dtype=torch.bfloat16, device="cuda")
    C = torch.zeros((M, N), dtype=torch.float32, device="cuda")
    assert _call(lib.gemm_no_alloc, A, B, C, M, N, K, "bf16", "f32", "k") == 2   # UNSUPPORTED
    torch.cuda.synchronize()
    assert torch.count_nonzero(C).item() == 0


def test_no_alloc_stream_k_workspace(lib):
    """Stream-K partial sums go into the fixed array after the re-pitched copies.
    3000 x 5000 x 2050 (A re-pitched, 12.7 MB; partials ~20 MB) fits: same plan and
    the same bits as gemm. 4000 x 5000 x 2050 (A re-pitched, 16.9 MB) leaves no room
    for the partials: the call keeps every tile whole and stays within the bound."""
    import ctypes
    import dense_tiled_gemm_gb300 as dtg
    for M, fits in ((3000, True), (4000, False)):
        N, K = 5000, 2050
        assert dtg.gemm_plan(M, N, K, dtype_in=torch.bfloat16, dtype_out=torch.float32,
                             layout_b="mn")["sk_tiles"] > 0
        A, B = workloads.make_operands(M, N, K, "bf16", "mn", ("uniform", -2.0, 2.0), 40 + M)
        Ad, Bd = A.cuda(), B.cuda()
        C_gemm = torch.empty((M, N), dtype=torch.float32, device="cuda")
        C_new = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
        assert _call(lib.gemm, Ad, Bd, C_gemm, M, N, K, "bf16", "f32", "mn") == 0
        assert _call(lib.gemm_no_alloc, Ad, Bd, C_new, M, N, K, "bf16", "f32", "mn") == 0
        torch.cuda.synchronize()
        detail = ctypes.c_uint32(0)
        assert lib.gemm_last_device_status(None, ctypes.byref(detail)) == 0
        if fits:
            assert torch.equal(C_new, C_gemm)
        else:
            C_abs = (A.double().abs() @ B.double().abs()).numpy()
            ok, ratio, n_bad, first = tolerance.check(C_new.double().cpu().numpy(),
                                                      C_gemm.double().cpu().numpy(), C_abs, "f32")
            assert ok, f"{n_bad} elements differ beyond the bound, first {first}"


class _DeviceBytes:
    """A raw device range as a CUDA array, so that torch can view it without a copy."""

    def __init__(self, ptr: int, n: int):
        self.__cuda_array_interface__ = {"shape": (n,), "typestr": "|u1", "data": (ptr, False), "version": 3}


def _used_bytes(plan, M, N, K, layout_b, eb=2):
    """The part of the array a call uses, from the layout gemm.h documents: the padded
    copies (row bytes rounded up to 128), A then B, each from a 256-byte boundary,
    then the stream-K workspace."""
    up = lambda v, m: -(-v // m) * m
    a_bytes = M * up(K * eb, 128) if plan["realign_a"] else 0
    b_rows, b_cols = (K, N) if layout_b == "mn" else (N, K)
    b_off = up(a_bytes, 256)
    b_bytes = b_rows * up(b_cols * eb, 128) if plan["realign_b"] else 0
    if plan["sk_tiles"]:
        return up(b_off + b_bytes, 256) + plan["workspace_bytes"]
    return b_off + b_bytes


@pytest.mark.parametrize("M,N,K,layout_b,opts_sk", [(3000, 5000, 2050, "mn", True), (1000, 1000, 1090, "k", False)],
                         ids=["repitched_a_stream_k", "repitched_a_and_b"])
def test_no_alloc_writes_only_the_used_part_of_its_array(lib, M, N, K, layout_b, opts_sk):
    """The fixed array, viewed through gemm_no_alloc_scratch and filled with a pattern:
    a call writes inside the part its plan uses and leaves every byte after it as it was."""
    import dense_tiled_gemm_gb300 as dtg
    ptr, size = dtg.gemm_no_alloc_scratch()
    assert ptr != 0 and size == 32 * 1024 * 1024
    arr = torch.as_tensor(_DeviceBytes(ptr, size), device="cuda")
    plan = dtg.gemm_plan(M, N, K, dtype_in=torch.bfloat16, dtype_out=torch.float32, layout_b=layout_b)
    assert plan["realign_a"] == 1 and (plan["sk_tiles"] > 0) == opts_sk
    used = _used_bytes(plan, M, N, K, layout_b)
    assert 0 < used <= size
    A, B = workloads.make_operands(M, N, K, "bf16", layout_b, ("uniform", -2.0, 2.0), 60 + M)
    C = torch.empty((M, N), dtype=torch.float32, device="cuda")
    Ad, Bd = A.cuda(), B.cuda()
    torch.cuda.synchronize()
    arr.fill_(0xA5)
    torch.cuda.synchronize()
    assert _call(lib.gemm_no_alloc, Ad, Bd, C, M, N, K, "bf16", "f32", layout_b) == 0
    torch.cuda.synchronize()
    assert bool((arr[used:] == 0xA5).all()), "a write past the used part of the array"
    assert not bool((arr[:used] == 0xA5).all()), "the used part was not written"
    rows = workloads.sample_rows(M, 16, M)
    C_ref, C_abs = oracle.gemm_ref(workloads.as_bits(A), workloads.as_bits(B), M, N, K, "bf16", layout_b, rows=rows)
    ok, ratio, n_bad, first = tolerance.check(C.cpu().numpy().astype(np.float64)[rows], C_ref, C_abs, "f32")
    assert ok, f"{n_bad} out of bound (worst {ratio:.3g}) first {first}"


def test_no_alloc_scratch_rejects_null_outputs(lib):
    import ctypes
    size = ctypes.c_size_t(0)
    assert lib.gemm_no_alloc_scratch(None, ctypes.byref(size)) == 1      # GEMM_ERR_INVALID_ARG
    ptr = ctypes.c_void_p(0)
    assert lib.gemm_no_alloc_scratch(ctypes.byref(ptr), None) == 1
