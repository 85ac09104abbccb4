"""The per-device launch cache, the clock trace and the re-pitch copy, on the GPU.

A repeated call must reuse its plan and tensor maps and give the same bits
as a call made with an empty cache; a call whose pointer or shape differs
must miss. The clock trace must report a plausible SM clock. The re-pitch
copy must be exact for every source alignment it meets (word widths 1 to 16
bytes).
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
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


def _ops(M, N, K, dtype_in="f16", layout_b="k", seed=0):
    A, B = workloads.make_operands(M, N, K, dtype_in, layout_b, ("normal", 1.0), seed)
    return A.cuda(), B.cuda()


def _delta(dtg, before):
    now = dtg.gemm_cache_stats()
    return {k: now[k] - before[k] for k in now}


@pytest.mark.parametrize("shape,layout_b", [((256, 256, 256), "k"), ((4096, 4096, 8192), "k"),
                                            ((3000, 5000, 2050), "mn"), ((1000, 999, 257), "k")],
                         ids=["c1", "headline", "ragged_repitch", "direct_store"])
def test_repeat_call_hits_and_matches_fresh(dtg, shape, layout_b):
    M, N, K = shape
    A, B = _ops(M, N, K, "bf16" if layout_b == "mn" else "f16", layout_b, seed=M)
    out = torch.float32 if layout_b == "mn" else torch.float16
    dtg.gemm_cache_clear()
    before = dtg.gemm_cache_stats()
    C_fresh = dtg.gemm(A, B, layout_b=layout_b, out_dtype=out)
    d = _delta(dtg, before)
    assert d["plan_misses"] == 1 and d["map_misses"] == 1 and d["plan_hits"] == 0 and d["map_hits"] == 0
    C = torch.empty_like(C_fresh)
    dtg.gemm(A, B, C, layout_b=layout_b)         # a new C: the plan hits, the maps are new
    for _ in range(3):
        C.fill_(float("nan"))
        before = dtg.gemm_cache_stats()
        dtg.gemm(A, B, C, layout_b=layout_b)
        d = _delta(dtg, before)
        assert d["plan_hits"] == 1 and d["plan_misses"] == 0
        # a re-pitched operand lives in the stream's scratch buffer, which stays put
        # once a call of this size has grown it
        assert d["map_hits"] == 1 and d["map_misses"] == 0
        torch.cuda.synchronize()
        assert torch.equal(C.view(torch.uint8), C_fresh.view(torch.uint8))
    assert dtg.gemm_last_device_status() == (dtg.GEMM_OK, 0)


def test_repeat_call_with_same_c_hits_the_maps(dtg):
    A, B = _ops(512, 768, 640, seed=3)
    C = torch.empty(512, 768, dtype=torch.float16, device="cuda")
    dtg.gemm(A, B, C)
    before = dtg.gemm_cache_stats()
    for _ in range(5):
        dtg.gemm(A, B, C)
    d = _delta(dtg, before)
    assert d == {"plan_hits": 5, "plan_misses": 0, "map_hits": 5, "map_misses": 0}


def test_changed_pointer_or_shape_misses(dtg):
    A, B = _ops(512, 768, 640, seed=4)
    C = torch.empty(512, 768, dtype=torch.float16, device="cuda")
    dtg.gemm(A, B, C)
    ref = C.clone()
    # another C: same plan, new tensor maps
    C2 = torch.empty_like(C)
    before = dtg.gemm_cache_stats()
    dtg.gemm(A, B, C2)
    d = _delta(dtg, before)
    assert d["plan_hits"] == 1 and d["map_misses"] == 1 and d["map_hits"] == 0
    torch.cuda.synchronize()
    assert torch.equal(C2, ref)
    # another A with the same contents at a new address
    A2 = A.clone()
    before = dtg.gemm_cache_stats()
    dtg.gemm(A2, B, C2)
    d = _delta(dtg, before)
    assert d["map_misses"] == 1 and d["map_hits"] == 0
    torch.cuda.synchronize()
    assert torch.equal(C2, ref)
    # a smaller M over the same buffers: a new plan and new maps, and the rows match
    before = dtg.gemm_cache_stats()
    C3 = dtg.gemm(A[:384], B)
    d = _delta(dtg, before)
    assert d["plan_misses"] == 1 and d["map_misses"] == 1
    torch.cuda.synchronize()
    assert torch.equal(C3, ref[:384])
    # a changed option: a new plan
    before = dtg.gemm_cache_stats()
    C4 = dtg.gemm(A, B, options={"cta_group": 1})
    d = _delta(dtg, before)
    assert d["plan_misses"] == 1
    exact = workloads.make_operands(512, 768, 640, "f16", "k", ("int", -3, 3), 5)
    Ai, Bi = exact[0].cuda(), exact[1].cuda()
    Ci1 = dtg.gemm(Ai, Bi, out_dtype=torch.float32, options={"cta_group": 1})
    Ci2 = dtg.gemm(Ai, Bi, out_dtype=torch.float32)
    assert torch.equal(Ci1, Ci2)
    assert C4.shape == ref.shape


def test_cache_survives_more_shapes_than_entries(dtg):
    """More distinct calls than cache entries: old entries are replaced, and every
    call still gives the oracle's exact result."""
    n = 40
    for i in range(n):
        M, N, K = 64 + 8 * i, 96 + 16 * (i % 5), 64 + 64 * (i % 3)
        A, B = workloads.make_operands(M, N, K, "f16", "k", ("int", -3, 3), 100 + i)
        C = dtg.gemm(A.cuda(), B.cuda(), out_dtype=torch.float32)
        if i % 8 == 0:
            C_ref, _ = oracle.gemm_ref(workloads.as_bits(A), workloads.as_bits(B), M, N, K, "f16", "k")
            assert np.array_equal(C.cpu().numpy().astype(np.float64), C_ref)
    assert dtg.gemm_last_device_status() == (dtg.GEMM_OK, 0)


def test_release_workspace_empties_the_cache(dtg):
    A, B = _ops(256, 256, 256, seed=6)
    C = dtg.gemm(A, B)
    dtg.gemm(A, B, C)
    dtg.gemm_release_workspace()
    before = dtg.gemm_cache_stats()
    dtg.gemm(A, B, C)
    d = _delta(dtg, before)
    assert d["plan_misses"] == 1 and d["map_misses"] == 1


@pytest.mark.parametrize("shape", [(4096, 4096, 8192), (256, 256, 256)], ids=["headline", "c1"])
def test_clock_trace_reports_the_sm_clock(dtg, shape):
    M, N, K = shape
    A, B = _ops(M, N, K, seed=7)
    trace = torch.zeros(4, dtype=torch.int64, device="cuda")
    o = dtg.GemmOptions()
    o.clock_trace = trace.data_ptr()
    C = dtg.gemm(A, B, options=o)
    ref = dtg.gemm(A, B)
    torch.cuda.synchronize()
    assert torch.equal(C, ref)                     # the trace does not change the result
    n0, c0, n1, c1 = trace.cpu().tolist()
    assert n1 > n0 > 0 and c1 > c0 > 0
    # %globaltimer advances in steps, so a launch of a few microseconds has its
    # interval only to within about a microsecond: bound the clock both ways with that
    dn, dc = n1 - n0, c1 - c0
    assert dc / (dn + 1000) * 1e3 < 2500.0, (dc, dn)
    assert dn <= 1000 or dc / (dn - 1000) * 1e3 > 300.0, (dc, dn)
    assert dn < 50e6                               # one launch, well under 50 ms


# Source offsets (elements) and K: the re-pitch copy's word width is the widest
# power of two dividing the source base and the row length in bytes.
REPITCH = [(0, 2050, "bf16", 4), (1, 2050, "bf16", 2), (0, 2052, "bf16", 8), (4, 2052, "bf16", 8),
           (0, 2049, "e4m3", 1), (1, 2056, "e4m3", 1), (2, 2050, "e4m3", 2), (0, 2060, "e4m3", 4),
           (8, 2056, "e4m3", 8), (1, 2048, "f16", 2), (4, 2048, "f16", 8), (8, 2048, "f16", 16)]


@pytest.mark.parametrize("offset,K,dtype_in,width", REPITCH,
                         ids=[f"off{o}_K{k}_{d}_w{w}" for o, k, d, w in REPITCH])
def test_repitch_copy_every_word_width(dtg, offset, K, dtype_in, width):
    """A placed `offset` elements into a larger buffer (so its base is misaligned
    when offset*esize is not a multiple of 16), and K chosen so its rows are
    not 16-byte multiples: the copy runs with `width`-byte words, and the
    product is exact on small integers."""
    M, N = 333, 200
    A, B = workloads.make_operands(M, N, K, dtype_in, "k", ("int", -3, 3), offset + K)
    esize = A.element_size()
    align = (offset * esize) | (K * esize)        # the buffer itself starts 256-byte aligned
    assert min(16, align & -align) == width
    bits = torch.uint8 if esize == 1 else torch.int16
    flat = torch.zeros(M * K + offset + 64, dtype=bits, device="cuda")
    flat[offset:offset + M * K] = A.view(bits).reshape(-1).cuda()
    Ad = flat[offset:offset + M * K].view(A.dtype).view(M, K)
    plan = dtg.gemm_plan(M, N, K, dtype_in=A.dtype, dtype_out=torch.float32, a_ptr=Ad.data_ptr(),
                         b_ptr=B.cuda().data_ptr())
    assert plan["realign_a"] == (1 if width < 16 else 0)
    C = dtg.gemm(Ad, B.cuda(), out_dtype=torch.float32)
    C_ref, _ = oracle.gemm_ref(workloads.as_bits(A), workloads.as_bits(B), M, N, K, dtype_in, "k")
    got = C.cpu().numpy().astype(np.float64)
    bad = np.argwhere(got != C_ref)
    assert bad.size == 0, f"{len(bad)} inexact elements, first {tuple(bad[0])}"


def _exact_inputs(M, N, K, seed):
    A, B = workloads.make_operands(M, N, K, "f16", "k", ("int", -3, 3), seed)
    C_ref, _ = oracle.gemm_ref(workloads.as_bits(A), workloads.as_bits(B), M, N, K, "f16", "k")
    A, B = A.cuda(), B.cuda()
    torch.cuda.synchronize()      # the side streams below do not wait for the default stream's uploads
    return A, B, C_ref


def test_stream_scratch_many_streams(dtg):
    """Re-pitched operands and stream-K partial sums on ten streams at once: eight
    streams keep a scratch buffer of their own, the other two take per-call scratch.
    Three calls per stream are queued before anything is waited for; every result
    is exact, and again after the buffers are released."""
    M, N, K = 640, 896, 1090          # K * 2 bytes not a multiple of 16: A and B re-pitched
    cases = [_exact_inputs(M, N, K, 200 + i) for i in range(10)]
    streams = [torch.cuda.Stream() for _ in range(10)]
    for rnd in range(2):
        outs = []
        for rep in range(3):
            for (A, B, _), st in zip(cases, streams):
                with torch.cuda.stream(st):
                    C = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
                    dtg.gemm(A, B, C, stream=st, options={"stream_k": 2})
                    outs.append(C)
        torch.cuda.synchronize()
        for j, C in enumerate(outs):
            ref = cases[j % 10][2]
            assert np.array_equal(C.cpu().numpy().astype(np.float64), ref), (rnd, j)
        assert dtg.gemm_last_device_status() == (dtg.GEMM_OK, 0)
        dtg.gemm_release_workspace()


def test_stream_scratch_grows(dtg):
    """One stream: a small re-pitched call, a larger one (its scratch buffer grows,
    the old one freed in stream order behind the first call), and the small one
    again, queued back to back; all exact."""
    st = torch.cuda.Stream()
    small = _exact_inputs(300, 333, 258, 210)
    large = _exact_inputs(2000, 3000, 1026, 211)
    outs = []
    with torch.cuda.stream(st):
        for (A, B, ref), opts in ((small, {"stream_k": 2}), (large, {"stream_k": 2}), (small, None)):
            outs.append((dtg.gemm(A, B, out_dtype=torch.float32, stream=st, options=opts), ref))
    torch.cuda.synchronize()
    for C, ref in outs:
        assert np.array_equal(C.cpu().numpy().astype(np.float64), ref)
    assert dtg.gemm_last_device_status() == (dtg.GEMM_OK, 0)


def test_default_stream_is_torchs_current(dtg):
    """With no stream given, a call goes to torch's current stream of A's device, also
    inside a torch.cuda.stream context."""
    s = torch.cuda.Stream()
    assert dtg._stream_ptr(None) == torch.cuda.current_stream().cuda_stream
    with torch.cuda.stream(s):
        assert dtg._stream_ptr(None) == s.cuda_stream
        assert dtg._stream_ptr(None, torch.cuda.current_device()) == s.cuda_stream
        A, B = _ops(384, 256, 320, seed=9)
        C = dtg.gemm(A, B)
    s.synchronize()
    ref = dtg.gemm(A, B)
    torch.cuda.synchronize()
    assert torch.equal(C, ref)
