"""Guard bytes around every output: no kernel writes outside what it owns.

Element-wise parity cannot see a store that lands past the end of C (or
before its start). Here each output tensor sits inside a larger device buffer
with GUARD bytes of a fixed pattern on each side; after the call the pattern
must be intact and the inputs unchanged. The cases cover every write path:
the tensor-memory-access store and the direct store (odd N, misaligned base),
ragged M/N/K tails, forced stream-K (partial sums in the workspace, then the
owners' stores), MN-major B with a re-pitched A, FP8, the block-scaled
products, attention's O and log-sum-exp, and the allocation-free entry point.
This is the range check that hardware buffer descriptors give the kernels of
"Porting High-Performance HIP Kernels to FlyDSL" (section "Buffer Resource
Descriptors"), tested from the outside.
"""
from __future__ import annotations

import ctypes

import pytest
import torch

import workloads

pytestmark = pytest.mark.gpu

GUARD = 4096
PATTERN = 0xA5


@pytest.fixture(scope="module")
def dtg():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import dense_tiled_gemm_gb300 as mod
    torch.cuda.set_device(0)
    mod.gemm_last_device_status()
    return mod


class Guarded:
    """A tensor of `shape` and `dtype` placed `offset` bytes past GUARD patterned
    bytes, with GUARD patterned bytes after it."""

    def __init__(self, shape, dtype, offset=0):
        esize = torch.empty((), dtype=dtype).element_size()
        assert offset % esize == 0
        n = esize
        for s in shape:
            n *= s
        self.lo, self.hi = GUARD + offset, GUARD + offset + n
        self.buf = torch.full((self.hi + GUARD,), PATTERN, dtype=torch.uint8, device="cuda")
        self.t = self.buf[self.lo:self.hi].view(dtype).view(shape)

    def intact(self) -> bool:
        torch.cuda.synchronize()
        return bool((self.buf[:self.lo] == PATTERN).all() and (self.buf[self.hi:] == PATTERN).all())


def _bits(t):
    return t.view(torch.uint8).clone()


def _gemm_case(dtg, M, N, K, din, dout, layout_b, offset=0, options=None, seed=0):
    A, B = workloads.make_operands(M, N, K, din, layout_b, ("int", -3, 3), seed)
    Ad, Bd = A.cuda(), B.cuda()
    a0, b0 = _bits(Ad), _bits(Bd)
    g = Guarded((M, N), dout, offset)
    dtg.gemm(Ad, Bd, g.t, layout_b=layout_b, options=options)
    assert dtg.gemm_last_device_status() == (dtg.GEMM_OK, 0)
    assert g.intact(), "a store landed outside C"
    assert torch.equal(_bits(Ad), a0) and torch.equal(_bits(Bd), b0), "an input was written"
    ref = dtg.gemm(Ad, Bd, layout_b=layout_b, out_dtype=dout, options=options)
    assert torch.equal(g.t, ref)
    return dtg.gemm_plan(M, N, K, dtype_in=Ad.dtype, dtype_out=dout, layout_b=layout_b, a_ptr=Ad.data_ptr(),
                         b_ptr=Bd.data_ptr(), c_ptr=g.t.data_ptr(), options=options)


@pytest.mark.parametrize("shape,din,dout,layout_b,offset,store", [
    ((300, 512, 256), "f16", torch.float16, "k", 0, "tma"),
    ((513, 1000, 77), "bf16", torch.float32, "mn", 0, "tma"),          # ragged M, N, K; A re-pitched
    ((300, 333, 2050), "bf16", torch.float32, "mn", 0, "direct"),      # odd N
    ((257, 333, 130), "f16", torch.float16, "k", 0, "direct"),         # odd N, 16-bit stores
    ((300, 512, 256), "f16", torch.float32, "k", 4, "direct"),         # C base off 16-byte alignment
    ((256, 256, 64), "bf16", torch.bfloat16, "k", 2, "direct"),
    ((3000, 5000, 2050), "bf16", torch.float32, "mn", 0, "tma"),       # the ragged workload's launch
    ((1, 1, 1), "f16", torch.float32, "k", 0, "direct"),
], ids=["tma_f16", "ragged_tma", "odd_n_f32", "odd_n_f16", "c_offset4", "c_offset2", "ragged_workload",
        "one_element"])
def test_gemm_writes_only_c(dtg, shape, din, dout, layout_b, offset, store):
    M, N, K = shape
    plan = _gemm_case(dtg, M, N, K, din, dout, layout_b, offset, seed=M + N)
    assert plan["direct_store"] == (1 if store == "direct" else 0)


@pytest.mark.parametrize("opts", [{"stream_k": 2}, {"stream_k": 2, "cta_group": 1},
                                  {"stream_k": 2, "block_n": 224}, {"stream_k": 2, "max_clusters": 5}],
                         ids=["cta2", "cta1", "n224", "five_units"])
@pytest.mark.parametrize("shape", [(1024, 1024, 1024), (1000, 777, 1000)], ids=["square", "ragged"])
def test_stream_k_writes_only_c(dtg, opts, shape):
    M, N, K = shape
    plan = _gemm_case(dtg, M, N, K, "f16", torch.float32, "k", options=opts, seed=K)
    assert plan["sk_tiles"] > 0


@pytest.mark.parametrize("dtype_in", ["e4m3", "e5m2"])
def test_fp8_writes_only_c(dtg, dtype_in):
    _gemm_case(dtg, 300, 224, 520, dtype_in, torch.bfloat16, "k", seed=7)
    _gemm_case(dtg, 257, 301, 130, dtype_in, torch.float32, "k", seed=8)    # odd N, re-pitched A and B


@pytest.mark.parametrize("mx", ["mxfp8", "mxfp4"])
def test_mx_writes_only_c(dtg, mx):
    M, N, K = 300, 250, 1000
    A, B, SFA, SFB = workloads.make_mx_operands(M, N, K, mx, ("int", -3, 3), 9, scale_range=2)
    ins = [t.cuda() for t in (A, B, SFA, SFB)]
    before = [_bits(t) for t in ins]
    g = Guarded((M, N), torch.float32)
    dtg.gemm_mx(*ins, g.t, K=K)
    assert dtg.gemm_last_device_status() == (dtg.GEMM_OK, 0)
    assert g.intact(), "a store landed outside C"
    assert all(torch.equal(_bits(t), b) for t, b in zip(ins, before)), "an input was written"
    assert torch.equal(g.t, dtg.gemm_mx(*ins, K=K, out_dtype=torch.float32))


@pytest.mark.parametrize("causal", [False, True], ids=["full", "causal"])
@pytest.mark.parametrize("shape", [(1, 2, 300, 200), (2, 3, 1000, 777), (1, 1, 1, 129)],
                         ids=lambda s: "x".join(map(str, s)))
def test_attention_writes_only_o_and_lse(dtg, shape, causal):
    from dense_tiled_gemm_gb300 import binding
    B, H, Lq, Lk = shape
    Q, K, V = (t.cuda() for t in workloads.make_attention_operands(B, H, Lq, Lk, 128, "bf16",
                                                                    ("normal", 1.0), sum(shape)))
    before = [_bits(t) for t in (Q, K, V)]
    gO = Guarded((B, H, Lq, 128), torch.bfloat16)
    gL = Guarded((B, H, Lq), torch.float32, offset=4)
    st = torch.cuda.current_stream().cuda_stream
    rc = binding.lib.attention_fwd(Q.data_ptr(), K.data_ptr(), V.data_ptr(), gO.t.data_ptr(), gL.t.data_ptr(),
                                   B, H, Lq, Lk, 128, binding.GEMM_BF16, int(causal), 128 ** -0.5, st)
    assert rc == 0
    assert dtg.gemm_last_device_status() == (dtg.GEMM_OK, 0)
    assert gO.intact() and gL.intact(), "a store landed outside O or the log-sum-exp"
    assert all(torch.equal(_bits(t), b) for t, b in zip((Q, K, V), before)), "an input was written"
    O, lse = dtg.attention(Q, K, V, causal=causal, return_lse=True)
    assert torch.equal(gO.t, O) and torch.equal(gL.t, lse)


@pytest.mark.parametrize("shape,layout_b", [((300, 333, 2050), "k"), ((3000, 5000, 2050), "mn"),
                                            ((257, 129, 1001), "mn")], ids=["odd_n", "stream_k", "repitch_b"])
def test_no_alloc_writes_only_c(dtg, shape, layout_b):
    M, N, K = shape
    A, B = workloads.make_operands(M, N, K, "bf16", layout_b, ("int", -3, 3), M)
    Ad, Bd = A.cuda(), B.cuda()
    a0, b0 = _bits(Ad), _bits(Bd)
    g = Guarded((M, N), torch.float32)
    dtg.gemm_no_alloc(Ad, Bd, g.t, layout_b=layout_b)
    assert dtg.gemm_last_device_status() == (dtg.GEMM_OK, 0)
    assert g.intact(), "a store landed outside C"
    assert torch.equal(_bits(Ad), a0) and torch.equal(_bits(Bd), b0), "an input was written"
    assert torch.equal(g.t, dtg.gemm(Ad, Bd, layout_b=layout_b, out_dtype=torch.float32))
