"""Dense tiled GEMM for GB300 (sm_103a): C = A·B with FP16/BF16 or FP8
(E4M3/E5M2) operands, FP32 accumulation and a cast-on-store epilogue.

Every function here has the name of a C-ABI entry point in include/gemm.h and
only marshals arguments: torch tensors become device pointers and sizes, and
torch's current stream is passed as the CUDA stream. The GEMM runs in the
library's own kernels (``libdtgemm.so``). Importing this package fails when
that library is not built, and every error status is raised as GemmError.
"""
from __future__ import annotations

import ctypes

import torch

from . import binding
from .binding import (GEMM_BF16, GEMM_E2M1, GEMM_E4M3, GEMM_E5M2, GEMM_F16, GEMM_F32, GEMM_K_MAJOR,
                      GEMM_MN_MAJOR, GEMM_OK, GEMM_ERR_TIMEOUT, GEMM_JOB_FULL, GEMM_JOB_OWNER,
                      GEMM_JOB_WRITER, GemmError, GemmJob, GemmOptions, GemmPlan, STATUS_NAMES)

__all__ = ["gemm", "gemm_ex", "gemm_mx", "attention", "gemm_plan", "gemm_from_host", "gemm_from_host_async",
           "gemm_release_workspace", "gemm_cache_stats", "gemm_cache_clear", "gemm_selftest_withheld_load",
           "gemm_last_device_status", "gemm_selftest_wait_timeout", "gemm_status_string", "gemm_no_alloc_scratch",
           "gemm_launch_count", "gemm_schedule_jobs", "GemmError", "GemmOptions", "GemmPlan"]

_DT_IN = {torch.float16: GEMM_F16, torch.bfloat16: GEMM_BF16,
          torch.float8_e4m3fn: GEMM_E4M3, torch.float8_e5m2: GEMM_E5M2}
_FP8 = (torch.float8_e4m3fn, torch.float8_e5m2)
_DT_OUT = {torch.float16: GEMM_F16, torch.bfloat16: GEMM_BF16, torch.float32: GEMM_F32}
_LAYOUT = {"k": GEMM_K_MAJOR, "mn": GEMM_MN_MAJOR}


# torch's current stream of a device as a raw cudaStream_t, without building a
# Stream object (about 0.2 us against 2.9 us for current_stream().cuda_stream on
# the GB300 host); the public call where a torch build lacks it
_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream_ptr(stream, dev: int | None = None) -> int:
    if stream is None:
        if _raw_stream is not None:
            return _raw_stream(torch.cuda.current_device() if dev is None else dev)
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _options(options) -> GemmOptions | None:
    if options is None or isinstance(options, GemmOptions):
        return options
    o = GemmOptions()
    for key, val in dict(options).items():
        setattr(o, key, int(val))
    return o


def _check(status: int, what: str):
    if status != GEMM_OK:
        raise GemmError(status, what)


def _prepare(A, B, C, layout_b, out_dtype, device_kind):
    """Check A, B (and C, or allocate it) for a GEMM on `device_kind` tensors.
    Returns M, N, K, C and the input type code. Type errors come first."""
    adt, bdt = A.dtype, B.dtype
    din = _DT_IN.get(adt)
    if din is None or bdt not in _DT_IN:
        name, t = ("A", A) if din is None else ("B", B)
        raise TypeError(f"{name} must be float16, bfloat16, float8_e4m3fn or float8_e5m2, got {t.dtype}")
    if adt != bdt:
        raise TypeError("A and B must have the same dtype")
    want_cuda = device_kind == "cuda"
    if not (A.is_contiguous() and B.is_contiguous()):
        raise ValueError("A and B must be contiguous")
    if A.is_cuda != want_cuda or B.is_cuda != want_cuda:
        raise ValueError(f"A and B must be {device_kind} tensors")
    sa, sb = A.shape, B.shape
    if len(sa) != 2 or len(sb) != 2:
        raise ValueError("A and B must be 2-D")
    M, K = sa
    if layout_b == "k":
        N, Kb = sb
    elif layout_b == "mn":
        Kb, N = sb
    else:
        raise ValueError("layout_b must be 'k' (B is N x K) or 'mn' (B is K x N)")
    if Kb != K:
        raise ValueError(f"K mismatch: A has {K}, B has {Kb}")
    if C is None:
        default_out = torch.bfloat16 if adt in _FP8 else adt
        C = torch.empty((M, N), dtype=out_dtype or default_out, device=A.device,
                        pin_memory=(not want_cuda and torch.cuda.is_available()))
    else:
        sc = C.shape
        if C.dtype not in _DT_OUT or len(sc) != 2 or sc[0] != M or sc[1] != N or not C.is_contiguous():
            raise ValueError("C must be a contiguous (M, N) float16/bfloat16/float32 tensor")
    if C.is_cuda != want_cuda:
        raise ValueError(f"C must be a {device_kind} tensor")
    return M, N, K, C, din


def _on_device(dev: int, fn, *args):
    """Call fn(*args) with CUDA device `dev` current (no device switch when it already is)."""
    if dev == torch.cuda.current_device():
        return fn(*args)
    with torch.cuda.device(dev):
        return fn(*args)


def _gemm_call(a, b, c, M, N, K, din, dout, lb, opts, stream, dev):
    st = _stream_ptr(stream, dev)
    if opts is None:
        return binding.lib.gemm(a, b, c, M, N, K, din, dout, GEMM_K_MAJOR, lb, st), "gemm"
    return binding.lib.gemm_ex(a, b, c, M, N, K, din, dout, GEMM_K_MAJOR, lb, ctypes.byref(opts), st), "gemm_ex"


def gemm(A: torch.Tensor, B: torch.Tensor, C: torch.Tensor | None = None, *,
         layout_b: str = "k", out_dtype: torch.dtype | None = None, stream=None,
         options=None) -> torch.Tensor:
    """C = A·B on A's CUDA device, asynchronously on ``stream`` (default: torch's current).

    A: (M, K). B: (N, K) for layout_b="k", (K, N) for layout_b="mn" (16-bit types
    only). C: (M, N) of ``out_dtype`` (default A.dtype, BF16 for FP8 inputs),
    allocated when not given.
    ``options``: dict or GemmOptions of gemm_ex overrides.
    """
    M, N, K, C, din = _prepare(A, B, C, layout_b, out_dtype, "cuda")
    dev = A.get_device()
    args = (A.data_ptr(), B.data_ptr(), C.data_ptr(), M, N, K, din, _DT_OUT[C.dtype], _LAYOUT[layout_b],
            _options(options), stream, dev)
    if dev == torch.cuda.current_device():
        status, what = _gemm_call(*args)
    else:
        with torch.cuda.device(dev):
            status, what = _gemm_call(*args)
    if status != GEMM_OK:
        raise GemmError(status, what)
    return C


def gemm_ex(A, B, C=None, *, options=None, **kw) -> torch.Tensor:
    """gemm with gemm_ex overrides (cta_group, block_n, max_clusters, group_m, timeout_ms,
    k_stage, stream_k)."""
    return gemm(A, B, C, options=options if options is not None else GemmOptions(), **kw)


def gemm_mx(A: torch.Tensor, B: torch.Tensor, SFA: torch.Tensor, SFB: torch.Tensor,
            C: torch.Tensor | None = None, *, K: int | None = None,
            out_dtype: torch.dtype = torch.bfloat16, stream=None, options=None) -> torch.Tensor:
    """Block-scaled C = (SFA o A)(SFB o B) on A's CUDA device (gemm_mx / gemm_mx_ex).

    MXFP8: A (M, K) and B (N, K) float8_e4m3fn or float8_e5m2. MXFP4: A (M, ceil(K/2))
    and B (N, ceil(K/2)) uint8 holding packed E2M1 pairs (lower k in the low nibble);
    K defaults to twice the byte width. SFA (M, ceil(K/32)) and SFB (N, ceil(K/32))
    uint8 E8M0 scale exponents. C: (M, N) of ``out_dtype``, allocated when not given.
    """
    for name, t in (("A", A), ("B", B), ("SFA", SFA), ("SFB", SFB)):
        if t.device.type != "cuda" or not t.is_contiguous() or t.dim() != 2:
            raise ValueError(f"{name} must be a contiguous 2-D CUDA tensor")
    if A.dtype != B.dtype:
        raise TypeError("A and B must have the same dtype")
    if A.dtype in _FP8:
        dtype_in, K_ = _DT_IN[A.dtype], int(A.shape[1])
        if K is not None and K != K_:
            raise ValueError("K must equal A.shape[1] for FP8 elements")
    elif A.dtype == torch.uint8:
        dtype_in, K_ = GEMM_E2M1, int(K if K is not None else 2 * A.shape[1])
        if (K_ + 1) // 2 != A.shape[1]:
            raise ValueError("packed E2M1 rows must hold ceil(K/2) bytes")
    else:
        raise TypeError("A must be float8_e4m3fn, float8_e5m2 or uint8 (packed E2M1)")
    M, N = int(A.shape[0]), int(B.shape[0])
    nb = (K_ + 31) // 32
    if tuple(B.shape) != (N, A.shape[1]):
        raise ValueError("B must be (N, K) like A")
    if tuple(SFA.shape) != (M, nb) or tuple(SFB.shape) != (N, nb) or SFA.dtype != torch.uint8 \
            or SFB.dtype != torch.uint8:
        raise ValueError(f"SFA must be uint8 ({M}, {nb}) and SFB uint8 ({N}, {nb})")
    if C is None:
        C = torch.empty((M, N), dtype=out_dtype, device=A.device)
    if C.dtype not in _DT_OUT or tuple(C.shape) != (M, N) or not C.is_contiguous():
        raise ValueError("C must be a contiguous (M, N) float16/bfloat16/float32 tensor")
    opts = _options(options)
    args = (A.data_ptr(), B.data_ptr(), SFA.data_ptr(), SFB.data_ptr(), C.data_ptr(), M, N, K_,
            dtype_in, _DT_OUT[C.dtype], GEMM_K_MAJOR, GEMM_K_MAJOR)
    with torch.cuda.device(A.device):
        if opts is None:
            _check(binding.lib.gemm_mx(*args, _stream_ptr(stream)), "gemm_mx")
        else:
            _check(binding.lib.gemm_mx_ex(*args, ctypes.byref(opts), _stream_ptr(stream)), "gemm_mx_ex")
    return C


def attention(Q: torch.Tensor, K: torch.Tensor, V: torch.Tensor, *, causal: bool = False,
              scale: float | None = None, O: torch.Tensor | None = None, return_lse: bool = False,
              stream=None, max_ctas: int = 0):
    """O = softmax(scale * Q K^T) V per (batch, head) on Q's CUDA device (attention_fwd_ex).

    Q: (B, H, Lq, 128), K and V: (B, H, Lk, 128), float16 or bfloat16, contiguous.
    ``causal``: key k is visible to row i iff k <= i + (Lk - Lq). ``scale`` defaults to
    1/sqrt(128). ``max_ctas`` > 0 caps the persistent grid (each CTA then takes more
    256-row blocks; the result is the same). Returns O (B, H, Lq, 128), and with
    ``return_lse`` also the FP32 row log-sum-exp (B, H, Lq).
    """
    for name, t in (("Q", Q), ("K", K), ("V", V)):
        if t.device.type != "cuda" or not t.is_contiguous() or t.dim() != 4:
            raise ValueError(f"{name} must be a contiguous 4-D CUDA tensor")
        if t.dtype not in (torch.float16, torch.bfloat16) or t.dtype != Q.dtype:
            raise TypeError("Q, K and V must share one dtype, float16 or bfloat16")
    B, H, Lq, d = Q.shape
    if tuple(K.shape[:2]) != (B, H) or K.shape[3] != d or V.shape != K.shape:
        raise ValueError("K and V must be (B, H, Lk, d) with Q's B, H and d")
    Lk = K.shape[2]
    if O is None:
        O = torch.empty_like(Q)
    if O.shape != Q.shape or O.dtype != Q.dtype or not O.is_contiguous():
        raise ValueError("O must be a contiguous tensor shaped and typed like Q")
    lse = torch.empty((B, H, Lq), dtype=torch.float32, device=Q.device) if return_lse else None
    scale = float(d) ** -0.5 if scale is None else float(scale)
    with torch.cuda.device(Q.device):
        _check(binding.lib.attention_fwd_ex(Q.data_ptr(), K.data_ptr(), V.data_ptr(), O.data_ptr(),
                                            lse.data_ptr() if lse is not None else None, B, H, Lq, Lk, d,
                                            _DT_IN[Q.dtype], int(bool(causal)), scale, int(max_ctas),
                                            _stream_ptr(stream)),
               "attention_fwd_ex")
    return (O, lse) if return_lse else O


def gemm_plan(M: int, N: int, K: int, *, dtype_in=torch.float16, dtype_out=torch.float16,
              layout_b: str = "k", a_ptr: int = 256, b_ptr: int = 256, c_ptr: int = 256,
              options=None, device=None, block_scaled: bool = False) -> dict:
    """The launch gemm_ex (or, with block_scaled, gemm_mx_ex) would make: tile, grid,
    stream-K split, realign/direct-store paths, as a dict. The pointers only matter
    for their alignment. For block-scaled packed FP4 pass dtype_in=torch.uint8."""
    plan = GemmPlan()
    opts = _options(options)
    din = GEMM_E2M1 if dtype_in == torch.uint8 else _DT_IN[dtype_in]
    fn = binding.lib.gemm_mx_plan if block_scaled else binding.lib.gemm_plan
    with torch.cuda.device(device if device is not None else torch.cuda.current_device()):
        _check(fn(M, N, K, din, _DT_OUT[dtype_out], GEMM_K_MAJOR, _LAYOUT[layout_b], a_ptr, b_ptr, c_ptr,
                  ctypes.byref(opts) if opts is not None else None, ctypes.byref(plan)), "gemm_plan")
    return plan.as_dict()


def gemm_from_host(A: torch.Tensor, B: torch.Tensor, C: torch.Tensor | None = None, *,
                   layout_b: str = "k", out_dtype: torch.dtype | None = None, stream=None,
                   device=None) -> torch.Tensor:
    """C = A·B with host (CPU) tensors; copies in, computes and copies out on the current
    CUDA device, and returns when C is complete."""
    M, N, K, C, din = _prepare(A, B, C, layout_b, out_dtype, "cpu")
    with torch.cuda.device(device if device is not None else torch.cuda.current_device()):
        _check(binding.lib.gemm_from_host(A.data_ptr(), B.data_ptr(), C.data_ptr(), M, N, K,
                                          din, _DT_OUT[C.dtype], GEMM_K_MAJOR,
                                          _LAYOUT[layout_b], _stream_ptr(stream)),
               "gemm_from_host")
    return C


def gemm_from_host_async(A: torch.Tensor, B: torch.Tensor, C: torch.Tensor | None = None, *,
                   layout_b: str = "k", out_dtype: torch.dtype | None = None, stream=None,
                   device=None) -> torch.Tensor:
    """gemm_from_host without the final synchronisation: C is complete once ``stream``
    (default: the current stream) has passed the call; A and B must stay unchanged until
    then. Consecutive calls overlap one call's uploads with the previous call's product
    and read-back. Use pinned host tensors for the overlap."""
    M, N, K, C, din = _prepare(A, B, C, layout_b, out_dtype, "cpu")
    with torch.cuda.device(device if device is not None else torch.cuda.current_device()):
        _check(binding.lib.gemm_from_host_async(A.data_ptr(), B.data_ptr(), C.data_ptr(), M, N, K,
                                          din, _DT_OUT[C.dtype], GEMM_K_MAJOR,
                                          _LAYOUT[layout_b], _stream_ptr(stream)),
               "gemm_from_host_async")
    return C


def gemm_release_workspace() -> None:
    _check(binding.lib.gemm_release_workspace(), "gemm_release_workspace")


def gemm_last_device_status(stream=None) -> tuple[int, int]:
    """Synchronise the stream, then read and clear the device status word.
    Returns (status, detail); status GEMM_ERR_TIMEOUT means a kernel wait timed out."""
    detail = ctypes.c_uint32(0)
    st = binding.lib.gemm_last_device_status(_stream_ptr(stream), ctypes.byref(detail))
    return int(st), int(detail.value)


def gemm_selftest_wait_timeout(timeout_ms: int = 50, stream=None) -> None:
    _check(binding.lib.gemm_selftest_wait_timeout(int(timeout_ms), _stream_ptr(stream)),
           "gemm_selftest_wait_timeout")


def gemm_selftest_withheld_load(A: torch.Tensor, B: torch.Tensor, C: torch.Tensor, *, layout_b: str = "k",
                                cta_group: int = 2, withhold_kb: int = 1, timeout_ms: int = 20,
                                stream=None) -> None:
    """Run the GEMM kernel with the first unit's producer withholding the loads of
    k-block ``withhold_kb`` of its first tile, so that its waits run out after
    ``timeout_ms``. Read the outcome with gemm_last_device_status."""
    M, N, K, C, din = _prepare(A, B, C, layout_b, None, "cuda")
    with torch.cuda.device(A.device):
        _check(binding.lib.gemm_selftest_withheld_load(A.data_ptr(), B.data_ptr(), C.data_ptr(), M, N, K, din,
                                                       _DT_OUT[C.dtype], _LAYOUT[layout_b], int(cta_group),
                                                       int(withhold_kb), int(timeout_ms), _stream_ptr(stream)),
               "gemm_selftest_withheld_load")


def gemm_cache_stats() -> dict:
    """Launch-cache counters of this process: plan and tensor-map hits and misses."""
    v = [ctypes.c_uint64(0) for _ in range(4)]
    binding.lib.gemm_cache_stats(*(ctypes.byref(x) for x in v))
    return dict(zip(("plan_hits", "plan_misses", "map_hits", "map_misses"), (int(x.value) for x in v)))


def gemm_cache_clear() -> None:
    """Empty the launch cache of the current device."""
    _check(binding.lib.gemm_cache_clear(), "gemm_cache_clear")


def gemm_status_string(status: int) -> str:
    return binding.lib.gemm_status_string(int(status)).decode()


def gemm_launch_count() -> int:
    return int(binding.lib.gemm_launch_count())


def gemm_schedule_jobs(num_tiles: int, units: int, k_blocks: int, sk_tiles: int,
                       unit: int) -> list[tuple[int, int, int, int]]:
    """The kernel's work list for one unit, as (tile, kb_begin, kb_end, kind) tuples in
    run order; kind is GEMM_JOB_FULL, GEMM_JOB_WRITER or GEMM_JOB_OWNER. No GPU needed."""
    n = ctypes.c_int32(0)
    _check(binding.lib.gemm_schedule_jobs(num_tiles, units, k_blocks, sk_tiles, unit, None, 0,
                                          ctypes.byref(n)), "gemm_schedule_jobs")
    jobs = (GemmJob * max(1, n.value))()
    _check(binding.lib.gemm_schedule_jobs(num_tiles, units, k_blocks, sk_tiles, unit, jobs, n.value,
                                          ctypes.byref(n)), "gemm_schedule_jobs")
    return [(j.tile, j.kb_begin, j.kb_end, j.kind) for j in jobs[:n.value]]


def gemm_no_alloc_scratch() -> tuple[int, int]:
    """(device address, size in bytes) of the current device's gemm_no_alloc array."""
    ptr, size = ctypes.c_void_p(0), ctypes.c_size_t(0)
    _check(binding.lib.gemm_no_alloc_scratch(ctypes.byref(ptr), ctypes.byref(size)), "gemm_no_alloc_scratch")
    return int(ptr.value or 0), int(size.value)


def gemm_no_alloc(A: torch.Tensor, B: torch.Tensor, C: torch.Tensor, *, layout_b: str = "k",
                  stream=None) -> torch.Tensor:
    """gemm for callers that must not allocate device memory, for example a serving
    runtime whose memory pool already owns the GPU, or a latency-critical loop where an
    allocation could stall or fail. The caller passes C. An operand that needs
    re-pitching goes into the library's fixed 32 MiB device array instead of newly
    allocated memory. Calls whose padded operands exceed that array raise GemmError
    (GEMM_ERR_UNSUPPORTED). Calls that overlap on the GPU share the array and race."""
    if C is None:
        raise ValueError("gemm_no_alloc needs the caller's C")
    M, N, K, C, din = _prepare(A, B, C, layout_b, None, "cuda")
    with torch.cuda.device(A.device):
        _check(binding.lib.gemm_no_alloc(A.data_ptr(), B.data_ptr(), C.data_ptr(), M, N, K,
                                         din, _DT_OUT[C.dtype], GEMM_K_MAJOR,
                                         _LAYOUT[layout_b], _stream_ptr(stream)),
               "gemm_no_alloc")
    return C
