"""C-ABI boundary checks that need no GPU: the library loads, it exports
every function include/gemm.h declares, the ctypes structs match the header,
and invalid arguments are rejected on the host before any CUDA call."""
from __future__ import annotations

import ctypes
import os
import re

import pytest

from dense_tiled_gemm_gb300 import binding
import dense_tiled_gemm_gb300 as dtg

INCLUDE = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include")
HEADER = os.path.join(INCLUDE, "gemm.h")
FAKE = 0x10000   # never dereferenced: every call below fails validation first


def header_text() -> str:
    with open(HEADER) as fh:
        return fh.read()


def declared_functions() -> list[str]:
    names = set()
    for name in sorted(os.listdir(INCLUDE)):
        if name.endswith(".h"):
            with open(os.path.join(INCLUDE, name)) as fh:
                text = re.sub(r"/\*.*?\*/", "", fh.read(), flags=re.S)
            names |= set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*((?:gemm|attention)\w*)\s*\(", text,
                                    flags=re.M))
    return sorted(names)


def test_header_declares_the_entry_points():
    names = declared_functions()
    for required in ("gemm", "gemm_ex", "gemm_plan", "gemm_from_host", "gemm_last_device_status",
                     "gemm_status_string", "gemm_selftest_wait_timeout", "gemm_launch_count",
                     "gemm_release_workspace", "gemm_mx", "gemm_mx_ex", "gemm_mx_plan",
                     "gemm_schedule_jobs", "gemm_no_alloc", "attention_fwd", "attention_fwd_ex",
                     "gemm_from_host_async", "gemm_cache_stats", "gemm_cache_clear",
                     "gemm_selftest_withheld_load"):
        assert required in names


def test_library_exports_every_declared_function():
    for name in declared_functions():
        assert hasattr(binding.lib, name), f"{name} declared in gemm.h but not exported"


def test_enums_match_header():
    text = header_text()
    for name, val in (("GEMM_F16", 0), ("GEMM_BF16", 1), ("GEMM_F32", 2), ("GEMM_E4M3", 3),
                      ("GEMM_E5M2", 4), ("GEMM_E2M1", 5), ("GEMM_K_MAJOR", 0),
                      ("GEMM_MN_MAJOR", 1), ("GEMM_OK", 0), ("GEMM_ERR_INVALID_ARG", 1),
                      ("GEMM_ERR_UNSUPPORTED", 2), ("GEMM_ERR_CUDA", 3), ("GEMM_ERR_TIMEOUT", 4),
                      ("GEMM_ERR_NO_DEVICE", 5), ("GEMM_ERR_OUT_OF_MEMORY", 6)):
        assert re.search(rf"\b{name}\s*=\s*{val}\b", text), name
        assert getattr(binding, name) == val


def test_struct_sizes():
    # gemm_options_t: 8 int32 fields, the clock-trace pointer, 2 int32 fields;
    # gemm_plan_t: 17 int32 fields
    assert ctypes.sizeof(binding.GemmOptions) == 48
    assert binding.GemmOptions.clock_trace.offset == 32
    assert binding.GemmOptions.epilogue_warps.offset == 40
    assert ctypes.sizeof(binding.GemmPlan) == 68
    assert re.search(r"int32_t cluster_pairs;\s*uint64_t \*clock_trace;\s*int32_t epilogue_warps;\s*"
                     r"int32_t reserved;[^\n]*\n\} gemm_options_t;", header_text())
    assert re.search(r"int32_t epilogue_warps;[^\n]*\n\} gemm_plan_t;", header_text())


def test_prototypes_use_the_enum_types():
    """Every entry point that takes an element type or a layout declares it with
    gemm_dtype_t / gemm_layout_t, so that a C caller gets type checking."""
    text = re.sub(r"/\*.*?\*/", "", header_text(), flags=re.S)
    assert not re.search(r"\bint\s+(dtype_in|dtype_out|layoutA|layoutB)\b", text)
    assert len(re.findall(r"gemm_dtype_t dtype_in", text)) >= 10
    assert len(re.findall(r"gemm_layout_t layoutB", text)) >= 10
    assert "const char *gemm_status_string(gemm_status_t status);" in text


def test_cache_entry_points_without_gpu():
    """The cache counters are readable without a device; clearing needs one."""
    stats = dtg.gemm_cache_stats()
    assert set(stats) == {"plan_hits", "plan_misses", "map_hits", "map_misses"}
    assert all(v >= 0 for v in stats.values())
    import torch
    if not torch.cuda.is_available():
        assert binding.lib.gemm_cache_clear() == binding.GEMM_ERR_NO_DEVICE


@pytest.mark.parametrize("cg,kb,ms,expect", [(3, 0, 20, 1), (0, 0, 20, 1), (2, -1, 20, 1), (2, 0, 0, 1),
                                              (1, 0, 20000, 1)])
def test_withheld_load_selftest_validates_on_host(cg, kb, ms, expect):
    rc = binding.lib.gemm_selftest_withheld_load(FAKE, FAKE, FAKE, 256, 256, 256, 0, 2, 0, cg, kb, ms, None)
    assert rc == expect


def test_status_strings():
    for code, name in binding.STATUS_NAMES.items():
        assert dtg.gemm_status_string(code) == name
    assert dtg.gemm_status_string(99) == "GEMM_ERR_UNKNOWN"


def call(M=64, N=64, K=64, din=0, dout=0, la=0, lb=0, a=FAKE, b=FAKE, c=FAKE):
    return binding.lib.gemm(a, b, c, M, N, K, din, dout, la, lb, None)


@pytest.mark.parametrize("kwargs,expect", [
    (dict(a=None), 1), (dict(b=None), 1), (dict(c=None), 1),
    (dict(M=0), 1), (dict(N=0), 1), (dict(K=0), 1), (dict(M=-5), 1), (dict(K=2 ** 31), 1),
    (dict(din=7), 1), (dict(din=2), 2), (dict(dout=5), 1), (dict(dout=-1), 1),
    (dict(la=1), 2), (dict(la=3), 1), (dict(lb=2), 1),
    (dict(dout=3), 2), (dict(dout=4), 2),                      # FP8 is an input type only
    (dict(din=3, lb=1), 2), (dict(din=4, lb=1), 2),            # FP8 B must be K-major
    (dict(din=3, lb=2), 1),
    (dict(din=5), 2),                                          # packed FP4 only through gemm_mx
])
def test_invalid_arguments_rejected_on_host(kwargs, expect):
    assert call(**kwargs) == expect


@pytest.mark.parametrize("fn", ["gemm_from_host", "gemm_from_host_async", "gemm_no_alloc"])
@pytest.mark.parametrize("kwargs,expect", [
    (dict(a=None), 1), (dict(c=None), 1), (dict(K=0), 1), (dict(N=-1), 1), (dict(din=7), 1),
    (dict(din=2), 2), (dict(dout=3), 2), (dict(la=1), 2), (dict(din=3, lb=1), 2), (dict(din=5), 2),
])
def test_other_entry_points_validate_on_host(fn, kwargs, expect):
    """The host-buffer and allocation-free entry points run the same argument
    checks before they touch a device (or, here, find none)."""
    args = dict(M=64, N=64, K=64, din=0, dout=0, la=0, lb=0, a=FAKE, b=FAKE, c=FAKE)
    args.update(kwargs)
    rc = getattr(binding.lib, fn)(args["a"], args["b"], args["c"], args["M"], args["N"], args["K"],
                                  args["din"], args["dout"], args["la"], args["lb"], None)
    assert rc == expect


def test_invalid_options_rejected_on_host():
    for field, val, expect in (("cta_group", 3, 1), ("cta_group", -1, 1), ("block_n", 96, 2),
                               ("max_clusters", -2, 1), ("group_m", -1, 1), ("timeout_ms", -1, 1),
                               ("k_stage", 96, 2), ("k_stage", -64, 1), ("stream_k", 3, 2),
                               ("stream_k", -1, 1), ("cluster_pairs", -1, 1), ("cluster_pairs", 3, 2),
                               ("epilogue_warps", -4, 1), ("epilogue_warps", 6, 2), ("reserved", 1, 1)):
        o = binding.GemmOptions()
        setattr(o, field, val)
        rc = binding.lib.gemm_ex(FAKE, FAKE, FAKE, 64, 64, 64, 0, 0, 0, 0, ctypes.byref(o), None)
        assert rc == expect, field


@pytest.mark.parametrize("din,k_stage,expect", [(0, 256, 2), (3, 64, 2), (4, 192, 2), (3, -128, 1)])
def test_k_stage_depends_on_input_width(din, k_stage, expect):
    """k_stage counts elements: one or two 128-byte slabs (64/128 for 16-bit, 128/256 for FP8)."""
    o = binding.GemmOptions()
    o.k_stage = k_stage
    rc = binding.lib.gemm_ex(FAKE, FAKE, FAKE, 64, 64, 64, din, 0, 0, 0, ctypes.byref(o), None)
    assert rc == expect


def test_python_wrapper_accepts_fp8_types():
    import torch
    A = torch.zeros(4, 8, dtype=torch.float8_e4m3fn)
    with pytest.raises(ValueError):
        dtg.gemm(A, torch.zeros(5, 8, dtype=torch.float8_e4m3fn))   # CPU tensors, not a type error
    with pytest.raises(TypeError):
        dtg.gemm_from_host(A, torch.zeros(5, 8, dtype=torch.float8_e5m2))   # mixed FP8 types


def mx_call(din=3, dout=1, lb=0, sfa=FAKE, sfb=FAKE, opts=None, M=64, N=64, K=64):
    if opts is None:
        return binding.lib.gemm_mx(FAKE, FAKE, sfa, sfb, FAKE, M, N, K, din, dout, 0, lb, None)
    return binding.lib.gemm_mx_ex(FAKE, FAKE, sfa, sfb, FAKE, M, N, K, din, dout, 0, lb,
                                  ctypes.byref(opts), None)


@pytest.mark.parametrize("kwargs,expect", [
    (dict(sfa=None), 1), (dict(sfb=None), 1), (dict(din=0), 2), (dict(din=1), 2), (dict(din=2), 2),
    (dict(din=9), 1), (dict(lb=1), 2), (dict(din=5, lb=1), 2), (dict(dout=3), 2), (dict(K=0), 1),
])
def test_gemm_mx_rejects_on_host(kwargs, expect):
    assert mx_call(**kwargs) == expect


def test_gemm_mx_options():
    o = binding.GemmOptions()
    o.k_stage = 128          # MXFP8 stages are one or two 128-K slabs: 128 is allowed in validation
    assert mx_call(opts=o) in (binding.GEMM_ERR_NO_DEVICE, binding.GEMM_ERR_UNSUPPORTED)
    o.k_stage = 384
    assert mx_call(opts=o) == binding.GEMM_ERR_UNSUPPORTED
    o.k_stage = 0
    o.stream_k = 5
    assert mx_call(opts=o) == binding.GEMM_ERR_UNSUPPORTED


def att_call(Q=FAKE, K=FAKE, V=FAKE, O=FAKE, lse=None, B=1, H=1, Lq=128, Lk=128, d=128, dt=1, causal=0,
             scale=0.088):
    return binding.lib.attention_fwd(Q, K, V, O, lse, B, H, Lq, Lk, d, dt, causal, scale, None)


@pytest.mark.parametrize("kwargs,expect", [
    (dict(Q=None), 1), (dict(O=None), 1), (dict(B=0), 1), (dict(Lk=0), 1), (dict(dt=7), 1),
    (dict(dt=2), 2), (dict(d=64), 2), (dict(causal=2), 1), (dict(scale=float("inf")), 1),
    (dict(scale=0.0), 1), (dict(scale=-0.5), 1),
    (dict(B=65536, H=32768), 2), (dict(B=1 << 31, H=1), 2), (dict(Q=FAKE + 8), 2), (dict(lse=FAKE + 2), 1),
])
def test_attention_rejects_on_host(kwargs, expect):
    assert att_call(**kwargs) == expect
    # the capped-grid entry validates the same way, whatever the cap
    a = dict(Q=FAKE, K=FAKE, V=FAKE, O=FAKE, lse=None, B=1, H=1, Lq=128, Lk=128, d=128, dt=1, causal=0,
             scale=0.088)
    a.update(kwargs)
    for cap in (0, 3, -1):
        assert binding.lib.attention_fwd_ex(a["Q"], a["K"], a["V"], a["O"], a["lse"], a["B"], a["H"], a["Lq"],
                                            a["Lk"], a["d"], a["dt"], a["causal"], a["scale"], cap,
                                            None) == expect


def test_attention_no_device():
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert att_call() == binding.GEMM_ERR_NO_DEVICE


def test_plan_requires_output_struct():
    assert binding.lib.gemm_plan(64, 64, 64, 0, 0, 0, 0, FAKE, FAKE, FAKE, None, None) == 1


def test_selftest_rejects_bad_limit():
    assert binding.lib.gemm_selftest_wait_timeout(0, None) == 1
    assert binding.lib.gemm_selftest_wait_timeout(20000, None) == 1


def test_python_wrapper_validates_shapes():
    import torch
    A = torch.zeros(4, 8, dtype=torch.float16)
    B = torch.zeros(5, 9, dtype=torch.float16)
    with pytest.raises(ValueError):
        dtg.gemm(A, B)               # K mismatch
    with pytest.raises(TypeError):
        dtg.gemm(A.float(), B)       # unsupported input dtype
    with pytest.raises(ValueError):
        dtg.gemm(A, torch.zeros(5, 8, dtype=torch.float16))   # CPU tensors on the device path


def test_no_gpu_gives_no_device():
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert call() == binding.GEMM_ERR_NO_DEVICE
    assert binding.lib.gemm_last_device_status(None, None) == binding.GEMM_ERR_NO_DEVICE
