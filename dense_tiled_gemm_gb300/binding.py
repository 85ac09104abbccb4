"""ctypes binding to libdtgemm.so (the C ABI in include/gemm.h).

Argument marshalling only: every computation runs in the library's CUDA
kernels. There is no fallback of any kind. If the library is missing, the
import fails; if it returns an error, a GemmError is raised.
"""
from __future__ import annotations

import ctypes
import os

from .build import LIB_PATH

GEMM_F16, GEMM_BF16, GEMM_F32, GEMM_E4M3, GEMM_E5M2, GEMM_E2M1 = 0, 1, 2, 3, 4, 5
GEMM_K_MAJOR, GEMM_MN_MAJOR = 0, 1
STATUS_NAMES = {
    0: "GEMM_OK",
    1: "GEMM_ERR_INVALID_ARG",
    2: "GEMM_ERR_UNSUPPORTED",
    3: "GEMM_ERR_CUDA",
    4: "GEMM_ERR_TIMEOUT",
    5: "GEMM_ERR_NO_DEVICE",
    6: "GEMM_ERR_OUT_OF_MEMORY",
}
GEMM_OK, GEMM_ERR_INVALID_ARG, GEMM_ERR_UNSUPPORTED, GEMM_ERR_CUDA = 0, 1, 2, 3
GEMM_ERR_TIMEOUT, GEMM_ERR_NO_DEVICE, GEMM_ERR_OUT_OF_MEMORY = 4, 5, 6


class GemmOptions(ctypes.Structure):
    _fields_ = [("cta_group", ctypes.c_int32), ("block_n", ctypes.c_int32),
                ("max_clusters", ctypes.c_int32), ("group_m", ctypes.c_int32),
                ("timeout_ms", ctypes.c_int32), ("k_stage", ctypes.c_int32),
                ("stream_k", ctypes.c_int32), ("cluster_pairs", ctypes.c_int32),
                ("clock_trace", ctypes.c_void_p), ("epilogue_warps", ctypes.c_int32),
                ("reserved", ctypes.c_int32)]


class GemmPlan(ctypes.Structure):
    _fields_ = [("cta_group", ctypes.c_int32), ("block_m", ctypes.c_int32),
                ("block_n", ctypes.c_int32), ("block_k", ctypes.c_int32),
                ("stages", ctypes.c_int32), ("num_tiles", ctypes.c_int32),
                ("grid_ctas", ctypes.c_int32), ("group_m", ctypes.c_int32),
                ("realign_a", ctypes.c_int32), ("realign_b", ctypes.c_int32),
                ("direct_store", ctypes.c_int32), ("smem_bytes", ctypes.c_int32),
                ("num_sms", ctypes.c_int32), ("sk_tiles", ctypes.c_int32),
                ("workspace_bytes", ctypes.c_int32), ("cluster_pairs", ctypes.c_int32),
                ("epilogue_warps", ctypes.c_int32)]

    def as_dict(self) -> dict:
        return {name: getattr(self, name) for name, _ in self._fields_}


class GemmJob(ctypes.Structure):
    _fields_ = [("tile", ctypes.c_int32), ("kb_begin", ctypes.c_int32),
                ("kb_end", ctypes.c_int32), ("kind", ctypes.c_int32)]


GEMM_JOB_FULL, GEMM_JOB_WRITER, GEMM_JOB_OWNER = 0, 1, 2


class GemmError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = int(status)
        super().__init__(f"{what}: {STATUS_NAMES.get(self.status, self.status)}")


def _declare(lib):
    vp, i64, i32, c_int = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_int
    gemm_args = [vp, vp, vp, i64, i64, i64, c_int, c_int, c_int, c_int]
    lib.gemm.restype = c_int
    lib.gemm.argtypes = gemm_args + [vp]
    lib.gemm_ex.restype = c_int
    lib.gemm_ex.argtypes = gemm_args + [ctypes.POINTER(GemmOptions), vp]
    mx_args = [vp, vp, vp, vp, vp, i64, i64, i64, c_int, c_int, c_int, c_int]
    lib.gemm_mx.restype = c_int
    lib.gemm_mx.argtypes = mx_args + [vp]
    lib.gemm_mx_ex.restype = c_int
    lib.gemm_mx_ex.argtypes = mx_args + [ctypes.POINTER(GemmOptions), vp]
    lib.gemm_plan.restype = c_int
    lib.gemm_plan.argtypes = [i64, i64, i64, c_int, c_int, c_int, c_int, vp, vp, vp,
                              ctypes.POINTER(GemmOptions), ctypes.POINTER(GemmPlan)]
    lib.gemm_mx_plan.restype = c_int
    lib.gemm_mx_plan.argtypes = lib.gemm_plan.argtypes
    lib.gemm_from_host.restype = c_int
    lib.gemm_from_host.argtypes = gemm_args + [vp]
    lib.gemm_from_host_async.restype = c_int
    lib.gemm_from_host_async.argtypes = gemm_args + [vp]
    lib.gemm_release_workspace.restype = c_int
    lib.gemm_release_workspace.argtypes = []
    lib.gemm_last_device_status.restype = c_int
    lib.gemm_last_device_status.argtypes = [vp, ctypes.POINTER(ctypes.c_uint32)]
    lib.gemm_selftest_wait_timeout.restype = c_int
    lib.gemm_selftest_wait_timeout.argtypes = [i32, vp]
    lib.gemm_status_string.restype = ctypes.c_char_p
    lib.gemm_status_string.argtypes = [c_int]
    lib.gemm_launch_count.restype = ctypes.c_uint64
    lib.gemm_launch_count.argtypes = []
    lib.attention_fwd.restype = c_int
    lib.attention_fwd_ex.restype = c_int
    lib.attention_fwd.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, i64, i64, c_int, c_int,
                                  ctypes.c_float, vp]
    lib.attention_fwd_ex.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, i64, i64, c_int, c_int,
                                     ctypes.c_float, c_int, vp]
    u64p = ctypes.POINTER(ctypes.c_uint64)
    lib.gemm_cache_stats.restype = None
    lib.gemm_cache_stats.argtypes = [u64p, u64p, u64p, u64p]
    lib.gemm_cache_clear.restype = c_int
    lib.gemm_cache_clear.argtypes = []
    lib.gemm_selftest_withheld_load.restype = c_int
    lib.gemm_selftest_withheld_load.argtypes = [vp, vp, vp, i64, i64, i64, c_int, c_int, c_int, i32, i32,
                                                i32, vp]
    lib.gemm_schedule_jobs.restype = c_int
    lib.gemm_schedule_jobs.argtypes = [i32, i32, i32, i32, i32, ctypes.POINTER(GemmJob), i32,
                                       ctypes.POINTER(i32)]
    lib.gemm_no_alloc.restype = c_int
    lib.gemm_no_alloc.argtypes = gemm_args + [vp]
    lib.gemm_no_alloc_scratch.restype = c_int
    lib.gemm_no_alloc_scratch.argtypes = [ctypes.POINTER(vp), ctypes.POINTER(ctypes.c_size_t)]
    return lib


def load(path: str = LIB_PATH):
    if not os.path.exists(path):
        raise ImportError(f"{path} is not built; call dense_tiled_gemm_gb300.build.build() "
                          "(needs nvcc) before importing the package")
    return _declare(ctypes.CDLL(path))


lib = load()
