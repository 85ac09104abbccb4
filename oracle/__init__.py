"""CPU FP64 oracle for the dense tiled GEMM: test infrastructure only.

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
and reference legs may import this package. The CUDA product path
(``dense_tiled_gemm_gb300``) never imports it, and this package imports
nothing from there. The two meet only in the seeded input generator
(``workloads.py``), which holds no GEMM arithmetic.

``gemm_ref`` is a ctypes wrapper around ``gemm_oracle.c``. It implements the
plain definition C[i][j] = sum_k a[i][k]*b[k][j] in FP64 over the exact
FP16/BF16 or FP8 (E4M3/E5M2) operand values (k ascending), plus
C_abs[i][j] = sum_k |a·b|. FP8 operands carry the identity block scale
(1.0) of "Porting High-Performance HIP Kernels to FlyDSL", section "A More
Complex Kernel", so their products are the plain products.
``gemm_ref_mx`` is the block-scaled (MX) form measured in "Two Waves, One Stage
Apart" (section "MI450", Table 1): E4M3/E5M2 or packed E2M1 elements, each
run of 32 consecutive K elements of a row of A (and of a column of B) scaled
by one E8M0 value 2^(e-127).
It follows "Two Waves, One Stage Apart" (opening paragraph: a tiled GEMM
sums operand-tile products) and counts 2·M·N·K flops as in that page's
Table 1 caption.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gemm_oracle.c")
_ATT_SRC = os.path.join(_HERE, "attention_oracle.c")
SOURCES = (_SRC, _ATT_SRC)
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

F16, BF16, E4M3, E5M2, E2M1 = 0, 1, 3, 4, 5
MX_BLOCK = 32
K_MAJOR, MN_MAJOR = 0, 1
_DTYPE = {"f16": F16, "bf16": BF16, "e4m3": E4M3, "e5m2": E5M2, "e2m1": E2M1}
# numpy type of the raw operand patterns for each input type
_STORAGE = {"f16": np.uint16, "bf16": np.uint16, "e4m3": np.uint8, "e5m2": np.uint8,
            "e2m1": np.uint8, "e8m0": np.uint8}
_LAYOUT = {"k": K_MAJOR, "mn": MN_MAJOR}


def compile_cmd(out: str, sources=SOURCES) -> list[str]:
    return ["gcc", "-std=c99", "-O2", "-ffp-contract=off", "-fno-fast-math",
            "-fPIC", "-shared", "-pthread", "-D_POSIX_C_SOURCE=200809L",
            "-o", out, *sources, "-lm"]


def build(force: bool = False) -> str:
    """Compile the oracle sources with gcc into liboracle.so (next to them)."""
    if (not force and os.path.exists(_LIB_PATH)
            and all(os.path.getmtime(_LIB_PATH) >= os.path.getmtime(p) for p in SOURCES)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = compile_cmd(tmp)
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def load_library(path: str):
    """Open a compiled oracle library and declare its C signatures."""
    lib = ctypes.CDLL(path)
    i64, dp, u16p = ctypes.c_int64, ctypes.POINTER(ctypes.c_double), ctypes.c_void_p
    lib.oracle_gemm.restype = ctypes.c_int
    lib.oracle_gemm.argtypes = [u16p, u16p, i64, i64, i64, ctypes.c_int, ctypes.c_int,
                                ctypes.c_void_p, i64, dp, dp, ctypes.c_int]
    lib.oracle_decode_f16.restype = ctypes.c_double
    lib.oracle_decode_f16.argtypes = [ctypes.c_uint16]
    lib.oracle_decode_bf16.restype = ctypes.c_double
    lib.oracle_decode_bf16.argtypes = [ctypes.c_uint16]
    for name in ("oracle_decode_e4m3", "oracle_decode_e5m2", "oracle_decode_e2m1",
                 "oracle_decode_e8m0"):
        getattr(lib, name).restype = ctypes.c_double
        getattr(lib, name).argtypes = [ctypes.c_uint8]
    lib.oracle_attention.restype = ctypes.c_int
    lib.oracle_attention.argtypes = [u16p, u16p, u16p, i64, i64, i64, i64, i64, ctypes.c_int,
                                     ctypes.c_int, ctypes.c_double, ctypes.c_void_p, i64, dp, dp,
                                     dp, ctypes.c_int]
    lib.oracle_gemm_mx.restype = ctypes.c_int
    lib.oracle_gemm_mx.argtypes = [u16p, u16p, u16p, u16p, i64, i64, i64, ctypes.c_int,
                                   ctypes.c_void_p, i64, dp, dp, ctypes.c_int]
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = load_library(build())
    return _lib


def host_threads() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def decode(bits, dtype: str, lib=None) -> np.ndarray:
    """Decode FP16/BF16 (16-bit), E4M3/E5M2/E8M0 (8-bit) or E2M1 (4-bit, one
    pattern per array entry) patterns to FP64 with the oracle's own decoders."""
    lib = lib or _load()
    fn = getattr(lib, f"oracle_decode_{dtype}")
    flat = np.asarray(bits, dtype=_STORAGE[dtype]).ravel()
    return np.array([fn(int(b)) for b in flat], dtype=np.float64).reshape(np.shape(bits))


def gemm_ref(A_bits: np.ndarray, B_bits: np.ndarray, M: int, N: int, K: int,
             dtype_in: str, layout_b: str, rows=None, threads: int | None = None,
             lib=None):
    """FP64 reference rows of C = A·B and of C_abs = sum_k |a·b|.

    A_bits: M×K patterns (row-major), uint16 for "f16"/"bf16" and uint8 for
    "e4m3"/"e5m2". B_bits: N×K for layout_b="k", K×N for layout_b="mn".
    ``rows``: output rows to compute (None = all).
    Returns (C, C_abs), each len(rows)×N (or M×N) float64. ``lib`` selects
    another compiled copy of the oracle (the tests' planted-mistake checks).
    """
    lib = lib or _load()
    A = np.ascontiguousarray(A_bits, dtype=_STORAGE[dtype_in])
    B = np.ascontiguousarray(B_bits, dtype=_STORAGE[dtype_in])
    if A.size != M * K or B.size != N * K:
        raise ValueError("operand sizes do not match M, N, K")
    if rows is None:
        rows_arr, n_rows, rows_ptr = None, M, None
    else:
        rows_arr = np.ascontiguousarray(rows, dtype=np.int64)
        n_rows = int(rows_arr.size)
        rows_ptr = rows_arr.ctypes.data_as(ctypes.c_void_p)
    C = np.empty((n_rows, N), dtype=np.float64)
    C_abs = np.empty((n_rows, N), dtype=np.float64)
    if n_rows == 0:
        return C, C_abs
    dp = ctypes.POINTER(ctypes.c_double)
    rc = lib.oracle_gemm(A.ctypes.data_as(ctypes.c_void_p), B.ctypes.data_as(ctypes.c_void_p),
                         M, N, K, _DTYPE[dtype_in], _LAYOUT[layout_b], rows_ptr, n_rows,
                         C.ctypes.data_as(dp), C_abs.ctypes.data_as(dp),
                         int(threads or host_threads()))
    if rc != 0:
        raise RuntimeError(f"oracle_gemm failed with code {rc}")
    return C, C_abs


def mx_blocks(K: int) -> int:
    """E8M0 scales per row: one per 32 consecutive K elements."""
    return (K + MX_BLOCK - 1) // MX_BLOCK


def gemm_ref_mx(A_bits: np.ndarray, B_bits: np.ndarray, SFA: np.ndarray, SFB: np.ndarray,
                M: int, N: int, K: int, dtype_in: str, rows=None, threads: int | None = None,
                lib=None):
    """FP64 reference rows of the block-scaled C = (SFA o A)(SFB o B) and its C_abs.

    A_bits: M x K bytes ("e4m3"/"e5m2") or M x ceil(K/2) bytes of packed E2M1
    ("e2m1", lower k in the low nibble). B_bits: N x K (K-major), same element
    layout. SFA: M x ceil(K/32), SFB: N x ceil(K/32) E8M0 bytes.
    """
    lib = lib or _load()
    width = (K + 1) // 2 if dtype_in == "e2m1" else K
    A = np.ascontiguousarray(A_bits, dtype=np.uint8)
    B = np.ascontiguousarray(B_bits, dtype=np.uint8)
    sa = np.ascontiguousarray(SFA, dtype=np.uint8)
    sb = np.ascontiguousarray(SFB, dtype=np.uint8)
    nb = mx_blocks(K)
    if A.size != M * width or B.size != N * width or sa.size != M * nb or sb.size != N * nb:
        raise ValueError("operand or scale sizes do not match M, N, K")
    if rows is None:
        n_rows, rows_ptr = M, None
    else:
        rows_arr = np.ascontiguousarray(rows, dtype=np.int64)
        n_rows = int(rows_arr.size)
        rows_ptr = rows_arr.ctypes.data_as(ctypes.c_void_p)
    C = np.empty((n_rows, N), dtype=np.float64)
    C_abs = np.empty((n_rows, N), dtype=np.float64)
    if n_rows == 0:
        return C, C_abs
    dp = ctypes.POINTER(ctypes.c_double)
    vp = ctypes.c_void_p
    rc = lib.oracle_gemm_mx(A.ctypes.data_as(vp), B.ctypes.data_as(vp), sa.ctypes.data_as(vp),
                            sb.ctypes.data_as(vp), M, N, K, _DTYPE[dtype_in], rows_ptr, n_rows,
                            C.ctypes.data_as(dp), C_abs.ctypes.data_as(dp),
                            int(threads or host_threads()))
    if rc != 0:
        raise RuntimeError(f"oracle_gemm_mx failed with code {rc}")
    return C, C_abs


def attention_ref(Q_bits, K_bits, V_bits, B: int, H: int, Lq: int, Lk: int, d: int, dtype: str,
                  causal: bool = False, scale: float | None = None, rows=None,
                  threads: int | None = None, lib=None):
    """FP64 attention forward rows: (O, O_abs, LSE) for the flat query rows
    r = (b*H + h)*Lq + i (None = all). Q_bits is [B][H][Lq][d], K_bits and
    V_bits [B][H][Lk][d], uint16 FP16/BF16 patterns. scale defaults to 1/sqrt(d).
    Follows "Two Waves, One Stage Apart", section "Beyond GEMM: FlashAttention"."""
    lib = lib or _load()
    Q = np.ascontiguousarray(Q_bits, dtype=np.uint16)
    K = np.ascontiguousarray(K_bits, dtype=np.uint16)
    V = np.ascontiguousarray(V_bits, dtype=np.uint16)
    if Q.size != B * H * Lq * d or K.size != B * H * Lk * d or V.size != B * H * Lk * d:
        raise ValueError("operand sizes do not match B, H, Lq, Lk, d")
    scale = 1.0 / np.sqrt(d) if scale is None else float(scale)
    if rows is None:
        n_rows, rows_ptr = B * H * Lq, None
    else:
        rows_arr = np.ascontiguousarray(rows, dtype=np.int64)
        n_rows = int(rows_arr.size)
        rows_ptr = rows_arr.ctypes.data_as(ctypes.c_void_p)
    O = np.empty((n_rows, d), dtype=np.float64)
    O_abs = np.empty((n_rows, d), dtype=np.float64)
    LSE = np.empty((n_rows,), dtype=np.float64)
    if n_rows == 0:
        return O, O_abs, LSE
    dp = ctypes.POINTER(ctypes.c_double)
    vp = ctypes.c_void_p
    rc = lib.oracle_attention(Q.ctypes.data_as(vp), K.ctypes.data_as(vp), V.ctypes.data_as(vp),
                              B, H, Lq, Lk, d, _DTYPE[dtype], int(bool(causal)), scale, rows_ptr,
                              n_rows, O.ctypes.data_as(dp), O_abs.ctypes.data_as(dp),
                              LSE.ctypes.data_as(dp), int(threads or host_threads()))
    if rc != 0:
        raise RuntimeError(f"oracle_attention failed with code {rc}")
    return O, O_abs, LSE
