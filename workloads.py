"""Seeded synthetic inputs for the dense GEMM C = A·B.

This module only draws random operands: it holds none of the GEMM's
arithmetic, so both the CPU oracle (``oracle/``) and the CUDA path
(``dense_tiled_gemm_gb300``) can be fed from it without sharing code.

Recipe (the pages fix no generator; this is the plain reading):
  * one CPU ``torch.Generator`` seeded with the workload's seed;
  * FP32 draws, A first and then B, each in its own storage order
    (A: M×K row-major; B K-major: N×K, K contiguous; B MN-major: K×N,
    N contiguous);
  * uniform[a, b] = a + (b − a)·rand, normal(0, σ) = σ·randn;
  * rounded to FP16/BF16 or FP8 (E4M3 "FN", E5M2) with round-to-nearest-even
    (``Tensor.to``); the draws stay well inside each type's finite range.

Block-scaled (MX) operands (``make_mx_operands``) are drawn already
quantised: elements as above (E2M1 rounds to nearest, ties to the even
code, and saturates at 6), packed two per byte for E2M1 (lower k in the low
nibble, rows padded to whole bytes), then E8M0 scale exponents drawn
uniformly from [127 - r, 127 + r], A's then B's, from the same generator.

The workloads are the five GEMM shapes the tiled-GEMM pages measure or that
exercise the method's edge paths (a small 256³ check, the compute-bound
4096×4096×8192 FP16 shape of "Two Waves, One Stage Apart", §"MI350 Series",
a BF16 8192³ shape, a ragged 3000×5000×2050 shape with N-contiguous B, and
a square FP16 sweep), plus the FP8 E4M3 squares of "Porting
High-Performance HIP Kernels to FlyDSL", section "Results" (8192 and 12288,
normally distributed data; the page does not give C's type, BF16 is taken).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

DTYPES = {"f16": torch.float16, "bf16": torch.bfloat16, "f32": torch.float32,
          "e4m3": torch.float8_e4m3fn, "e5m2": torch.float8_e5m2}
FP8 = ("e4m3", "e5m2")
MX_ELEMENT = {"mxfp8": "e4m3", "mxfp8_e5m2": "e5m2", "mxfp4": "e2m1"}   # MX type -> element type
MX_BLOCK = 32


@dataclass(frozen=True)
class Workload:
    name: str
    M: int
    N: int
    K: int
    dtype_in: str          # "f16" | "bf16" | "e4m3" | "e5m2"
    dtype_out: str         # "f16" | "bf16" | "f32"
    layout_b: str          # "k": B stored N×K (K contiguous); "mn": B stored K×N
    dist: tuple            # ("uniform", lo, hi) | ("normal", sigma) | ("int", lo, hi)
    seed: int
    note: str = field(default="", compare=False)

    @property
    def flops(self) -> int:
        return 2 * self.M * self.N * self.K


def _sweep():
    out = []
    for i, n in enumerate((1024, 2048, 4096, 8192, 16384)):
        out.append(Workload(f"square_f16_{n}", n, n, n, "f16", "f16", "k",
                            ("normal", 1.0), 4 + i, "square FP16 sweep"))
    return out


WORKLOADS = {w.name: w for w in [
    Workload("gemm_256_f16_f32", 256, 256, 256, "f16", "f32", "k",
             ("uniform", -1.0, 1.0), 0, "small check"),
    Workload("gemm_4096x4096x8192_f16", 4096, 4096, 8192, "f16", "f16", "k",
             ("normal", 1.0), 1, "compute-bound headline shape"),
    Workload("gemm_8192_bf16", 8192, 8192, 8192, "bf16", "bf16", "k",
             ("normal", 1.0 / math.sqrt(8192)), 2, "BF16 square"),
    Workload("gemm_3000x5000x2050_bf16_f32_bmn", 3000, 5000, 2050, "bf16", "f32", "mn",
             ("uniform", -2.0, 2.0), 3, "ragged tails, N-contiguous B"),
] + _sweep() + [
    Workload("gemm_8192_e4m3", 8192, 8192, 8192, "e4m3", "bf16", "k",
             ("normal", 1.0), 9, "FP8 E4M3 square"),
    Workload("gemm_12288_e4m3", 12288, 12288, 12288, "e4m3", "bf16", "k",
             ("normal", 1.0), 10, "FP8 E4M3 square"),
    Workload("gemm_4096x4096x65536_mxfp8", 4096, 4096, 65536, "mxfp8", "bf16", "k",
             ("normal", 1.0), 11, "MXFP8, long K"),
    Workload("gemm_4096x4096x65536_mxfp4", 4096, 4096, 65536, "mxfp4", "bf16", "k",
             ("normal", 2.0), 12, "MXFP4, long K"),
]}
MX_SCALE_RANGE = 3      # scale exponents 2^-3 .. 2^3 around 1.0

HEADLINE = "gemm_4096x4096x8192_f16"


def _draw(gen: torch.Generator, n: int, dist: tuple) -> torch.Tensor:
    kind = dist[0]
    if kind == "uniform":
        lo, hi = dist[1], dist[2]
        return lo + (hi - lo) * torch.rand(n, generator=gen, dtype=torch.float32)
    if kind == "normal":
        return dist[1] * torch.randn(n, generator=gen, dtype=torch.float32)
    if kind == "int":
        lo, hi = dist[1], dist[2]
        return torch.randint(lo, hi + 1, (n,), generator=gen).to(torch.float32)
    raise ValueError(f"unknown distribution {dist!r}")


def b_shape(M: int, N: int, K: int, layout_b: str) -> tuple:
    """Storage shape of B for a layout: (N, K) when K-major, (K, N) when MN-major."""
    if layout_b == "k":
        return (N, K)
    if layout_b == "mn":
        return (K, N)
    raise ValueError(f"layout_b must be 'k' or 'mn', got {layout_b!r}")


def make_operands(M: int, N: int, K: int, dtype_in: str, layout_b: str,
                  dist: tuple, seed: int) -> tuple[torch.Tensor, torch.Tensor]:
    """Return CPU tensors (A, B) in storage layout, rounded to ``dtype_in``."""
    gen = torch.Generator().manual_seed(int(seed))
    dt = DTYPES[dtype_in]
    A = _draw(gen, M * K, dist).to(dt).reshape(M, K)
    B = _draw(gen, N * K, dist).to(dt).reshape(b_shape(M, N, K, layout_b))
    return A, B


def workload_operands(w: Workload):
    """(A, B) for plain workloads, (A, B, SFA, SFB) for block-scaled (MX) ones."""
    if w.dtype_in in MX_ELEMENT:
        return make_mx_operands(w.M, w.N, w.K, w.dtype_in, w.dist, w.seed)
    return make_operands(w.M, w.N, w.K, w.dtype_in, w.layout_b, w.dist, w.seed)


# E2M1 codes 0..7 have magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6. Between codes c and
# c + 1 the midpoint rounds to the even code: up when c is odd, down when c is even.
_E2M1_MIDPOINTS = ((0.25, False), (0.75, True), (1.25, False), (1.75, True), (2.5, False),
                   (3.5, True), (5.0, False))   # (midpoint, a tie rounds up)


def round_e2m1(x: torch.Tensor) -> torch.Tensor:
    """FP32 values -> E2M1 codes (uint8, 0..15): nearest magnitude, ties to the
    even code, saturating at 6; sign in bit 3 (never on zero)."""
    mag = x.abs()
    code = torch.zeros(x.shape, dtype=torch.uint8)
    for mid, tie_up in _E2M1_MIDPOINTS:
        code += (mag >= mid if tie_up else mag > mid).to(torch.uint8)
    return code | ((x < 0) & (code != 0)).to(torch.uint8) << 3


def pack_e2m1(codes: torch.Tensor) -> torch.Tensor:
    """rows x K codes -> rows x ceil(K/2) bytes, lower k in the low nibble."""
    rows, K = codes.shape
    if K % 2:
        codes = torch.cat([codes, torch.zeros((rows, 1), dtype=torch.uint8)], dim=1)
    return (codes[:, 0::2] | (codes[:, 1::2] << 4)).contiguous()


def make_mx_operands(M: int, N: int, K: int, mx_type: str, dist: tuple, seed: int,
                     scale_range: int = MX_SCALE_RANGE):
    """CPU tensors (A, B, SFA, SFB) of a block-scaled GEMM.

    A: M x K float8 (MXFP8) or M x ceil(K/2) uint8 of packed E2M1 (MXFP4);
    B: N x K (K-major), same element layout. SFA: M x ceil(K/32), SFB:
    N x ceil(K/32) uint8 E8M0 scale exponents."""
    gen = torch.Generator().manual_seed(int(seed))
    elem = MX_ELEMENT[mx_type]
    a = _draw(gen, M * K, dist).reshape(M, K)
    b = _draw(gen, N * K, dist).reshape(N, K)
    if elem == "e2m1":
        A, B = pack_e2m1(round_e2m1(a)), pack_e2m1(round_e2m1(b))
    else:
        A, B = a.to(DTYPES[elem]), b.to(DTYPES[elem])
    nb = (K + MX_BLOCK - 1) // MX_BLOCK
    lo, hi = 127 - scale_range, 127 + scale_range
    SFA = torch.randint(lo, hi + 1, (M, nb), generator=gen).to(torch.uint8)
    SFB = torch.randint(lo, hi + 1, (N, nb), generator=gen).to(torch.uint8)
    return A, B, SFA, SFB


def as_bits(t: torch.Tensor):
    """Raw patterns of a CPU tensor: numpy uint16 for FP16/BF16, uint8 for FP8 and
    for byte tensors (packed E2M1, E8M0 scales)."""
    import numpy as np
    assert t.device.type == "cpu"
    if t.dtype in (torch.float16, torch.bfloat16):
        return t.contiguous().view(torch.int16).numpy().view(np.uint16)
    assert t.dtype in (torch.float8_e4m3fn, torch.float8_e5m2, torch.uint8), t.dtype
    return t.contiguous().view(torch.uint8).numpy()


def sample_rows(M: int, count: int, seed: int, tile: int = 128) -> list[int]:
    """Rows to check at full size: both edges of every ``tile``-row block
    (up to ``count``), the last row, and seeded random rows."""
    g = torch.Generator().manual_seed(10_000 + int(seed))
    rows = {0, M - 1}
    for b in range(0, M, tile):
        rows.add(b)
        rows.add(min(M - 1, b + tile - 1))
        if len(rows) >= count // 2:
            break
    extra = torch.randint(0, M, (count,), generator=g).tolist()
    for r in extra:
        if len(rows) >= count:
            break
        rows.add(int(r))
    return sorted(rows)


# ---------------------------------------------------------------------------- attention
@dataclass(frozen=True)
class AttentionWorkload:
    """Attention forward O = softmax(scale Q K^T) V over B x H heads."""
    name: str
    B: int
    H: int
    Lq: int
    Lk: int
    d: int
    dtype: str          # "f16" | "bf16"
    causal: bool
    dist: tuple
    seed: int
    note: str = field(default="", compare=False)

    @property
    def flops(self) -> int:
        """Two products of 2 * Lq * Lk * d per head; a causal mask keeps the visible half."""
        full = 4 * self.B * self.H * self.Lq * self.Lk * self.d
        if not self.causal:
            return full
        # visible (query, key) pairs: row i sees min(Lk, i + Lk - Lq + 1) keys
        off = self.Lk - self.Lq
        seen = sum(max(0, min(self.Lk, i + off + 1)) for i in range(self.Lq))
        return 4 * self.B * self.H * seen * self.d


ATTENTION_WORKLOADS = {w.name: w for w in [
    AttentionWorkload("attention_4x16x4096x128_bf16", 4, 16, 4096, 4096, 128, "bf16", False,
                      ("normal", 1.0), 20, "attention forward, long sequence"),
    AttentionWorkload("attention_4x16x4096x128_bf16_causal", 4, 16, 4096, 4096, 128, "bf16", True,
                      ("normal", 1.0), 21, "attention forward, causal"),
]}


def make_attention_operands(B: int, H: int, Lq: int, Lk: int, d: int, dtype: str, dist: tuple,
                            seed: int):
    """CPU tensors Q (B, H, Lq, d), K and V (B, H, Lk, d), drawn Q, K, V in that order."""
    gen = torch.Generator().manual_seed(int(seed))
    dt = DTYPES[dtype]
    Q = _draw(gen, B * H * Lq * d, dist).to(dt).reshape(B, H, Lq, d)
    K = _draw(gen, B * H * Lk * d, dist).to(dt).reshape(B, H, Lk, d)
    V = _draw(gen, B * H * Lk * d, dist).to(dt).reshape(B, H, Lk, d)
    return Q, K, V
