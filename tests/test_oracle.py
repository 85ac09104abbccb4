"""Pins for the CPU FP64 oracle (no GPU).

The oracle is checked against things other than itself: the IEEE/bfloat16/
OCP FP8 format definitions (hand-written fixtures), numpy's and torch's own
FP16/BF16/FP8 conversions, the bit-level identity E5M2 = upper byte of FP16,
exact rational arithmetic (``fractions``) on tiny shapes, closed
forms (identity, all-ones, rank-1), exact integer arithmetic, and
``torch.matmul`` in float64. ``test_planted_mistakes`` compiles copies of the
oracle with one deliberate bug each and requires every copy to fail at least
one of these pins.
"""
from __future__ import annotations

import math
import os
import subprocess
import sys
import tempfile
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from oracle import tolerance

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
U = 2.0 ** -53
DTYPES = ("f16", "bf16", "e4m3", "e5m2")
FP8_TORCH = {"e4m3": torch.float8_e4m3fn, "e5m2": torch.float8_e5m2}


# ---------------------------------------------------------------- helpers
def f16_bits(vals) -> np.ndarray:
    return np.asarray(vals, dtype=np.float64).astype(np.float16).view(np.uint16)


def bf16_bits(vals) -> np.ndarray:
    t = torch.tensor(np.asarray(vals, dtype=np.float64), dtype=torch.float64).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def fp8_bits(vals, dtype) -> np.ndarray:
    t = torch.tensor(np.asarray(vals, dtype=np.float64), dtype=torch.float64)
    return t.to(torch.float32).to(FP8_TORCH[dtype]).view(torch.uint8).numpy()


def bits_of(vals, dtype):
    if dtype in FP8_TORCH:
        return fp8_bits(vals, dtype)
    return f16_bits(vals) if dtype == "f16" else bf16_bits(vals)


def exact_value(bits: int, dtype: str) -> float:
    """FP64 value of a pattern via numpy/torch conversions (not the oracle's decoder)."""
    if dtype == "f16":
        return float(np.array([bits], dtype=np.uint16).view(np.float16)[0])
    if dtype in FP8_TORCH:
        return float(torch.tensor([bits], dtype=torch.uint8).view(FP8_TORCH[dtype]).double()[0])
    return float(np.array([bits << 16], dtype=np.uint32).view(np.float32)[0])


def random_finite_bits(rng: np.random.Generator, n: int, dtype: str) -> np.ndarray:
    """Finite patterns with every exponent represented, subnormals included."""
    if dtype == "e4m3":
        # every byte but the two NaNs (S.1111.111)
        low = rng.integers(0, 127, n)
        return (low | (rng.integers(0, 2, n) << 7)).astype(np.uint8)
    if dtype == "e5m2":
        e = rng.integers(0, 31, n)
        f = rng.integers(0, 4, n)
        return ((e << 2) | f | (rng.integers(0, 2, n) << 7)).astype(np.uint8)
    if dtype == "f16":
        e = rng.integers(0, 31, n)
        f = rng.integers(0, 1024, n)
        word = (e << 10) | f
    else:
        e = rng.integers(0, 255, n)
        f = rng.integers(0, 128, n)
        word = (e << 7) | f
    sign = rng.integers(0, 2, n) << 15
    return (word | sign).astype(np.uint16)


def b_storage(Bkn: np.ndarray, layout_b: str) -> np.ndarray:
    """Store a K×N matrix of patterns in the requested B layout."""
    return np.ascontiguousarray(Bkn.T if layout_b == "k" else Bkn)


def gamma(K: int) -> float:
    """Bound on FP64 sequential-summation error relative to sum |terms|."""
    return K * U / (1 - K * U)


# ---------------------------------------------------------------- pin battery
def _pin_decoders(lib):
    allbits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    out = []
    for dtype in ("f16", "bf16"):
        mine = oracle.decode(allbits, dtype, lib=lib)
        if dtype == "f16":
            ref = allbits.view(np.float16).astype(np.float64)
        else:
            with np.errstate(invalid="ignore"):
                ref = (allbits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
        same = (mine == ref) | (np.isnan(mine) & np.isnan(ref))
        if not same.all():
            out.append(f"decoder_{dtype}")
    bytes_ = np.arange(256, dtype=np.uint32).astype(np.uint8)
    for dtype, tdt in FP8_TORCH.items():
        mine = oracle.decode(bytes_, dtype, lib=lib)
        ref = torch.from_numpy(bytes_.copy()).view(tdt).double().numpy()
        same = (mine == ref) | (np.isnan(mine) & np.isnan(ref))
        if not same.all():
            out.append(f"decoder_{dtype}")
    # E5M2 is the upper byte of an FP16 pattern (same sign and exponent fields)
    e5 = oracle.decode(bytes_, "e5m2", lib=lib)
    f16 = oracle.decode(bytes_.astype(np.uint16) << 8, "f16", lib=lib)
    if not ((e5 == f16) | (np.isnan(e5) & np.isnan(f16))).all():
        out.append("decoder_e5m2_vs_f16")
    return out


def _parse_format_fixture(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as fh:
        for line in fh:
            line = line.split("#")[0].strip()
            if not line:
                continue
            bits, mant, expo = line.split()[:3]
            if mant in ("inf", "-inf", "nan"):
                val = float(mant)
            else:
                val = math.ldexp(float(int(mant)), int(expo))
            rows.append((int(bits, 16), val))
    return rows


def _pin_format_fixtures(lib):
    out = []
    for name, dtype in (("binary16_values.txt", "f16"), ("bfloat16_values.txt", "bf16"),
                        ("e4m3_values.txt", "e4m3"), ("e5m2_values.txt", "e5m2")):
        for bits, val in _parse_format_fixture(name):
            got = float(oracle.decode(np.array([bits]), dtype, lib=lib)[0])
            if not (got == val or (math.isnan(got) and math.isnan(val))):
                out.append(f"fixture_{dtype}_{bits:#06x}")
    return out


def _parse_gemm_fixture():
    cases, cur, key = [], None, None
    with open(os.path.join(GOLDEN, "gemm_hand_2x2.txt")) as fh:
        for line in fh:
            line = line.split("#")[0].strip()
            if not line:
                continue
            tok = line.split()
            if tok[0] == "case":
                cur = {"name": tok[1], "dtypes": tuple(tok[2:]) or DTYPES}
                cases.append(cur)
            elif tok[0] in ("A", "B", "C", "C_abs"):
                key = tok[0]
                cur[key] = []
            else:
                cur[key].append([float(t) for t in tok])
    return [{k: (np.array(v) if k not in ("name", "dtypes") else v) for k, v in c.items()}
            for c in cases]


def _pin_hand_gemm(lib):
    out = []
    for case in _parse_gemm_fixture():
        A, Bkn, C, Cabs = case["A"], case["B"], case["C"], case["C_abs"]
        M, K = A.shape
        N = Bkn.shape[1]
        for dtype in case["dtypes"]:
            for lay in ("k", "mn"):
                got, gabs = oracle.gemm_ref(bits_of(A, dtype), b_storage(bits_of(Bkn, dtype), lay),
                                            M, N, K, dtype, lay, lib=lib)
                if not (np.array_equal(got, C) and np.array_equal(gabs, Cabs)):
                    out.append(f"hand_{case['name']}_{dtype}_{lay}")
    return out


def _pin_brute_force(lib):
    out = []
    rng = np.random.default_rng(1234)
    for (M, N, K) in ((1, 1, 1), (2, 3, 4), (5, 7, 3), (17, 9, 33)):
        for dtype in DTYPES:
            for lay in ("k", "mn"):
                Ab = random_finite_bits(rng, M * K, dtype).reshape(M, K)
                Bkn = random_finite_bits(rng, K * N, dtype).reshape(K, N)
                got, gabs = oracle.gemm_ref(Ab, b_storage(Bkn, lay), M, N, K, dtype, lay, lib=lib)
                av = [[Fraction(exact_value(int(x), dtype)) for x in row] for row in Ab]
                bv = [[Fraction(exact_value(int(x), dtype)) for x in row] for row in Bkn]
                for i in range(M):
                    for j in range(N):
                        terms = [av[i][k] * bv[k][j] for k in range(K)]
                        ex = sum(terms)
                        ea = sum(abs(t) for t in terms)
                        lim = gamma(K) * float(ea)
                        if abs(Fraction(got[i, j]) - ex) > Fraction(lim):
                            out.append(f"brute_{M}x{N}x{K}_{dtype}_{lay}")
                            break
                        if abs(Fraction(gabs[i, j]) - ea) > Fraction(lim):
                            out.append(f"brute_abs_{M}x{N}x{K}_{dtype}_{lay}")
                            break
                    else:
                        continue
                    break
    return out


def _pin_closed_forms(lib):
    out = []
    rng = np.random.default_rng(7)
    for dtype in DTYPES:
        for lay in ("k", "mn"):
            # identity B (N = K): C = A exactly
            M, K = 13, 24
            Ab = random_finite_bits(rng, M * K, dtype).reshape(M, K)
            eye = bits_of(np.eye(K), dtype)
            got, _ = oracle.gemm_ref(Ab, b_storage(eye, lay), M, K, K, dtype, lay, lib=lib)
            ref = np.vectorize(lambda b: exact_value(int(b), dtype))(Ab)
            if not np.array_equal(got, ref):
                out.append(f"identity_{dtype}_{lay}")
            # all-ones A: C[i][j] = column sum of B (math.fsum is correctly rounded)
            M, N, K = 3, 11, 40
            vals = rng.uniform(-4, 4, (K, N))
            Bkn = bits_of(vals, dtype)
            ones = bits_of(np.ones((M, K)), dtype)
            got, gabs = oracle.gemm_ref(ones, b_storage(Bkn, lay), M, N, K, dtype, lay, lib=lib)
            bv = np.vectorize(lambda b: exact_value(int(b), dtype))(Bkn)
            for j in range(N):
                col = math.fsum(bv[:, j])
                lim = 2 * gamma(K) * float(np.abs(bv[:, j]).sum())
                if np.any(np.abs(got[:, j] - col) > lim):
                    out.append(f"ones_{dtype}_{lay}")
                    break
            # rank-1: a[i][k] = u_i, b[k][j] = v_j gives K * u_i * v_j exactly
            M, N, K = 6, 5, 37
            u = bits_of(rng.uniform(-3, 3, M), dtype)
            v = bits_of(rng.uniform(-3, 3, N), dtype)
            Ab = np.repeat(u[:, None], K, axis=1)
            Bkn = np.repeat(v[None, :], K, axis=0)
            got, _ = oracle.gemm_ref(Ab, b_storage(Bkn, lay), M, N, K, dtype, lay, lib=lib)
            uv = np.array([exact_value(int(b), dtype) for b in u])
            vv = np.array([exact_value(int(b), dtype) for b in v])
            if not np.array_equal(got, K * np.outer(uv, vv)):
                out.append(f"rank1_{dtype}_{lay}")
    return out


def _pin_integers(lib):
    """Small integers: every partial sum is exact, so C equals int64 matmul."""
    out = []
    rng = np.random.default_rng(11)
    for dtype in DTYPES:
        for lay in ("k", "mn"):
            M, N, K = 19, 23, 300
            Ai = rng.integers(-3, 4, (M, K))
            Bi = rng.integers(-3, 4, (K, N))
            got, gabs = oracle.gemm_ref(bits_of(Ai, dtype), b_storage(bits_of(Bi, dtype), lay),
                                        M, N, K, dtype, lay, lib=lib)
            if not (np.array_equal(got, (Ai @ Bi).astype(np.float64))
                    and np.array_equal(gabs, (np.abs(Ai) @ np.abs(Bi)).astype(np.float64))):
                out.append(f"integer_{dtype}_{lay}")
    return out


def _pin_torch_matmul(lib):
    out = []
    g = torch.Generator().manual_seed(5)
    for dtype, tdt in (("f16", torch.float16), ("bf16", torch.bfloat16)) + tuple(FP8_TORCH.items()):
        for lay in ("k", "mn"):
            M, N, K = 40, 33, 200
            A = torch.randn(M, K, generator=g).to(tdt)
            Bkn = torch.randn(K, N, generator=g).to(tdt)
            ref = (A.double() @ Bkn.double()).numpy()
            refabs = (A.double().abs() @ Bkn.double().abs()).numpy()
            view = torch.uint8 if dtype in FP8_TORCH else torch.int16
            Ab = A.view(view).numpy()
            Bb = Bkn.contiguous().view(view).numpy()
            if view is torch.int16:
                Ab, Bb = Ab.view(np.uint16), Bb.view(np.uint16)
            got, gabs = oracle.gemm_ref(Ab, b_storage(Bb, lay), M, N, K, dtype, lay, lib=lib)
            lim = 2 * gamma(K) * refabs
            if np.any(np.abs(got - ref) > lim) or np.any(np.abs(gabs - refabs) > lim):
                out.append(f"torch_{dtype}_{lay}")
    return out


def _pin_row_subset(lib):
    out = []
    rng = np.random.default_rng(3)
    M, N, K = 21, 10, 17
    for dtype in DTYPES:
        Ab = random_finite_bits(rng, M * K, dtype).reshape(M, K)
        Bb = random_finite_bits(rng, K * N, dtype).reshape(N, K)
        full, fabs_ = oracle.gemm_ref(Ab, Bb, M, N, K, dtype, "k", lib=lib)
        rows = [20, 0, 7, 7, 13]
        part, pabs = oracle.gemm_ref(Ab, Bb, M, N, K, dtype, "k", rows=rows, lib=lib)
        same = (part == full[rows]) | (np.isnan(part) & np.isnan(full[rows]))
        if not same.all() or not np.array_equal(pabs, fabs_[rows]):
            out.append(f"rows_{dtype}")
    return out


# ---------------------------------------------------------------- block-scaled (MX) pins
E2M1_TABLE = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]   # magnitudes of codes 0..7 (OCP E2M1)
MX_TYPES = ("e4m3", "e5m2", "e2m1")


def e2m1_value(code: int) -> float:
    v = E2M1_TABLE[code & 7]
    return -v if code & 8 else v


def pack_e2m1(codes: np.ndarray) -> np.ndarray:
    """Rows of 4-bit codes -> bytes, two per byte, lower k in the low nibble (odd K padded)."""
    rows, K = codes.shape
    padded = np.zeros((rows, K + (K & 1)), dtype=np.uint8)
    padded[:, :K] = codes
    return (padded[:, 0::2] | (padded[:, 1::2] << 4)).astype(np.uint8)


def random_mx_elements(rng, rows, K, dtype):
    """(storage array, exact values) for random finite elements of an MX type."""
    if dtype == "e2m1":
        codes = rng.integers(0, 16, (rows, K)).astype(np.uint8)
        return pack_e2m1(codes), np.vectorize(e2m1_value)(codes)
    bits = random_finite_bits(rng, rows * K, dtype).reshape(rows, K)
    return bits, np.vectorize(lambda b: exact_value(int(b), dtype))(bits)


def _pin_mx_fixtures(lib):
    out = []
    for name, dtype in (("e2m1_values.txt", "e2m1"), ("e8m0_values.txt", "e8m0")):
        for bits, val in _parse_format_fixture(name):
            got = float(oracle.decode(np.array([bits]), dtype, lib=lib)[0])
            if not (got == val or (math.isnan(got) and math.isnan(val))):
                out.append(f"fixture_{dtype}_{bits:#04x}")
    e8 = oracle.decode(np.arange(255), "e8m0", lib=lib)
    if not all(e8[e] == math.ldexp(1.0, e - 127) for e in range(255)):
        out.append("decoder_e8m0")
    e2 = oracle.decode(np.arange(16), "e2m1", lib=lib)
    if not all(e2[c] == e2m1_value(c) for c in range(16)):
        out.append("decoder_e2m1")
    return out


def _pin_mx_brute_force(lib):
    """Random elements and scales on tiny shapes, K across block edges and odd
    (E2M1 rows padded), against exact Fraction sums of the scaled products."""
    out = []
    rng = np.random.default_rng(77)
    for (M, N, K) in ((1, 1, 1), (2, 3, 33), (3, 2, 64), (4, 5, 65), (2, 2, 97)):
        nb = oracle.mx_blocks(K)
        for dtype in MX_TYPES:
            Ast, Av = random_mx_elements(rng, M, K, dtype)
            Bst, Bv = random_mx_elements(rng, N, K, dtype)
            sfa = rng.integers(110, 145, (M, nb)).astype(np.uint8)
            sfb = rng.integers(110, 145, (N, nb)).astype(np.uint8)
            got, gabs = oracle.gemm_ref_mx(Ast, Bst, sfa, sfb, M, N, K, dtype, lib=lib)
            for i in range(M):
                for j in range(N):
                    terms = [Fraction(Av[i, k]) * Fraction(2) ** (int(sfa[i, k // 32]) - 127)
                             * Fraction(Bv[j, k]) * Fraction(2) ** (int(sfb[j, k // 32]) - 127)
                             for k in range(K)]
                    ex, ea = sum(terms), sum(abs(t) for t in terms)
                    lim = Fraction(gamma(K) * float(ea))
                    if abs(Fraction(got[i, j]) - ex) > lim or abs(Fraction(gabs[i, j]) - ea) > lim:
                        out.append(f"mx_brute_{M}x{N}x{K}_{dtype}")
                        break
                else:
                    continue
                break
    return out


def _pin_mx_unit_scales(lib):
    """Scales of 1.0 (E8M0 127) reduce the MX GEMM to the plain FP8 GEMM, bit for bit."""
    out = []
    rng = np.random.default_rng(78)
    M, N, K = 9, 7, 100
    for dtype in ("e4m3", "e5m2"):
        A = random_finite_bits(rng, M * K, dtype).reshape(M, K)
        B = random_finite_bits(rng, N * K, dtype).reshape(N, K)
        ones_a = np.full((M, oracle.mx_blocks(K)), 127, np.uint8)
        ones_b = np.full((N, oracle.mx_blocks(K)), 127, np.uint8)
        mx, mxa = oracle.gemm_ref_mx(A, B, ones_a, ones_b, M, N, K, dtype, lib=lib)
        plain, pa = oracle.gemm_ref(A, B, M, N, K, dtype, "k", lib=lib)
        if not (np.array_equal(mx, plain) and np.array_equal(mxa, pa)):
            out.append(f"mx_unit_scales_{dtype}")
    return out


def _pin_mx_block_scaling(lib):
    """Closed form: raising one row's scale for one 32-block by 2^t adds
    (2^t - 1) times that block's partial sum, and a column scale scales the
    whole column; with small integers every sum is exact."""
    out = []
    rng = np.random.default_rng(79)
    M, N, K = 4, 6, 96
    for dtype in MX_TYPES:
        ints = rng.integers(-3, 4, (M, K)).astype(np.float64)
        intb = rng.integers(-3, 4, (N, K)).astype(np.float64)
        if dtype == "e2m1":
            enc = {0: 0, 1: 2, 2: 4, 3: 5, -1: 10, -2: 12, -3: 13}
            Ast = pack_e2m1(np.vectorize(enc.get)(ints.astype(int)).astype(np.uint8))
            Bst = pack_e2m1(np.vectorize(enc.get)(intb.astype(int)).astype(np.uint8))
        else:
            Ast, Bst = bits_of(ints, dtype), bits_of(intb, dtype)
        nb = oracle.mx_blocks(K)
        sfa = np.full((M, nb), 127, np.uint8)
        sfb = np.full((N, nb), 127, np.uint8)
        base, _ = oracle.gemm_ref_mx(Ast, Bst, sfa, sfb, M, N, K, dtype, lib=lib)
        sfa2 = sfa.copy()
        sfa2[2, 1] = 127 + 3                       # row 2, k in [32, 64): x 8
        sfb2 = sfb.copy()
        sfb2[4, :] = 127 - 2                       # column 4: x 1/4
        got, _ = oracle.gemm_ref_mx(Ast, Bst, sfa2, sfb2, M, N, K, dtype, lib=lib)
        expect = base.copy()
        expect[2, :] += 7 * (ints[2, 32:64] @ intb[:, 32:64].T)
        expect[:, 4] *= 0.25
        if not np.array_equal(got, expect):
            out.append(f"mx_block_scaling_{dtype}")
    return out


def _pin_mx_nibble_order(lib):
    """E2M1 packing: code 2 (1.0) at k = 0 of row 0 sits in the low nibble of
    byte 0; at k = 1 in the high nibble. A one-hot row picks one k of B."""
    out = []
    K, N = 8, 3
    for k_hot in (0, 1, 6, 7):
        codes_a = np.zeros((1, K), np.uint8)
        codes_a[0, k_hot] = 2
        codes_b = (np.arange(N * K).reshape(N, K) % 8).astype(np.uint8)
        sf = np.full((1, 1), 127, np.uint8)
        got, _ = oracle.gemm_ref_mx(pack_e2m1(codes_a), pack_e2m1(codes_b), sf,
                                    np.full((N, 1), 127, np.uint8), 1, N, K, "e2m1", lib=lib)
        if not np.array_equal(got[0], [E2M1_TABLE[c] for c in codes_b[:, k_hot]]):
            out.append(f"mx_nibble_{k_hot}")
    return out


PINS = [_pin_decoders, _pin_format_fixtures, _pin_hand_gemm, _pin_brute_force,
        _pin_closed_forms, _pin_integers, _pin_torch_matmul, _pin_row_subset,
        _pin_mx_fixtures, _pin_mx_brute_force, _pin_mx_unit_scales, _pin_mx_block_scaling,
        _pin_mx_nibble_order]


def pin_battery(lib):
    failed = []
    for pin in PINS:
        try:
            failed += pin(lib)
        except Exception as exc:  # a crash in a mutant counts as a caught mistake
            failed.append(f"{pin.__name__}: {type(exc).__name__}")
    return failed


# ---------------------------------------------------------------- tests
@pytest.fixture(scope="module")
def lib():
    return oracle._load()


@pytest.mark.parametrize("pin", PINS, ids=lambda p: p.__name__[5:])
def test_pin(lib, pin):
    assert pin(lib) == []


def test_argument_errors(lib):
    import ctypes
    dp = ctypes.POINTER(ctypes.c_double)
    a = np.zeros(4, dtype=np.uint16)
    c = np.zeros(4)
    args = (a.ctypes.data_as(ctypes.c_void_p), a.ctypes.data_as(ctypes.c_void_p))
    out = (c.ctypes.data_as(dp), c.ctypes.data_as(dp))
    assert lib.oracle_gemm(*args, 0, 2, 2, 0, 0, None, 0, *out, 1) == -1       # M = 0
    assert lib.oracle_gemm(*args, 2, 2, 2, 5, 0, None, 0, *out, 1) == -1       # bad dtype
    assert lib.oracle_gemm(*args, 2, 2, 2, 0, 9, None, 0, *out, 1) == -1       # bad layout
    bad_rows = np.array([2], dtype=np.int64)                                     # row >= M
    assert lib.oracle_gemm(*args, 2, 2, 2, 0, 0, bad_rows.ctypes.data_as(ctypes.c_void_p),
                           1, *out, 1) == -1


def test_threads_do_not_change_bits(lib):
    rng = np.random.default_rng(9)
    M, N, K = 37, 29, 64
    Ab = random_finite_bits(rng, M * K, "f16").reshape(M, K)
    Bb = random_finite_bits(rng, K * N, "f16").reshape(N, K)
    c1, a1 = oracle.gemm_ref(Ab, Bb, M, N, K, "f16", "k", threads=1)
    c8, a8 = oracle.gemm_ref(Ab, Bb, M, N, K, "f16", "k", threads=8)
    assert np.array_equal(np.nan_to_num(c1), np.nan_to_num(c8)) and np.array_equal(a1, a8)


# Each entry plants one plausible mistake in a copy of the oracle's source.
MUTANTS = {
    "dropped_term": ("for (int64_t k = 0; k < K; ++k) {", "for (int64_t k = 1; k < K; ++k) {"),
    "transposed_b": ("j->layout_b == ORACLE_K_MAJOR ? c * j->row_elems + k : k * j->N + c",
                     "j->layout_b == ORACLE_K_MAJOR ? k * j->N + c : k * j->N + c"),
    "wrong_sign": ("c[col] += p;", "c[col] -= p;"),
    "f16_bias": ("e - 25", "e - 24"),
    "f16_subnormal": ("ldexp((double)f, -24)", "ldexp((double)f, -25)"),
    "bf16_bias": ("e - 134", "e - 133"),
    "bf16_hidden_bit": ("(double)(128 + f)", "(double)(f)"),
    "abs_dropped": ("cabs[col] += fabs(p);", "cabs[col] += p;"),
    "row_map_ignored": ("j->rows ? j->rows[r] : r", "r"),
    "a_index_reversed": ("decode(j->A, i * j->row_elems + k, j->dtype)",
                         "decode(j->A, i * j->row_elems + (K - 1 - k), j->dtype)"),
    "e4m3_bias": ("e - 10", "e - 11"),
    "e4m3_subnormal": ("ldexp((double)f, -9)", "ldexp((double)f, -10)"),
    "e4m3_top_binade_as_nan": ("e == 0xf && f == 0x7", "e == 0xf"),
    "e4m3_fraction_width": ("int f = h & 0x7;", "int f = h & 0x3;"),
    "e5m2_bias": ("e - 17", "e - 16"),
    "e5m2_hidden_bit": ("(double)(4 + f)", "(double)(8 + f)"),
    "e2m1_bias": ("ldexp((double)(2 + f), e - 2)", "ldexp((double)(2 + f), e - 1)"),
    "e2m1_subnormal": ("ldexp((double)f, -1) :", "ldexp((double)f, 0) :"),
    "e2m1_nibble_order": ("(idx & 1) ? (uint8_t)(byte >> 4) : (uint8_t)(byte & 0xF)",
                          "(idx & 1) ? (uint8_t)(byte & 0xF) : (uint8_t)(byte >> 4)"),
    "e2m1_row_pitch": ("dtype == ORACLE_E2M1 ? (K + 1) / 2 * 2 : K", "K"),
    "e8m0_bias": ("ldexp(1.0, (int)e - 127)", "ldexp(1.0, (int)e - 128)"),
    "mx_scale_a_ignored": ("if (j->sfa)", "if (!j->sfa)"),
    "mx_scale_b_wrong_row": ("j->sfb[c * j->n_blocks", "j->sfb[0 * j->n_blocks"),
    "mx_block_size": ("enum { ORACLE_MX_BLOCK = 32 };", "enum { ORACLE_MX_BLOCK = 64 };"),
    "fp8_read_as_16bit": ("case ORACLE_E4M3: return oracle_decode_e4m3(((const uint8_t *)base)[idx]);",
                          "case ORACLE_E4M3: return oracle_decode_e4m3((uint8_t)((const uint16_t *)base)[idx]);"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistakes(name, tmp_path):
    src = open(oracle._SRC).read()
    old, new = MUTANTS[name]
    assert src.count(old) == 1, f"mutation anchor for {name} not unique"
    path = tmp_path / "mutant.c"
    path.write_text(src.replace(old, new))
    so = tmp_path / "libmutant.so"
    subprocess.run(oracle.compile_cmd(str(so), (str(path), oracle._ATT_SRC)), check=True)
    # The battery runs in a child process: a mutant that reads out of bounds may
    # crash, and a crash counts as a caught mistake.
    here = os.path.dirname(os.path.abspath(__file__))
    code = ("import sys; sys.path[:0] = [%r, %r]; import oracle, test_oracle as t; "
            "failed = t.pin_battery(oracle.load_library(%r)); print(len(failed)); "
            "sys.exit(0 if failed else 3)") % (here, os.path.dirname(here), str(so))
    res = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=600)
    assert res.returncode != 3, f"no pin caught the planted mistake {name}"
    assert res.returncode == 0 or res.returncode < 0 or "Error" in res.stderr, res.stderr[-2000:]


# ---------------------------------------------------------------- tolerance
def test_ulp_matches_numpy_spacing():
    rng = np.random.default_rng(2)
    # below 2^15, where numpy's next FP16 value is still finite
    x16 = np.concatenate([rng.uniform(-32000, 32000, 2000), rng.uniform(-1e-4, 1e-4, 2000),
                          [1.0, 2.0, 2.0 ** -14, 2.0 ** -24]]).astype(np.float16)
    assert np.array_equal(tolerance.ulp_out(x16.astype(np.float64), "f16"),
                          np.spacing(np.abs(x16)).astype(np.float64))
    # in the top binade [2^15, 65504] the spacing is 2^(15-10)
    assert tolerance.ulp_out(np.array([65504.0, 32768.0]), "f16").tolist() == [32.0, 32.0]
    x32 = np.concatenate([rng.standard_normal(2000) * 1e3, [1.0, 2.0 ** -126, 2.0 ** -140]]
                         ).astype(np.float32)
    assert np.array_equal(tolerance.ulp_out(x32.astype(np.float64), "f32"),
                          np.spacing(np.abs(x32)).astype(np.float64))


def test_ulp_bf16_against_neighbouring_pattern():
    rng = np.random.default_rng(4)
    bits = rng.integers(0x0001, 0x7F7F, 3000).astype(np.uint32)
    x = (bits << 16).view(np.float32).astype(np.float64)
    nxt = ((bits + 1) << 16).view(np.float32).astype(np.float64)
    assert np.array_equal(tolerance.ulp_out(x, "bf16"), nxt - x)
    assert tolerance.ulp_out(np.array([1.0]), "bf16")[0] == 2.0 ** -7


def test_check_flags_errors():
    ref = np.array([[1.0, -2.0], [100.0, 0.0]])
    cabs = np.array([[1.0, 2.0], [100.0, 0.0]])
    ok, *_ = tolerance.check(ref, ref, cabs, "f16")
    assert ok
    bad = ref.copy()
    bad[1, 0] += 0.3 + 2e-3 * 100      # beyond 2e-3*C_abs + ulp(100) = 0.2 + 0.0625
    ok, ratio, n_bad, first = tolerance.check(bad, ref, cabs, "f16")
    assert not ok and n_bad == 1 and first == (1, 0) and ratio > 1
    nan = ref.copy()
    nan[0, 0] = np.nan
    assert not tolerance.check(nan, ref, cabs, "f32")[0]
