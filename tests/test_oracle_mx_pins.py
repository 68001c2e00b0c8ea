"""Pins for the MXFP8 GEMM oracle, against things other than itself.

The operation (HipKittens "L2" detail page, §3 "Target operation" table, the
FP8 GEMM row: MXFP8 operands, FP32 accumulation; bf16 output here): E4M3
operands whose K dimension is cut into blocks of 32, each block of each row
scaled by a UE8M0 byte E (value 2^(E-127), 255 = NaN),

    C[i, j] = RNE_bf16( Σ_b 2^(SA[i,b]-127) · 2^(SB[j,b]-127) · Σ_{k∈b} A[i,k]·B[j,k] ).

Pins: exact rational arithmetic on small cases; unit scales reduce it to the
per-tensor FP8 oracle (itself pinned by exact arithmetic); a scale moves only
its own block; scaling a row's scales by 2^d scales its outputs by 2^d; the
decoding of the scale byte. ``test_mx_mutants_fail_pins`` plants mistakes
into a copy of the oracle's C source and checks that the pins catch them.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from fractions import Fraction

import numpy as np
import pytest

import synth
from exact_bf16 import bits_to_fraction, round_fraction

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _e4m3_fraction(code: int) -> Fraction:
    """Exact value of an E4M3 code, decoded here from the format's definition."""
    s = -1 if code & 0x80 else 1
    e = (code >> 3) & 0xF
    m = code & 7
    if e == 0:
        return s * Fraction(m, 8) * Fraction(1, 2 ** 6)
    return s * (1 + Fraction(m, 8)) * (Fraction(2) ** (e - 7))


def _exact_mx(A, B, SA, SB):
    M, K = A.shape
    N = B.shape[0]
    C = np.zeros((M, N), dtype=np.uint16)
    for i in range(M):
        for j in range(N):
            total = Fraction(0)
            for b in range(K // 32):
                d = sum(_e4m3_fraction(int(A[i, k])) * _e4m3_fraction(int(B[j, k])) for k in range(32 * b, 32 * b + 32))
                total += (Fraction(2) ** (int(SA[i, b]) - 127)) * (Fraction(2) ** (int(SB[j, b]) - 127)) * d
            C[i, j] = round_fraction(total)
    return C


class _MxLib:
    def __init__(self, path):
        lib = ctypes.CDLL(path)
        P, I = ctypes.c_void_p, ctypes.c_int64
        lib.oracle_gemm_mxfp8.argtypes = [P, P, P, P, P, I, I, I, I, I, I, I, I, ctypes.c_int]
        lib.oracle_ue8m0_to_double.argtypes = [ctypes.c_uint8]
        lib.oracle_ue8m0_to_double.restype = ctypes.c_double
        lib.oracle_gemm_fp8e4m3.argtypes = [P, P, P, I, I, I, I, I, I, ctypes.c_double, ctypes.c_int]
        self.lib = lib

    def ue8m0_value(self, e):
        return float(self.lib.oracle_ue8m0_to_double(int(e)))

    def gemm_mxfp8(self, A, B, SA, SB):
        A, B, SA, SB = (np.ascontiguousarray(x, dtype=np.uint8) for x in (A, B, SA, SB))
        M, K = A.shape
        N = B.shape[0]
        C = np.zeros((M, N), dtype=np.uint16)
        self.lib.oracle_gemm_mxfp8(A.ctypes.data, B.ctypes.data, SA.ctypes.data, SB.ctypes.data, C.ctypes.data,
                                   M, N, K, K, K, K // 32, K // 32, N, 1)
        return C

    def gemm_fp8(self, A, B):
        A, B = (np.ascontiguousarray(x, dtype=np.uint8) for x in (A, B))
        M, K = A.shape
        N = B.shape[0]
        C = np.zeros((M, N), dtype=np.uint16)
        self.lib.oracle_gemm_fp8e4m3(A.ctypes.data, B.ctypes.data, C.ctypes.data, M, N, K, K, K, N, 1.0, 1)
        return C


class _Packaged:
    def __init__(self, o):
        self.o = o

    def ue8m0_value(self, e):
        return self.o.ue8m0_value(e)

    def gemm_mxfp8(self, A, B, SA, SB):
        return self.o.gemm_mxfp8(A, B, SA, SB)

    def gemm_fp8(self, A, B):
        return self.o.gemm_fp8(A, B)


def _scales(rows, blocks, seed, lo=124, hi=130):
    g = np.random.Generator(np.random.PCG64(seed))
    return g.integers(lo, hi + 1, size=(rows, blocks)).astype(np.uint8)


# ---------------------------------------------------------------- the pins --

def pin_scale_decoding(o):
    """UE8M0: 127 -> 1, 0 -> 2^-127, 254 -> 2^127, 130 -> 8, 255 -> NaN."""
    for e, want in ((127, 1.0), (0, 2.0 ** -127), (254, 2.0 ** 127), (130, 8.0), (120, 2.0 ** -7)):
        if o.ue8m0_value(e) != want:
            return f"UE8M0 {e} decodes to {o.ue8m0_value(e)}"
    if not np.isnan(o.ue8m0_value(255)):
        return "UE8M0 255 is not NaN"
    return None


def pin_exact_small(o):
    """Exact rational arithmetic on small cases with mixed scales (normal E4M3
    draws and integer draws, K = 32, 64, 96)."""
    cases = [(3, 4, 64, 1), (2, 3, 96, 2), (4, 2, 32, 3)]
    for M, N, K, seed in cases:
        for A, B in ((synth.normal_e4m3(M, K, 10 * seed), synth.normal_e4m3(N, K, 10 * seed + 1)),
                     (synth.int_e4m3(M, K, 10 * seed + 2), synth.int_e4m3(N, K, 10 * seed + 3))):
            SA, SB = _scales(M, K // 32, seed), _scales(N, K // 32, seed + 100)
            got = o.gemm_mxfp8(A, B, SA, SB)
            want = _exact_mx(A, B, SA, SB)
            if not np.array_equal(got, want):
                return f"exact mismatch at M={M} N={N} K={K}: {np.argwhere(got != want)[:3].tolist()}"
    return None


def pin_unit_scales_are_fp8(o):
    """All scales 127 (= 1): the per-tensor FP8 GEMM with scale 1."""
    A = synth.normal_e4m3(9, 128, 51)
    B = synth.normal_e4m3(7, 128, 52)
    ones_a = np.full((9, 4), 127, np.uint8)
    ones_b = np.full((7, 4), 127, np.uint8)
    if not np.array_equal(o.gemm_mxfp8(A, B, ones_a, ones_b), o.gemm_fp8(A, B)):
        return "unit scales differ from the FP8 GEMM"
    return None


def pin_scale_moves_only_its_block(o):
    """With block 1 of A zero, its scale has no effect; a scale of a nonzero
    block does."""
    A = synth.normal_e4m3(5, 96, 61)
    A[:, 32:64] = 0
    B = synth.normal_e4m3(4, 96, 62)
    SA, SB = _scales(5, 3, 63), _scales(4, 3, 64)
    base = o.gemm_mxfp8(A, B, SA, SB)
    SA2 = SA.copy()
    SA2[:, 1] = 140
    if not np.array_equal(o.gemm_mxfp8(A, B, SA2, SB), base):
        return "the scale of an all-zero block changed the result"
    SA3 = SA.copy()
    SA3[:, 2] += 3
    if np.array_equal(o.gemm_mxfp8(A, B, SA3, SB), base):
        return "the scale of a nonzero block had no effect"
    return None


def pin_row_scaling(o):
    """Adding d to every scale of row i multiplies row i of the result by 2^d
    (no overflow or subnormals at these magnitudes) and leaves other rows."""
    A = synth.normal_e4m3(6, 64, 71)
    B = synth.normal_e4m3(5, 64, 72)
    SA, SB = _scales(6, 2, 73), _scales(5, 2, 74)
    base = synth.bf16_bits_to_f32(o.gemm_mxfp8(A, B, SA, SB)).astype(np.float64)
    SA2 = SA.copy()
    SA2[2] += 5
    got = synth.bf16_bits_to_f32(o.gemm_mxfp8(A, B, SA2, SB)).astype(np.float64)
    want = base.copy()
    want[2] *= 32.0
    if not np.array_equal(got, want):
        return "row scaling is not a power-of-two factor on that row only"
    return None


PINS = [pin_scale_decoding, pin_exact_small, pin_unit_scales_are_fp8, pin_scale_moves_only_its_block,
        pin_row_scaling]


@pytest.mark.parametrize("pin", PINS, ids=lambda p: p.__name__)
def test_mx_oracle_pin(oracle_lib, pin):
    assert pin(_Packaged(oracle_lib)) is None


def test_mx_entries_agree_with_full(oracle_lib):
    A = synth.normal_e4m3(20, 128, 81)
    B = synth.normal_e4m3(30, 128, 82)
    SA, SB = _scales(20, 4, 83), _scales(30, 4, 84)
    full = oracle_lib.gemm_mxfp8(A, B, SA, SB)
    r = np.array([0, 5, 19, 7])
    c = np.array([29, 0, 3, 14])
    assert np.array_equal(oracle_lib.gemm_mxfp8_entries(A, B, SA, SB, r, c), full[r, c])


def test_mx_rejects_bad_shapes(oracle_lib):
    A = np.zeros((2, 40), np.uint8)
    with pytest.raises(ValueError):
        oracle_lib.gemm_mxfp8(A, A, np.zeros((2, 1), np.uint8), np.zeros((2, 1), np.uint8))


MX_MUTANTS = {
    "last_block_dropped": ("for (int64_t blk = 0; blk < w->K / 32; ++blk) {",
                           "for (int64_t blk = 0; blk + 1 < w->K / 32; ++blk) {"),
    "scale_bias_128": ("return ldexp(1.0, (int)e - 127);", "return ldexp(1.0, (int)e - 128);"),
    "b_scale_dropped": ("s += oracle_ue8m0_to_double(sa[blk]) * oracle_ue8m0_to_double(sb[blk]) * d;",
                        "s += oracle_ue8m0_to_double(sa[blk]) * d;"),
    "scale_block_shift": ("const uint8_t* sa = w->SA + i * w->ldsa;", "const uint8_t* sa = w->SA + i * w->ldsa + 1;"),
    "nan_ignored": ("if (e == 255) return NAN;", "if (e == 254) return NAN;"),
    "block_range": ("for (int64_t k = 32 * blk; k < 32 * blk + 32; ++k)", "for (int64_t k = 32 * blk; k < 32 * blk + 31; ++k)"),
}


@pytest.mark.parametrize("name", sorted(MX_MUTANTS))
def test_mx_mutants_fail_pins(tmp_path, name):
    src = open(os.path.join(ROOT, "oracle", "gemm_ref.c")).read()
    old, new = MX_MUTANTS[name]
    assert src.count(old) == 1, f"mutation anchor for {name} not found exactly once"
    path_c = tmp_path / f"{name}.c"
    path_so = tmp_path / f"{name}.so"
    path_c.write_text(src.replace(old, new))
    subprocess.run(["gcc", "-std=c99", "-O2", "-ffp-contract=off", "-fPIC", "-shared", "-pthread",
                    "-D_GNU_SOURCE", str(path_c), "-o", str(path_so), "-lm"], check=True)
    mutant = _MxLib(str(path_so))
    with np.errstate(all="ignore"):
        failures = [p.__name__ for p in PINS if p(mutant) is not None]
    assert failures, f"mutant {name} passed every MXFP8 pin"
