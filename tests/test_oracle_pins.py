"""Pins for the CPU oracle, against things other than the oracle itself.

The operation (HipKittens "L2" detail page, §3 "Target operation" table and
§7/§9.2 "ABt" hot loop): C = RNE_bf16(A·Bᵀ), bf16 in, bf16 out, with A M×K
and B N×K row-major. The pages print no element values for it, so the pins
are exact rational arithmetic (brute force), hand-built rounding ties, closed
forms, algebraic invariants and integer arithmetic. ``test_mutants_fail_pins``
plants plausible mistakes into a copy of the oracle's C source and checks that
the pins catch every one of them.
"""
from __future__ import annotations

import ctypes
import os
import re
import subprocess
from fractions import Fraction

import numpy as np
import pytest

import synth
from exact_bf16 import bits_to_fraction, exact_gemm, fraction_to_bf16_exact, round_fraction

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


class _Lib:
    """Minimal driver for a compiled copy of the oracle's C source."""

    def __init__(self, path):
        lib = ctypes.CDLL(path)
        P, I = ctypes.c_void_p, ctypes.c_int64
        lib.oracle_round_bf16.argtypes = [ctypes.c_double]
        lib.oracle_round_bf16.restype = ctypes.c_uint16
        lib.oracle_gemm_bf16.argtypes = [P, P, P, I, I, I, I, I, I, ctypes.c_int]
        lib.oracle_gemm_bf16.restype = ctypes.c_int
        self.lib = lib

    def round_bf16(self, x):
        return int(self.lib.oracle_round_bf16(float(x)))

    def gemm(self, A, B, threads=1):
        A = np.ascontiguousarray(A, dtype=np.uint16)
        B = np.ascontiguousarray(B, dtype=np.uint16)
        M, K = A.shape
        N = B.shape[0]
        C = np.zeros((M, N), dtype=np.uint16)
        if M and N:
            self.lib.oracle_gemm_bf16(A.ctypes.data, B.ctypes.data, C.ctypes.data, M, N, K, K, K, N,
                                      threads)
        return C


# ---------------------------------------------------------------- the pins --

def _bf(x: float) -> int:
    return fraction_to_bf16_exact(Fraction(x))


def pin_bruteforce(o):
    """Random bf16 normals on tiny shapes == exact rational GEMM, bit for bit."""
    for seed, (M, N, K) in enumerate([(1, 1, 1), (3, 5, 7), (8, 8, 16), (16, 9, 13), (5, 16, 16)]):
        A = synth.normal_bf16(M, K, 50 + seed)
        B = synth.normal_bf16(N, K, 80 + seed, 0.5)
        want = np.array(exact_gemm(A, B), dtype=np.uint16)
        got = o.gemm(A, B)
        if not np.array_equal(got, want):
            return f"bruteforce mismatch at {(M, N, K)}"
    return None


def pin_ties(o):
    """Hand-built exact midpoints pin ties-to-even, and a sum just above a
    midpoint pins single (not double) rounding."""
    cases = [
        # (a values, b values, expected C bits)
        ([1.0, 2 ** -4], [1.0, 2 ** -4], 0x3F80),           # 1 + 2^-8: tie between 0x3F80 and 0x3F81 -> even 0x3F80
        ([1.0, 3 * 2 ** -4], [1.0, 2 ** -4], 0x3F82),       # 1 + 3·2^-8: tie between 0x3F81 and 0x3F82 -> 0x3F82
        ([1.0, 2 ** -4, 2 ** -15], [1.0, 2 ** -4, 2 ** -15], 0x3F81),  # 1 + 2^-8 + 2^-30: above the tie -> up
        ([-1.0, 2 ** -4], [1.0, -(2 ** -4)], 0xBF80),       # negative tie -> even magnitude
        ([2.0, 2 ** -3], [1.0, 2 ** -4], 0x4000),           # 2 + 2^-7: tie at the next binade -> 0x4000
    ]
    for a, b, want in cases:
        A = np.array([[_bf(x) for x in a]], dtype=np.uint16)
        B = np.array([[_bf(x) for x in b]], dtype=np.uint16)
        got = int(o.gemm(A, B)[0, 0])
        if got != want:
            return f"tie case {a}·{b}: got {got:#06x}, want {want:#06x}"
    return None


def pin_identity_permutation(o):
    K = 24
    A = synth.normal_bf16(11, K, 7)
    one = _bf(1.0)
    eye = np.zeros((K, K), dtype=np.uint16)
    eye[np.arange(K), np.arange(K)] = one
    if not np.array_equal(o.gemm(A, eye), A):
        return "B = I does not reproduce A"
    perm = np.random.Generator(np.random.PCG64(3)).permutation(K)
    P = np.zeros((K, K), dtype=np.uint16)
    P[np.arange(K), perm] = one          # row j of B selects column perm[j] of A
    if not np.array_equal(o.gemm(A, P), A[:, perm]):
        return "B = permutation does not permute the columns of A"
    return None


def pin_closed_form(o):
    """A ≡ a, B ≡ b  =>  C ≡ RNE(K·a·b), exactly."""
    for a, b, K in [(0.75, -1.25, 1), (0.1015625, 3.0, 7), (1.5, 1.5, 300), (-0.3359375, 0.046875, 1024)]:
        ab, bb = _bf(a), _bf(b)
        A = np.full((3, K), ab, dtype=np.uint16)
        B = np.full((2, K), bb, dtype=np.uint16)
        want = round_fraction(K * bits_to_fraction(ab) * bits_to_fraction(bb))
        C = o.gemm(A, B)
        if not np.all(C == want):
            return f"closed form a={a} b={b} K={K}: got {C[0,0]:#06x}, want {want:#06x}"
    return None


def pin_invariants(o):
    A = synth.normal_bf16(9, 40, 11)
    B = synth.normal_bf16(6, 40, 12)
    C = o.gemm(A, B)
    if not np.array_equal(o.gemm(B, A), C.T):
        return "swapping A and B does not transpose C"
    negC = o.gemm(A ^ np.uint16(0x8000), B)
    nz = (C & 0x7FFF) != 0
    if not np.array_equal(negC[nz], C[nz] ^ np.uint16(0x8000)):
        return "negating A does not negate C"
    if np.any(o.gemm(np.zeros_like(A), B) != 0):
        return "zero A does not give +0"
    # not symmetric in the operand roles: a non-square case distinguishes A·Bᵀ from A·B
    return None


def pin_integer(o):
    """Integer-valued inputs: C = RNE(int64 A·Bᵀ)."""
    for M, N, K in [(7, 5, 33), (16, 16, 256)]:
        A = synth.int_bf16(M, K, 101)
        B = synth.int_bf16(N, K, 102)
        Ai = synth.bf16_bits_to_f32(A).astype(np.int64)
        Bi = synth.bf16_bits_to_f32(B).astype(np.int64)
        Ci = Ai @ Bi.T
        want = np.array([[round_fraction(Fraction(int(v))) for v in row] for row in Ci], dtype=np.uint16)
        if not np.array_equal(o.gemm(A, B), want):
            return f"integer case {(M, N, K)}"
    return None


def pin_rounding(o):
    """binary64 -> bf16 on normals, subnormals, ties, overflow and zeros."""
    rng = np.random.Generator(np.random.PCG64(5))
    xs = list(rng.standard_normal(400) * np.exp2(rng.integers(-140, 128, 400)))
    xs += [0.0, -0.0, 1.0, -1.0, 1 + 2 ** -8, 1 + 3 * 2 ** -8, 2 ** -133, 2 ** -134, 3 * 2 ** -134,
           2 ** -126, 2 ** -126 - 2 ** -134, float(2 ** 128 - 2 ** 119), float(2 ** 128 - 2 ** 120),
           1.0000001, 65504.0, 3.0e38, -3.4e38]
    for x in xs:
        want = round_fraction(Fraction(float(x)))
        if np.isfinite(x) and abs(x) >= 2 ** 128:
            want = (0x8000 if x < 0 else 0) | 0x7F80
        got = o.round_bf16(x)
        if x == 0:
            want = 0x8000 if np.signbit(x) else 0
        if got != want:
            return f"round_bf16({x!r}) = {got:#06x}, want {want:#06x}"
    return None


def pin_non_finite(o):
    """IEEE 754 on non-finite values: ±Inf round to themselves and NaN to a
    NaN; in a dot product Inf·k is ±Inf, Inf·0 and Inf + (−Inf) are NaN,
    and a NaN operand makes its whole row NaN. Expected entries worked out
    by hand from those rules."""
    def is_nan(b):
        return (b & 0x7F80) == 0x7F80 and (b & 0x7F) != 0
    if o.round_bf16(float("inf")) != 0x7F80 or o.round_bf16(float("-inf")) != 0xFF80:
        return "round_bf16(±inf)"
    if not is_nan(o.round_bf16(float("nan"))):
        return "round_bf16(nan) is not a NaN"
    INF, NINF, NAN, ONE, TWO, ZERO, M1 = 0x7F80, 0xFF80, 0x7FC0, 0x3F80, 0x4000, 0x0000, 0xBF80
    A = np.array([[INF, ONE], [INF, NINF], [NAN, ZERO], [ONE, TWO]], dtype=np.uint16)
    B = np.array([[TWO, ONE], [ZERO, ONE], [M1, ZERO], [ONE, ONE]], dtype=np.uint16)
    N_ = None   # a NaN entry
    want = [[INF, N_, NINF, INF],           # Inf·2+1, Inf·0+1, Inf·(−1)+0, Inf+1
            [N_, N_, N_, N_],               # Inf−Inf, NaN+(−Inf), −Inf+NaN, Inf−Inf
            [N_, N_, N_, N_],               # NaN·anything
            [0x4080, 0x4000, M1, 0x4040]]   # 4, 2, −1, 3
    C = o.gemm(A, B)
    for i in range(4):
        for j in range(4):
            w, g = want[i][j], int(C[i, j])
            if (w is None and not is_nan(g)) or (w is not None and g != w):
                return f"non-finite case C[{i},{j}] = {g:#06x}"
    return None


PINS = [pin_bruteforce, pin_ties, pin_identity_permutation, pin_closed_form, pin_invariants,
        pin_integer, pin_rounding, pin_non_finite]


@pytest.mark.parametrize("pin", PINS, ids=lambda p: p.__name__)
def test_oracle_pin(oracle_lib, pin):
    assert pin(oracle_lib) is None


def test_transposed_operand_is_distinguished(oracle_lib):
    """C = A·Bᵀ, not A·B: a non-symmetric square case separates the two."""
    K = 8
    A = synth.int_bf16(K, K, 21)
    B = synth.int_bf16(K, K, 22)
    Ai = synth.bf16_bits_to_f32(A).astype(np.int64)
    Bi = synth.bf16_bits_to_f32(B).astype(np.int64)
    C = synth.bf16_bits_to_f32(oracle_lib.gemm(A, B)).astype(np.int64)
    assert np.array_equal(C, Ai @ Bi.T)
    assert not np.array_equal(C, Ai @ Bi)


def test_rows_and_entries_agree_with_full(oracle_lib):
    A = synth.normal_bf16(37, 70, 31)
    B = synth.normal_bf16(29, 70, 32)
    C = oracle_lib.gemm(A, B, threads=3)
    rows = np.array([0, 5, 36])
    R, used = oracle_lib.gemm_rows(A, B, rows, threads=2)
    assert used >= 1 and np.array_equal(R, C[rows])
    r, c = synth.sample_positions(37, 29, 9, count=50, tile_m=16, tile_n=16)
    E, _ = oracle_lib.gemm_entries(A, B, r, c)
    assert np.array_equal(E, C[r, c])
    # strided operands (leading dimension > K)
    Aw = np.zeros((37, 80), dtype=np.uint16)
    Aw[:, :70] = A
    assert np.array_equal(oracle_lib.gemm(Aw[:, :70], B), C)


def test_empty_k_gives_zero(oracle_lib):
    A = np.zeros((4, 0), dtype=np.uint16)
    B = np.zeros((3, 0), dtype=np.uint16)
    assert np.all(oracle_lib.gemm(A, B) == 0)


# ------------------------------------------------------------- mutations --

MUTANTS = {
    "dropped_last_term": ("for (int64_t k = 0; k < K; ++k) s +=", "for (int64_t k = 0; k + 1 < K; ++k) s +="),
    "transposed_B": ("const uint16_t* b = B + j * ldb;", "const uint16_t* b = B + j;"),
    "swapped_index": ("for (int64_t j = 0; j < w->N; ++j) o[j] = entry(w, i, j);",
                      "for (int64_t j = 0; j < w->N; ++j) o[j] = entry(w, (i + 1) % w->end, j);"),
    "ties_away": ("if (fmod(fl, 2.0) != 0.0) n = fl + 1.0;", "n = fl + 1.0;"),
    "truncation": ("if (frac > 0.5) {", "if (frac > 2.0) {"),
    "sign_error": ("s += bf16_bits_to_double(a[k]) * bf16_bits_to_double(b[k]);",
                   "s += fabs(bf16_bits_to_double(a[k])) * bf16_bits_to_double(b[k]);"),
    "via_binary32": ("double a = fabs(x);", "double a = (double)(float)fabs(x);"),
    "subnormal_quantum": ("int qexp = (E < -126 ? -126 : E) - 7;", "int qexp = E - 7;"),
    "nan_as_inf": ("if (isnan(x)) return (uint16_t)(sign | 0x7FC0u);", "if (isnan(x)) return (uint16_t)(sign | 0x7F80u);"),
    "nan_terms_skipped": ("s += bf16_bits_to_double(a[k]) * bf16_bits_to_double(b[k]);",
                          "{ double t = bf16_bits_to_double(a[k]) * bf16_bits_to_double(b[k]); if (t == t) s += t; }"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutants_fail_pins(tmp_path, name):
    src = open(os.path.join(ROOT, "oracle", "gemm_ref.c")).read()
    old, new = MUTANTS[name]
    assert src.count(old) == 1, f"mutation anchor for {name} not found exactly once"
    path_c = tmp_path / f"{name}.c"
    path_so = tmp_path / f"{name}.so"
    path_c.write_text(src.replace(old, new))
    subprocess.run(["gcc", "-std=c99", "-O2", "-ffp-contract=off", "-fPIC", "-shared", "-pthread",
                    "-D_GNU_SOURCE", str(path_c), "-o", str(path_so), "-lm"], check=True)
    mutant = _Lib(str(path_so))
    failures = [p.__name__ for p in PINS if p(mutant) is not None]
    assert failures, f"mutant {name} passed every pin"


# ------------------------------------------------------ fused epilogue --

def pin_activation_values(o):
    """Activation values fixed by mathematics, not by re-typing the formulas:
    Φ(1) from the normal table, σ(ln 3) = 3/4, the odd-part identities
    GELU(x) − GELU(−x) = x (Φ(x) + Φ(−x) = 1) and SiLU(x) − SiLU(−x) = x
    (σ(x) + σ(−x) = 1), ReLU's definition and GELU's limits."""
    act = o.activation if hasattr(o, "activation") else None
    if act is None:
        return "no activation entry"
    if abs(act(1.0, 2) - 0.8413447460685429) > 1e-15:
        return "GELU(1) != Φ(1)"
    if abs(act(np.log(3.0), 3) - 0.75 * np.log(3.0)) > 1e-15:
        return "SiLU(ln 3) != 3/4 ln 3"
    for x in (0.3, 1.7, 4.25, 9.0):
        if abs((act(x, 2) - act(-x, 2)) - x) > 1e-12 or abs((act(x, 3) - act(-x, 3)) - x) > 1e-12:
            return f"odd-part identity fails at {x}"
        if act(x, 1) != x or act(-x, 1) != 0.0:
            return f"ReLU({x})"
    if abs(act(8.0, 2) - 8.0) > 1e-12 or abs(act(-8.0, 2)) > 1e-12:
        return "GELU limits"
    if act(0.0, 2) != 0.0 or act(0.0, 3) != 0.0 or act(2.5, 0) != 2.5:
        return "activation at 0 / identity"
    return None


def pin_epilogue_gemm(o):
    """Bias and activation on top of the GEMM: exact rational bias sums on
    tiny shapes; A = 0 gives RNE(act(bias)); ReLU on integer inputs against
    int64 arithmetic."""
    if not hasattr(o, "gemm_epilogue"):
        return "no epilogue entry"
    M, N, K = 5, 7, 9
    A = synth.normal_bf16(M, K, 91)
    B = synth.normal_bf16(N, K, 92)
    bias = synth.normal_bf16(1, N, 93, 2.0)[0]
    want = np.zeros((M, N), dtype=np.uint16)
    Af = [[bits_to_fraction(int(x)) for x in r] for r in A]
    Bf = [[bits_to_fraction(int(x)) for x in r] for r in B]
    for i in range(M):
        for j in range(N):
            s = sum(Af[i][k] * Bf[j][k] for k in range(K)) + bits_to_fraction(int(bias[j]))
            want[i, j] = round_fraction(s)
    if not np.array_equal(o.gemm_epilogue(A, B, bias, 0), want):
        return "bias sum is not exact"
    Z = np.zeros_like(A)
    for act in (1, 2, 3):
        got = o.gemm_epilogue(Z, B, bias, act)
        ref = np.array([round_fraction(Fraction(o.activation(float(bits_to_fraction(int(b))), act))) for b in bias],
                       dtype=np.uint16)
        if not np.array_equal(got[0], ref) or not np.all(got == got[0]):
            return f"A = 0 with act {act}"
    Ai, Bi = synth.int_bf16(6, 40, 94), synth.int_bf16(8, 40, 95)
    bi = synth.int_bf16(1, 8, 96)[0]
    ref = synth.bf16_bits_to_f32(Ai).astype(np.int64) @ synth.bf16_bits_to_f32(Bi).astype(np.int64).T
    ref = np.maximum(ref + synth.bf16_bits_to_f32(bi).astype(np.int64), 0)
    want = np.array([[round_fraction(Fraction(int(v))) for v in r] for r in ref], dtype=np.uint16)
    if not np.array_equal(o.gemm_epilogue(Ai, Bi, bi, 1), want):
        return "ReLU on integers"
    return None


@pytest.mark.parametrize("pin", [pin_activation_values, pin_epilogue_gemm], ids=lambda p: p.__name__)
def test_epilogue_pin(oracle_lib, pin):
    assert pin(oracle_lib) is None


EPILOGUE_MUTANTS = {
    "bias_by_row": ("if (w->bias) x += bf16_bits_to_double(w->bias[j]);",
                    "if (w->bias) x += bf16_bits_to_double(w->bias[i % 5]);"),
    "gelu_no_sqrt2": ("case 2: return 0.5 * x * (1.0 + erf(x / sqrt(2.0)));",
                      "case 2: return 0.5 * x * (1.0 + erf(x));"),
    "silu_sign": ("case 3: return x / (1.0 + exp(-x));", "case 3: return x / (1.0 + exp(x));"),
    "relu_leaky": ("case 1: return x > 0.0 ? x : 0.0;", "case 1: return x > 0.0 ? x : 0.01 * x;"),
    "act_before_bias": ("        if (w->bias) x += bf16_bits_to_double(w->bias[j]);\n        x = oracle_activation(x, w->act);",
                        "        x = oracle_activation(x, w->act);\n        if (w->bias) x += bf16_bits_to_double(w->bias[j]);"),
}


class _EpiLib(_Lib):
    def __init__(self, path):
        super().__init__(path)
        P, I = ctypes.c_void_p, ctypes.c_int64
        self.lib.oracle_activation.argtypes = [ctypes.c_double, ctypes.c_int]
        self.lib.oracle_activation.restype = ctypes.c_double
        self.lib.oracle_gemm_bf16_epilogue.argtypes = [P, P, P, P, I, I, I, I, I, I, ctypes.c_int, ctypes.c_int]

    def activation(self, x, act):
        return float(self.lib.oracle_activation(float(x), int(act)))

    def gemm_epilogue(self, A, B, bias, act):
        A = np.ascontiguousarray(A, dtype=np.uint16)
        B = np.ascontiguousarray(B, dtype=np.uint16)
        bias = np.ascontiguousarray(bias, dtype=np.uint16)
        M, K = A.shape
        N = B.shape[0]
        C = np.zeros((M, N), dtype=np.uint16)
        self.lib.oracle_gemm_bf16_epilogue(A.ctypes.data, B.ctypes.data, bias.ctypes.data, C.ctypes.data, M, N,
                                           K, K, K, N, act, 1)
        return C


@pytest.mark.parametrize("name", sorted(EPILOGUE_MUTANTS))
def test_epilogue_mutants_fail_pins(tmp_path, name):
    src = open(os.path.join(ROOT, "oracle", "gemm_ref.c")).read()
    old, new = EPILOGUE_MUTANTS[name]
    assert src.count(old) == 1, f"mutation anchor for {name} not found exactly once"
    path_c = tmp_path / f"{name}.c"
    path_so = tmp_path / f"{name}.so"
    path_c.write_text(src.replace(old, new))
    subprocess.run(["gcc", "-std=c99", "-O2", "-ffp-contract=off", "-fPIC", "-shared", "-pthread",
                    "-D_GNU_SOURCE", str(path_c), "-o", str(path_so), "-lm"], check=True)
    mutant = _EpiLib(str(path_so))
    assert pin_activation_values(mutant) is not None or pin_epilogue_gemm(mutant) is not None, \
        f"mutant {name} passed the epilogue pins"


# ------------------------------------------------- fused residual add --

def pin_residual(o):
    """The residual R is added after the activation, per (row, column), before
    the one rounding. Exact rational sums on a tiny non-square shape with a
    padded leading dimension for R (a transposed or mis-strided R reads other
    values); ReLU on sums that are negative where R is positive (so adding R
    before the activation gives another value); A = 0 gives RNE(act(bias) + R)
    for every activation; integer data against int64 arithmetic."""
    if not hasattr(o, "gemm_fused"):
        return "no residual entry"
    M, N, K = 5, 7, 9
    A = synth.normal_bf16(M, K, 191)
    B = synth.normal_bf16(N, K, 192)
    bias = synth.normal_bf16(1, N, 193, 2.0)[0]
    Rstore = synth.normal_bf16(M, N + 9, 194, 3.0)      # leading dimension 16 > N
    R = Rstore[:, :N]
    Af = [[bits_to_fraction(int(x)) for x in r] for r in A]
    Bf = [[bits_to_fraction(int(x)) for x in r] for r in B]
    dots = [[sum(Af[i][k] * Bf[j][k] for k in range(K)) for j in range(N)] for i in range(M)]
    for act in (0, 1):
        want = np.zeros((M, N), dtype=np.uint16)
        for i in range(M):
            for j in range(N):
                x = dots[i][j] + bits_to_fraction(int(bias[j]))
                if act == 1:
                    x = max(x, Fraction(0))
                want[i, j] = round_fraction(x + bits_to_fraction(int(R[i, j])))
        if not np.array_equal(o.gemm_fused(A, B, bias, R, act), want):
            return f"act {act}: act(dot + bias) + R is not exact"
    # no bias, no activation: only the residual
    want = np.array([[round_fraction(dots[i][j] + bits_to_fraction(int(R[i, j]))) for j in range(N)]
                     for i in range(M)], dtype=np.uint16)
    if not np.array_equal(o.gemm_fused(A, B, None, R, 0), want):
        return "dot + R is not exact"
    Z = np.zeros_like(A)
    for act in (1, 2, 3):
        got = o.gemm_fused(Z, B, bias, R, act)
        ref = np.array([[round_fraction(Fraction(o.activation(float(bits_to_fraction(int(bias[j]))), act))
                                        + bits_to_fraction(int(R[i, j]))) for j in range(N)] for i in range(M)],
                       dtype=np.uint16)
        if not np.array_equal(got, ref):
            return f"A = 0 with act {act}"
    Ai, Bi = synth.int_bf16(6, 40, 195), synth.int_bf16(8, 40, 196)
    bi, Ri = synth.int_bf16(1, 8, 197)[0], synth.int_bf16(6, 8, 198, -40, 40)
    ref = synth.bf16_bits_to_f32(Ai).astype(np.int64) @ synth.bf16_bits_to_f32(Bi).astype(np.int64).T
    ref = np.maximum(ref + synth.bf16_bits_to_f32(bi).astype(np.int64), 0) + synth.bf16_bits_to_f32(Ri).astype(np.int64)
    want = np.array([[round_fraction(Fraction(int(v))) for v in r] for r in ref], dtype=np.uint16)
    if not np.array_equal(o.gemm_fused(Ai, Bi, bi, Ri, 1), want):
        return "ReLU + residual on integers"
    return None


def test_residual_pin(oracle_lib):
    assert pin_residual(_FusedView(oracle_lib)) is None


def test_residual_entries_agree_with_full():
    import oracle
    M, N, K = 37, 29, 50
    A, B = synth.normal_bf16(M, K, 181), synth.normal_bf16(N, K, 182)
    bias, R = synth.normal_bf16(1, N, 183)[0], synth.normal_bf16(M, N, 184)
    full = oracle.gemm_epilogue(A, B, bias, 2, residual=R)
    rows, cols = np.meshgrid(np.arange(M), np.arange(N), indexing="ij")
    got = oracle.gemm_epilogue_entries(A, B, rows.ravel(), cols.ravel(), bias, 2, residual=R)
    assert np.array_equal(got.reshape(M, N), full)
    # without a residual the fused function is the epilogue GEMM
    assert np.array_equal(oracle.gemm_epilogue(A, B, bias, 2), oracle.gemm_epilogue(A, B, bias, 2, residual=None))


class _FusedView:
    """The package oracle seen through the interface the residual pin uses."""

    def __init__(self, lib):
        import oracle
        self._o = oracle

    def activation(self, x, act):
        return self._o.activation(x, act)

    def gemm_fused(self, A, B, bias, R, act):
        return self._o.gemm_epilogue(A, B, bias, act, residual=R)


RESIDUAL_MUTANTS = {
    "residual_transposed": ("x += bf16_bits_to_double(w->res[i * w->ldr + j]);",
                            "x += bf16_bits_to_double(w->res[j * w->ldr + i]);"),
    "residual_ld_ignored": ("x += bf16_bits_to_double(w->res[i * w->ldr + j]);",
                            "x += bf16_bits_to_double(w->res[i * w->N + j]);"),
    "residual_subtracted": ("x += bf16_bits_to_double(w->res[i * w->ldr + j]);",
                            "x -= bf16_bits_to_double(w->res[i * w->ldr + j]);"),
    "residual_before_activation": (
        "        x = oracle_activation(x, w->act);\n    }\n    if (w->res) x += bf16_bits_to_double(w->res[i * w->ldr + j]);",
        "        if (w->res) x += bf16_bits_to_double(w->res[i * w->ldr + j]);\n        x = oracle_activation(x, w->act);\n    }"),
    "residual_dropped_when_no_epilogue": ("    if (w->res) x += bf16_bits_to_double(w->res[i * w->ldr + j]);",
                                          "    if (w->res && (w->bias || w->act)) x += bf16_bits_to_double(w->res[i * w->ldr + j]);"),
    "residual_rounded_separately": (
        "    if (w->res) x += bf16_bits_to_double(w->res[i * w->ldr + j]);",
        "    if (w->res) x = bf16_bits_to_double(oracle_round_bf16(x)) + bf16_bits_to_double(w->res[i * w->ldr + j]);"),
}


class _ResLib(_EpiLib):
    def __init__(self, path):
        super().__init__(path)
        P, I = ctypes.c_void_p, ctypes.c_int64
        self.lib.oracle_gemm_bf16_fused.argtypes = [P, P, P, P, I, P, I, I, I, I, I, I, ctypes.c_int, ctypes.c_int]

    def gemm_fused(self, A, B, bias, R, act):
        A = np.ascontiguousarray(A, dtype=np.uint16)
        B = np.ascontiguousarray(B, dtype=np.uint16)
        M, K = A.shape
        N = B.shape[0]
        ldr = R.strides[0] // 2
        C = np.zeros((M, N), dtype=np.uint16)
        bptr = None if bias is None else np.ascontiguousarray(bias, dtype=np.uint16)
        self.lib.oracle_gemm_bf16_fused(A.ctypes.data, B.ctypes.data, None if bptr is None else bptr.ctypes.data,
                                        R.ctypes.data, ldr, C.ctypes.data, M, N, K, K, K, N, act, 1)
        return C


@pytest.mark.parametrize("name", sorted(RESIDUAL_MUTANTS))
def test_residual_mutants_fail_pins(tmp_path, name):
    src = open(os.path.join(ROOT, "oracle", "gemm_ref.c")).read()
    old, new = RESIDUAL_MUTANTS[name]
    assert src.count(old) == 1, f"mutation anchor for {name} not found exactly once"
    path_c = tmp_path / f"{name}.c"
    path_so = tmp_path / f"{name}.so"
    path_c.write_text(src.replace(old, new))
    subprocess.run(["gcc", "-std=c99", "-O2", "-ffp-contract=off", "-fPIC", "-shared", "-pthread",
                    "-D_GNU_SOURCE", str(path_c), "-o", str(path_so), "-lm"], check=True)
    mutant = _ResLib(str(path_so))
    assert pin_residual(mutant) is not None, f"mutant {name} passed the residual pin"


# ------------------------------------------------------------ FP8 (E4M3) --

def pin_e4m3_decode(o):
    """All 256 E4M3 codes against PyTorch's float8_e4m3fn (a library routine),
    plus the format's documented landmarks: 448 = largest (0x7E), 2^-6 =
    smallest normal (0x08), 2^-9 = smallest subnormal (0x01), 1.0 = 0x38,
    NaN = 0x7F / 0xFF."""
    import torch
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = np.array([o.e4m3_value(int(c)) for c in codes])
    same = (got == ref) | (np.isnan(got) & np.isnan(ref))
    if not same.all():
        return f"decode differs at codes {np.nonzero(~same)[0][:5].tolist()}"
    marks = {0x7E: 448.0, 0x08: 2.0 ** -6, 0x01: 2.0 ** -9, 0x38: 1.0, 0xB8: -1.0}
    for c, v in marks.items():
        if o.e4m3_value(c) != v:
            return f"landmark {c:#x}"
    if not (np.isnan(o.e4m3_value(0x7F)) and np.isnan(o.e4m3_value(0xFF))):
        return "NaN codes"
    return None


def _exact_fp8_gemm(o, A, B, sa, sb):
    val = {c: Fraction(o.e4m3_value(c)) for c in range(256) if not np.isnan(o.e4m3_value(c))}
    scale = Fraction(float(np.float32(sa))) * Fraction(float(np.float32(sb)))
    M, K = A.shape
    N = B.shape[0]
    C = np.zeros((M, N), dtype=np.uint16)
    for i in range(M):
        for j in range(N):
            C[i, j] = round_fraction(scale * sum(val[int(A[i, k])] * val[int(B[j, k])] for k in range(K)))
    return C


def pin_fp8_gemm(o):
    """Exact rational FP8 GEMMs on tiny shapes (power-of-two and general
    float32 scales), integer inputs against int64, and the closed form
    A ≡ a, B ≡ b ⇒ C ≡ RNE(K·a·b·sa·sb)."""
    if not hasattr(o, "gemm_fp8"):
        return "no FP8 entry"
    for seed, (M, N, K, sa, sb) in enumerate([(3, 4, 5, 1.0, 1.0), (6, 5, 17, 0.5, 0.25), (4, 7, 33, 0.3, 1.7)]):
        A = synth.normal_e4m3(M, K, 600 + seed, 2.0)
        B = synth.normal_e4m3(N, K, 700 + seed, 3.0)
        if not np.array_equal(o.gemm_fp8(A, B, sa, sb), _exact_fp8_gemm(o, A, B, sa, sb)):
            return f"exact FP8 GEMM {(M, N, K, sa, sb)}"
    Ai, Bi = synth.int_e4m3(9, 64, 801), synth.int_e4m3(7, 64, 802)
    dec = np.vectorize(o.e4m3_value)
    ref = dec(Ai).astype(np.int64) @ dec(Bi).astype(np.int64).T
    want = np.array([[round_fraction(Fraction(int(v))) for v in r] for r in ref], dtype=np.uint16)
    if not np.array_equal(o.gemm_fp8(Ai, Bi), want):
        return "integer FP8 GEMM"
    a, b = 0x3A, 0xC4          # 1.25 and -3.0
    A = np.full((2, 100), a, dtype=np.uint8)
    B = np.full((3, 100), b, dtype=np.uint8)
    want = round_fraction(Fraction(100) * Fraction(1.25) * Fraction(-3) * Fraction(0.5) * Fraction(0.25))
    if not np.all(o.gemm_fp8(A, B, 0.5, 0.25) == want):
        return "closed form"
    return None


@pytest.mark.parametrize("pin", [pin_e4m3_decode, pin_fp8_gemm], ids=lambda p: p.__name__)
def test_fp8_pin(oracle_lib, pin):
    assert pin(oracle_lib) is None


def test_e4m3_generator_matches_library_rounding():
    import torch
    g = np.random.Generator(np.random.PCG64(9))
    x = (g.standard_normal(50000) * np.exp2(g.integers(-12, 8, 50000))).astype(np.float32)
    x = x[np.abs(x) <= 448]
    want = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = synth.f32_to_e4m3_codes(x)
    zero = (want & 0x7F) == 0
    assert np.array_equal(got[~zero], want[~zero]) and np.all((got[zero] & 0x7F) == 0)


FP8_MUTANTS = {
    "bias8": ("else v = ldexp(1.0 + (double)m / 8.0, e - 7);", "else v = ldexp(1.0 + (double)m / 8.0, e - 8);"),
    "subnormal_exp": ("if (e == 0) v = ldexp((double)m / 8.0, -6);", "if (e == 0) v = ldexp((double)m / 8.0, -7);"),
    "no_nan": ("if (e == 0xF && m == 7) return NAN;", "if (e == 0xF && m == 8) return NAN;"),
    "scale_dropped": ("return oracle_round_bf16(w->scale * s);", "return oracle_round_bf16(s);"),
    "mantissa_bits": ("int s = (b >> 7) & 1, e = (b >> 3) & 0xF, m = b & 7;",
                      "int s = (b >> 7) & 1, e = (b >> 2) & 0x1F, m = b & 3;"),
}


class _Fp8Lib(_Lib):
    def __init__(self, path):
        super().__init__(path)
        P, I = ctypes.c_void_p, ctypes.c_int64
        self.lib.oracle_e4m3_to_double.argtypes = [ctypes.c_uint8]
        self.lib.oracle_e4m3_to_double.restype = ctypes.c_double
        self.lib.oracle_gemm_fp8e4m3.argtypes = [P, P, P, I, I, I, I, I, I, ctypes.c_double, ctypes.c_int]

    def e4m3_value(self, c):
        return float(self.lib.oracle_e4m3_to_double(int(c) & 0xFF))

    def gemm_fp8(self, A, B, sa=1.0, sb=1.0):
        A = np.ascontiguousarray(A, dtype=np.uint8)
        B = np.ascontiguousarray(B, dtype=np.uint8)
        M, K = A.shape
        N = B.shape[0]
        C = np.zeros((M, N), dtype=np.uint16)
        self.lib.oracle_gemm_fp8e4m3(A.ctypes.data, B.ctypes.data, C.ctypes.data, M, N, K, K, K, N,
                                     float(np.float32(sa)) * float(np.float32(sb)), 1)
        return C


@pytest.mark.parametrize("name", sorted(FP8_MUTANTS))
def test_fp8_mutants_fail_pins(tmp_path, name):
    src = open(os.path.join(ROOT, "oracle", "gemm_ref.c")).read()
    old, new = FP8_MUTANTS[name]
    assert src.count(old) == 1, f"mutation anchor for {name} not found exactly once"
    path_c = tmp_path / f"{name}.c"
    path_so = tmp_path / f"{name}.so"
    path_c.write_text(src.replace(old, new))
    subprocess.run(["gcc", "-std=c99", "-O2", "-ffp-contract=off", "-fPIC", "-shared", "-pthread",
                    "-D_GNU_SOURCE", str(path_c), "-o", str(path_so), "-lm"], check=True)
    mutant = _Fp8Lib(str(path_so))
    assert pin_e4m3_decode(mutant) is not None or pin_fp8_gemm(mutant) is not None, \
        f"mutant {name} passed the FP8 pins"
