"""Exact rational arithmetic on bf16 values, used to pin the oracle.

Independent of the oracle's C code: rounding here is "pick the nearest of the
two neighbouring representable values, ties to the one whose bit pattern is
even", found by bisection over the sorted list of every finite bf16 value,
which is the IEEE 754 definition of round-to-nearest-even taken literally.
"""
from __future__ import annotations

import bisect
import struct
from fractions import Fraction
from functools import lru_cache


def bits_to_fraction(h: int) -> Fraction:
    """Exact value of a finite bf16 bit pattern."""
    f = struct.unpack("<f", struct.pack("<I", (h & 0xFFFF) << 16))[0]
    return Fraction(f)


@lru_cache(maxsize=1)
def _positive_table():
    # every positive finite bf16 value, ascending with the bit pattern
    bits = list(range(0x0001, 0x7F80))
    vals = [bits_to_fraction(b) for b in bits]
    return bits, vals


_MAX = bits_to_fraction(0x7F7F)
_OVER = Fraction(2) ** 128  # where the next binade would start; IEEE treats it as the neighbour above MAX


def round_fraction(q: Fraction) -> int:
    """Exact value -> bf16 bit pattern, IEEE round-to-nearest-even."""
    if q == 0:
        return 0x0000
    sign = 0x8000 if q < 0 else 0
    a = -q if q < 0 else q
    bits, vals = _positive_table()
    if a >= _MAX:
        # neighbours: MAX (0x7F7F, odd) and 2^128 (the infinity encoding 0x7F80, even)
        lo_v, lo_b, hi_v, hi_b = _MAX, 0x7F7F, _OVER, 0x7F80
    elif a < vals[0]:
        lo_v, lo_b, hi_v, hi_b = Fraction(0), 0x0000, vals[0], bits[0]
    else:
        i = bisect.bisect_right(vals, a) - 1
        if vals[i] == a:
            return sign | bits[i]
        lo_v, lo_b, hi_v, hi_b = vals[i], bits[i], vals[i + 1], bits[i + 1]
    dlo, dhi = a - lo_v, hi_v - a
    if dlo < dhi:
        b = lo_b
    elif dhi < dlo:
        b = hi_b
    else:
        b = lo_b if lo_b % 2 == 0 else hi_b
    return sign | b


def exact_gemm(A_bits, B_bits):
    """Exact C = RNE(A·Bᵀ) with Fractions (tiny shapes only)."""
    M, K = len(A_bits), len(A_bits[0]) if len(A_bits) else 0
    N = len(B_bits)
    Af = [[bits_to_fraction(int(x)) for x in row] for row in A_bits]
    Bf = [[bits_to_fraction(int(x)) for x in row] for row in B_bits]
    C = [[0] * N for _ in range(M)]
    for i in range(M):
        for j in range(N):
            s = Fraction(0)
            for k in range(K):
                s += Af[i][k] * Bf[j][k]
            C[i][j] = round_fraction(s)
    return C


def fraction_to_bf16_exact(x: Fraction) -> int:
    """Bit pattern of a value that IS a bf16 (asserts exactness)."""
    b = round_fraction(x)
    assert bits_to_fraction(b) == x, x
    return b
