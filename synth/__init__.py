"""Seeded synthetic inputs for the BF16 GEMM, shared by the tests and the bench.

This module holds none of the GEMM's arithmetic: it only draws random numbers,
rounds them to bf16 bit patterns and lists the workload shapes. Both the CUDA
path and the CPU oracle receive the bytes it produces.

Recipe (the workloads the HipKittens pages measure are square BF16 GEMMs with
M = N = K from 1024 to 14592, "L2" detail page §3 "Evaluated regimes", and the
headline 8192³ of §2 Q3 / §5 Tab. 2; the other shapes are LLM-projection
shapes of the same operation):

* normal entries: ``numpy.random.Generator(PCG64(seed)).standard_normal`` in
  float32, multiplied by the workload's scale in float32, rounded to bf16 with
  round-to-nearest-even on the float32 bit pattern;
* integer entries: ``integers(-4, 5)`` (uniform on {-4..4}), exact in bf16;
* seeds: A = 1000 + workload id, B = 2000 + workload id (integer variant 1100+,
  2100+), sample positions 3000 + workload id;
* FP8 workloads: the same normal draws rounded to E4M3 codes (nearest value,
  ties to the even code, saturating at ±448);
* attention workloads (the pages' GQA forward of §5 Fig. 7: batch 16, 64
  query heads, 8 KV heads, head dim 64 or 128, prefill lengths 1k-8k):
  Q, K, V entries N(0,1) rounded to bf16, laid out [B, H, S, D], seeds
  Q = 4000 + id, K = 5000 + id, V = 6000 + id.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

_CHUNK = 1 << 24  # elements per generation chunk (keeps host temporaries small)


@dataclass(frozen=True)
class Workload:
    name: str
    wid: int        # workload id, fixes the seeds
    M: int
    N: int
    K: int
    scale: float    # standard deviation of the entries (nominal sigma)
    sampled: bool   # oracle checks sampled entries + full rows rather than all of C


WORKLOADS = {
    "gemm_256": Workload("gemm_256", 1, 256, 256, 256, 1.0, False),
    "gemm_4096": Workload("gemm_4096", 2, 4096, 4096, 4096, 1.0, False),
    "gemm_8192": Workload("gemm_8192", 3, 8192, 8192, 8192, 0.5, True),
    "gemm_16384": Workload("gemm_16384", 4, 16384, 16384, 16384, 1.0, True),
    "proj_16384x28672x8192": Workload("proj_16384x28672x8192", 5, 16384, 28672, 8192, 0.02, True),
    "skinny_128x28672x8192": Workload("skinny_128x28672x8192", 6, 128, 28672, 8192, 0.02, False),
    # decode-regime projections (one token; a batch of 64) over a 448 MiB weight matrix, 3.5x the L2
    "decode_1x28672x8192": Workload("decode_1x28672x8192", 11, 1, 28672, 8192, 0.02, False),
    "decode_64x8192x28672": Workload("decode_64x8192x28672", 12, 64, 8192, 28672, 0.02, True),
    # 256 rows over an 8192 x 8192 weight matrix: just below the roofline knee (the 256x128 pair's shape)
    "decode_256x8192x8192": Workload("decode_256x8192x8192", 13, 256, 8192, 8192, 0.02, True),
}

# FP8 (E4M3) workloads: operands N(0,1) rounded to E4M3, per-tensor scales
# (the FP8 GEMM of the pages, headline shape 8192^3).
FP8_WORKLOADS = {
    "fp8_gemm_8192": Workload("fp8_gemm_8192", 7, 8192, 8192, 8192, 1.0, True),
    "fp8_gemm_256": Workload("fp8_gemm_256", 8, 256, 256, 256, 1.0, False),
}
FP8_SCALES = (0.5, 0.25)   # scale_a, scale_b of the FP8 workloads

# MXFP8 workloads: E4M3 operands N(0,1) and UE8M0 block scales (one per 32 K
# elements) uniform on [124, 130], i.e. 2^-3 .. 2^3, seeds 3100/3200 + id.
MX_WORKLOADS = {
    "mxfp8_gemm_8192": Workload("mxfp8_gemm_8192", 9, 8192, 8192, 8192, 1.0, True),
    "mxfp8_gemm_256": Workload("mxfp8_gemm_256", 10, 256, 256, 256, 1.0, False),
}


def mx_scales(rows: int, blocks: int, seed: int, lo: int = 124, hi: int = 130) -> np.ndarray:
    """rows × blocks UE8M0 scale bytes uniform on {lo..hi}."""
    g = np.random.Generator(np.random.PCG64(seed))
    return g.integers(lo, hi + 1, size=(rows, blocks)).astype(np.uint8)


def operands_mx(w: Workload) -> tuple[np.ndarray, np.ndarray, np.ndarray, np.ndarray]:
    """(A, B, SA, SB) for an MXFP8 workload."""
    A, B = normal_e4m3(w.M, w.K, 1000 + w.wid), normal_e4m3(w.N, w.K, 2000 + w.wid)
    return A, B, mx_scales(w.M, w.K // 32, 3100 + w.wid), mx_scales(w.N, w.K // 32, 3200 + w.wid)


@dataclass(frozen=True)
class AttnWorkload:
    name: str
    wid: int
    B: int
    Hq: int
    Hkv: int
    S: int
    D: int
    causal: bool
    sampled: bool   # oracle checks sampled rows rather than every row


ATTN_WORKLOADS = {
    "attn_gqa_b16_s4096_d128": AttnWorkload("attn_gqa_b16_s4096_d128", 20, 16, 64, 8, 4096, 128, False, True),
    "attn_gqa_b16_s4096_d128_causal": AttnWorkload("attn_gqa_b16_s4096_d128_causal", 21, 16, 64, 8, 4096, 128,
                                                   True, True),
    "attn_gqa_b16_s4096_d64": AttnWorkload("attn_gqa_b16_s4096_d64", 22, 16, 64, 8, 4096, 64, False, True),
    "attn_gqa_small": AttnWorkload("attn_gqa_small", 23, 2, 8, 2, 300, 128, False, False),
    "attn_gqa_b2_s4096_d128": AttnWorkload("attn_gqa_b2_s4096_d128", 24, 2, 64, 8, 4096, 128, False, True),
}


def attn_operands(w: AttnWorkload) -> tuple[np.ndarray, np.ndarray, np.ndarray]:
    """(Q, K, V) bf16 bits for an attention workload, shapes [B, H, S, D]."""
    Q = normal_bf16(w.B * w.Hq * w.S, w.D, 4000 + w.wid).reshape(w.B, w.Hq, w.S, w.D)
    K = normal_bf16(w.B * w.Hkv * w.S, w.D, 5000 + w.wid).reshape(w.B, w.Hkv, w.S, w.D)
    V = normal_bf16(w.B * w.Hkv * w.S, w.D, 6000 + w.wid).reshape(w.B, w.Hkv, w.S, w.D)
    return Q, K, V


def operands_fp8(w: Workload, integer: bool = False) -> tuple[np.ndarray, np.ndarray]:
    """(A, B) E4M3 codes for an FP8 workload."""
    if integer:
        return int_e4m3(w.M, w.K, 1100 + w.wid), int_e4m3(w.N, w.K, 2100 + w.wid)
    return (normal_e4m3(w.M, w.K, 1000 + w.wid, w.scale), normal_e4m3(w.N, w.K, 2000 + w.wid, w.scale))


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit patterns, round-to-nearest-even on the low 16 bits.

    Inputs are finite (normal draws); NaN handling is not needed here.
    """
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    lsb = (u >> np.uint32(16)) & np.uint32(1)
    return ((u + np.uint32(0x7FFF) + lsb) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(h: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> float32 values (exact)."""
    return (np.asarray(h, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def _e4m3_table():
    """Non-negative finite E4M3 values for codes 0x00..0x7E (ascending)."""
    codes = np.arange(0x7F, dtype=np.int64)
    e = codes >> 3
    m = codes & 7
    vals = np.where(e == 0, m / 8.0 * 2.0 ** -6, (1.0 + m / 8.0) * np.exp2(e - 7.0))
    return vals


_E4M3 = _e4m3_table()


def f32_to_e4m3_codes(x: np.ndarray) -> np.ndarray:
    """float32 -> E4M3 codes: nearest representable value, ties to the even
    code, magnitudes above 448 saturate to 448."""
    x = np.asarray(x, dtype=np.float64)
    a = np.minimum(np.abs(x), _E4M3[-1])
    hi = np.clip(np.searchsorted(_E4M3, a, side="left"), 0, len(_E4M3) - 1)
    lo = np.clip(hi - 1, 0, len(_E4M3) - 1)
    dlo = np.abs(a - _E4M3[lo])
    dhi = np.abs(_E4M3[hi] - a)
    pick = np.where(dlo < dhi, lo, np.where(dhi < dlo, hi, np.where(lo % 2 == 0, lo, hi)))
    sign = (np.signbit(x) & (pick != 0)).astype(np.int64) << 7
    return (pick | sign).astype(np.uint8)


def normal_e4m3(rows: int, cols: int, seed: int, scale: float = 1.0) -> np.ndarray:
    """rows×cols E4M3 codes of N(0,1)·scale, drawn row-major from PCG64(seed)."""
    g = np.random.Generator(np.random.PCG64(seed))
    out = np.empty(rows * cols, dtype=np.uint8)
    s = np.float32(scale)
    for off in range(0, rows * cols, _CHUNK):
        n = min(_CHUNK, rows * cols - off)
        x = g.standard_normal(n, dtype=np.float32)
        if scale != 1.0:
            x *= s
        out[off:off + n] = f32_to_e4m3_codes(x)
    return out.reshape(rows, cols)


def int_e4m3(rows: int, cols: int, seed: int, lo: int = -4, hi: int = 4) -> np.ndarray:
    """rows×cols E4M3 codes of integers uniform on {lo..hi} (exact in E4M3)."""
    g = np.random.Generator(np.random.PCG64(seed))
    return f32_to_e4m3_codes(g.integers(lo, hi + 1, size=(rows, cols)).astype(np.float32))


def normal_bf16(rows: int, cols: int, seed: int, scale: float = 1.0) -> np.ndarray:
    """rows×cols bf16 bits of N(0,1)·scale, drawn row-major from PCG64(seed)."""
    g = np.random.Generator(np.random.PCG64(seed))
    out = np.empty(rows * cols, dtype=np.uint16)
    s = np.float32(scale)
    for off in range(0, rows * cols, _CHUNK):
        n = min(_CHUNK, rows * cols - off)
        x = g.standard_normal(n, dtype=np.float32)
        if scale != 1.0:
            x *= s
        out[off:off + n] = f32_to_bf16_bits(x)
    return out.reshape(rows, cols)


def int_bf16(rows: int, cols: int, seed: int, lo: int = -4, hi: int = 4) -> np.ndarray:
    """rows×cols bf16 bits of integers uniform on {lo..hi}."""
    g = np.random.Generator(np.random.PCG64(seed))
    x = g.integers(lo, hi + 1, size=(rows, cols)).astype(np.float32)
    return f32_to_bf16_bits(x)


def operands(w: Workload, integer: bool = False) -> tuple[np.ndarray, np.ndarray]:
    """(A, B) bf16 bits for a workload: A is M×K, B is N×K."""
    if integer:
        return int_bf16(w.M, w.K, 1100 + w.wid), int_bf16(w.N, w.K, 2100 + w.wid)
    return (normal_bf16(w.M, w.K, 1000 + w.wid, w.scale),
            normal_bf16(w.N, w.K, 2000 + w.wid, w.scale))


def sample_positions(M: int, N: int, seed: int, count: int = 4096,
                     tile_m: int = 128, tile_n: int = 256) -> tuple[np.ndarray, np.ndarray]:
    """Seeded output positions: uniform draws plus the corners of C and the
    first/last row and column of every tile along the edges of the tile grid."""
    g = np.random.Generator(np.random.PCG64(seed))
    r = list(g.integers(0, M, size=count))
    c = list(g.integers(0, N, size=count))
    edge_r = sorted({0, M - 1} | {min(M - 1, x) for t in range(0, M, tile_m) for x in (t, t + tile_m - 1)})
    edge_c = sorted({0, N - 1} | {min(N - 1, x) for t in range(0, N, tile_n) for x in (t, t + tile_n - 1)})
    for i in (0, M - 1):
        for j in edge_c:
            r.append(i)
            c.append(j)
    for j in (0, N - 1):
        for i in edge_r:
            r.append(i)
            c.append(j)
    return np.asarray(r, dtype=np.int64), np.asarray(c, dtype=np.int64)


def full_rows(M: int, seed: int, count: int = 8) -> np.ndarray:
    """``count`` distinct seeded row indices including rows 0 and M-1."""
    g = np.random.Generator(np.random.PCG64(seed + 7))
    rows = {0, M - 1}
    while len(rows) < min(count, M):
        rows.add(int(g.integers(0, M)))
    return np.asarray(sorted(rows), dtype=np.int64)
