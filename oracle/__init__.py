"""CPU oracle for the dense BF16 GEMM C = A·Bᵀ — TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package. The CUDA library never imports, links or
calls it, and the two share no code: the product path has no CPU fallback.

The arithmetic lives in ``gemm_ref.c`` (plain C, binary64): the exact
definition of the operation on the HipKittens "L2" detail page, §3 "Target
operation" table (BF16 GEMM: bf16 in, FP32 accumulate, bf16 out) with the
second operand used transposed as in the "ABt" GEMM of §7/§9.2:

    C[i, j] = RNE_bf16( Σ_k  A[i, k] · B[j, k] )      (sum in binary64)

It also holds the fused-epilogue GEMM (bias + activation + residual), the FP8 (E4M3)
GEMM with per-tensor scales, and the attention forward of the same page's
"MHA fwd" / "GQA fwd" rows (softmax(Q·Kᵀ/√D)·V, bf16 in and out).

This module only marshals numpy arrays of bf16 bit patterns (``uint16``) to
that C code. Every function here is pinned by ``tests/test_oracle_pins.py``
and ``tests/test_oracle_attention_pins.py`` against exact rational
arithmetic, closed forms and invariants.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gemm_ref.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")

_lib = None
_lock = threading.Lock()

_I64 = ctypes.c_int64
_P = ctypes.c_void_p


def build(force: bool = False) -> str:
    """Compile ``gemm_ref.c`` into ``oracle/_build/liboracle.so`` with gcc."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-std=c99", "-O2", "-ffp-contract=off", "-fno-fast-math",
           "-fPIC", "-shared", "-pthread", "-D_GNU_SOURCE", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            lib.oracle_round_bf16.argtypes = [ctypes.c_double]
            lib.oracle_round_bf16.restype = ctypes.c_uint16
            lib.oracle_dot_f64.argtypes = [_P, _P, _I64, _I64, _I64, _I64, _I64]
            lib.oracle_dot_f64.restype = ctypes.c_double
            lib.oracle_gemm_bf16.argtypes = [_P, _P, _P, _I64, _I64, _I64, _I64, _I64, _I64,
                                             ctypes.c_int]
            lib.oracle_gemm_bf16.restype = ctypes.c_int
            lib.oracle_gemm_bf16_rows.argtypes = [_P, _P, _P, _I64, _I64, _I64, _I64, _P, _I64,
                                                  ctypes.c_int]
            lib.oracle_gemm_bf16_rows.restype = ctypes.c_int
            lib.oracle_gemm_bf16_entries.argtypes = [_P, _P, _P, _I64, _I64, _I64, _P, _P, _I64,
                                                     ctypes.c_int]
            lib.oracle_gemm_bf16_entries.restype = ctypes.c_int
            lib.oracle_activation.argtypes = [ctypes.c_double, ctypes.c_int]
            lib.oracle_activation.restype = ctypes.c_double
            lib.oracle_gemm_bf16_epilogue.argtypes = [_P, _P, _P, _P, _I64, _I64, _I64, _I64, _I64, _I64,
                                                      ctypes.c_int, ctypes.c_int]
            lib.oracle_gemm_bf16_epilogue.restype = ctypes.c_int
            lib.oracle_gemm_bf16_epilogue_entries.argtypes = [_P, _P, _P, _P, _I64, _I64, _I64, ctypes.c_int,
                                                              _P, _P, _I64, ctypes.c_int]
            lib.oracle_gemm_bf16_epilogue_entries.restype = ctypes.c_int
            lib.oracle_gemm_bf16_fused.argtypes = [_P, _P, _P, _P, _I64, _P, _I64, _I64, _I64, _I64, _I64, _I64,
                                                   ctypes.c_int, ctypes.c_int]
            lib.oracle_gemm_bf16_fused.restype = ctypes.c_int
            lib.oracle_gemm_bf16_fused_entries.argtypes = [_P, _P, _P, _P, _I64, _P, _I64, _I64, _I64, ctypes.c_int,
                                                           _P, _P, _I64, ctypes.c_int]
            lib.oracle_gemm_bf16_fused_entries.restype = ctypes.c_int
            lib.oracle_e4m3_to_double.argtypes = [ctypes.c_uint8]
            lib.oracle_e4m3_to_double.restype = ctypes.c_double
            lib.oracle_gemm_fp8e4m3.argtypes = [_P, _P, _P, _I64, _I64, _I64, _I64, _I64, _I64, ctypes.c_double,
                                                ctypes.c_int]
            lib.oracle_gemm_fp8e4m3.restype = ctypes.c_int
            lib.oracle_gemm_fp8e4m3_entries.argtypes = [_P, _P, _P, _I64, _I64, _I64, ctypes.c_double, _P, _P,
                                                        _I64, ctypes.c_int]
            lib.oracle_gemm_fp8e4m3_entries.restype = ctypes.c_int
            lib.oracle_ue8m0_to_double.argtypes = [ctypes.c_uint8]
            lib.oracle_ue8m0_to_double.restype = ctypes.c_double
            lib.oracle_gemm_mxfp8.argtypes = [_P, _P, _P, _P, _P, _I64, _I64, _I64, _I64, _I64, _I64, _I64, _I64,
                                              ctypes.c_int]
            lib.oracle_gemm_mxfp8.restype = ctypes.c_int
            lib.oracle_gemm_mxfp8_entries.argtypes = [_P, _P, _P, _P, _P, _I64, _I64, _I64, _I64, _I64, _P, _P,
                                                      _I64, ctypes.c_int]
            lib.oracle_gemm_mxfp8_entries.restype = ctypes.c_int
            lib.oracle_attention_fwd.argtypes = [_P, _P, _P, _P, _P, _I64, _I64, _I64, _I64, _I64, ctypes.c_int,
                                                 _I64, _I64, ctypes.c_int]
            lib.oracle_attention_fwd.restype = ctypes.c_int
            _lib = lib
    return _lib


def _as_bits(x: np.ndarray, name: str) -> np.ndarray:
    if x.dtype != np.uint16 or x.ndim != 2:
        raise TypeError(f"{name} must be a 2-D uint16 array of bf16 bit patterns")
    if x.shape[1] > 1 and x.strides[1] != 2 or x.strides[0] % 2:
        raise ValueError(f"{name} must have a unit stride along K")
    return x


def _ptr(x: np.ndarray) -> int:
    return x.ctypes.data


def round_bf16(x: float) -> int:
    """binary64 -> bf16 bit pattern, IEEE round-to-nearest-even."""
    return int(_load().oracle_round_bf16(float(x)))


def dot_f64(A: np.ndarray, B: np.ndarray, i: int, j: int) -> float:
    """The unrounded binary64 sum Σ_k A[i,k]·B[j,k] (increasing k)."""
    A = _as_bits(A, "A")
    B = _as_bits(B, "B")
    K = A.shape[1]
    assert B.shape[1] == K
    return float(_load().oracle_dot_f64(_ptr(A), _ptr(B), K, A.strides[0] // 2,
                                        B.strides[0] // 2, int(i), int(j)))


def gemm(A: np.ndarray, B: np.ndarray, threads: int = 0) -> np.ndarray:
    """Full C = RNE_bf16(A·Bᵀ): A (M×K), B (N×K) bf16 bits -> C (M×N) bf16 bits."""
    A = _as_bits(A, "A")
    B = _as_bits(B, "B")
    M, K = A.shape
    N, K2 = B.shape
    if K != K2:
        raise ValueError("A and B disagree on K")
    C = np.zeros((M, N), dtype=np.uint16)
    if M and N:
        _load().oracle_gemm_bf16(_ptr(A), _ptr(B), _ptr(C), M, N, K, max(A.strides[0] // 2, K),
                                 max(B.strides[0] // 2, K), N, int(threads))
    return C


def gemm_rows(A: np.ndarray, B: np.ndarray, rows, threads: int = 0) -> tuple[np.ndarray, int]:
    """Full rows ``rows`` of C. Returns (len(rows)×N bf16 bits, threads used)."""
    A = _as_bits(A, "A")
    B = _as_bits(B, "B")
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    M, K = A.shape
    N = B.shape[0]
    if rows.size and (rows.min() < 0 or rows.max() >= M):
        raise IndexError("row index out of range")
    out = np.zeros((rows.size, N), dtype=np.uint16)
    used = 0
    if rows.size and N:
        used = _load().oracle_gemm_bf16_rows(_ptr(A), _ptr(B), _ptr(out), N, K,
                                             A.strides[0] // 2, B.strides[0] // 2,
                                             _ptr(rows), rows.size, int(threads))
    return out, used


def gemm_entries(A: np.ndarray, B: np.ndarray, rows, cols, threads: int = 0) -> tuple[np.ndarray, int]:
    """Entries C[rows[t], cols[t]]. Returns (bf16 bits per entry, threads used)."""
    A = _as_bits(A, "A")
    B = _as_bits(B, "B")
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    cols = np.ascontiguousarray(np.asarray(cols, dtype=np.int64))
    if rows.shape != cols.shape:
        raise ValueError("rows and cols differ in length")
    M, K = A.shape
    N = B.shape[0]
    if rows.size and (rows.min() < 0 or rows.max() >= M or cols.min() < 0 or cols.max() >= N):
        raise IndexError("entry index out of range")
    out = np.zeros(rows.size, dtype=np.uint16)
    used = 0
    if rows.size:
        used = _load().oracle_gemm_bf16_entries(_ptr(A), _ptr(B), _ptr(out), K,
                                                A.strides[0] // 2, B.strides[0] // 2,
                                                _ptr(rows), _ptr(cols), rows.size, int(threads))
    return out, used


# ---- fused epilogue: C = RNE_bf16(act(A·Bᵀ + bias)) -----------------------
ACT_NONE, ACT_RELU, ACT_GELU, ACT_SILU = 0, 1, 2, 3


def activation(x: float, act: int) -> float:
    """The activation in binary64 (0 none, 1 ReLU, 2 GELU with erf, 3 SiLU)."""
    return float(_load().oracle_activation(float(x), int(act)))


def _bias_ptr(bias, N):
    if bias is None:
        return None, 0
    bias = np.ascontiguousarray(np.asarray(bias, dtype=np.uint16))
    if bias.shape != (N,):
        raise ValueError("bias must hold N bf16 values")
    return bias, bias.ctypes.data


def _residual(residual, M, N):
    """(array kept alive, pointer, leading dimension in elements) of an M×N bf16 residual, or (None, None, 0)."""
    if residual is None:
        return None, None, 0
    if residual.dtype != np.uint16 or residual.ndim != 2 or residual.shape != (M, N):
        raise TypeError(f"residual must be an {M}x{N} uint16 array of bf16 bit patterns")
    if N > 1 and residual.strides[1] != 2 or residual.strides[0] % 2:
        raise ValueError("residual must have a unit stride along N")
    return residual, _ptr(residual), max(residual.strides[0] // 2, N)


def gemm_epilogue(A: np.ndarray, B: np.ndarray, bias=None, act: int = ACT_NONE, threads: int = 0,
                  residual=None) -> np.ndarray:
    """C = RNE_bf16(act(A·Bᵀ + bias) + R), bias a length-N bf16 vector or None,
    R (``residual``) an M×N bf16 matrix or None."""
    A = _as_bits(A, "A")
    B = _as_bits(B, "B")
    M, K = A.shape
    N = B.shape[0]
    keep, bptr = _bias_ptr(bias, N)
    keep_r, rptr, ldr = _residual(residual, M, N)
    C = np.zeros((M, N), dtype=np.uint16)
    if M and N:
        if rptr is None:
            _load().oracle_gemm_bf16_epilogue(_ptr(A), _ptr(B), bptr, _ptr(C), M, N, K, max(A.strides[0] // 2, K),
                                              max(B.strides[0] // 2, K), N, int(act), int(threads))
        else:
            _load().oracle_gemm_bf16_fused(_ptr(A), _ptr(B), bptr, rptr, ldr, _ptr(C), M, N, K,
                                           max(A.strides[0] // 2, K), max(B.strides[0] // 2, K), N, int(act),
                                           int(threads))
    return C


def gemm_epilogue_entries(A: np.ndarray, B: np.ndarray, rows, cols, bias=None, act: int = ACT_NONE,
                          threads: int = 0, residual=None) -> np.ndarray:
    """Entries of RNE_bf16(act(A·Bᵀ + bias) + R) at (rows[t], cols[t])."""
    A = _as_bits(A, "A")
    B = _as_bits(B, "B")
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    cols = np.ascontiguousarray(np.asarray(cols, dtype=np.int64))
    keep, bptr = _bias_ptr(bias, B.shape[0])
    keep_r, rptr, ldr = _residual(residual, A.shape[0], B.shape[0])
    out = np.zeros(rows.size, dtype=np.uint16)
    if rows.size:
        if rows.min() < 0 or rows.max() >= A.shape[0] or cols.min() < 0 or cols.max() >= B.shape[0]:
            raise IndexError("entry index out of range")
        if rptr is None:
            _load().oracle_gemm_bf16_epilogue_entries(_ptr(A), _ptr(B), bptr, _ptr(out), A.shape[1],
                                                      A.strides[0] // 2, B.strides[0] // 2, int(act), _ptr(rows),
                                                      _ptr(cols), rows.size, int(threads))
        else:
            _load().oracle_gemm_bf16_fused_entries(_ptr(A), _ptr(B), bptr, rptr, ldr, _ptr(out), A.shape[1],
                                                   A.strides[0] // 2, B.strides[0] // 2, int(act), _ptr(rows),
                                                   _ptr(cols), rows.size, int(threads))
    return out


# ---- FP8 (E4M3) GEMM with per-tensor scales ------------------------------

def e4m3_value(code: int) -> float:
    """Exact value of an E4M3 byte (NaN for S.1111.111)."""
    return float(_load().oracle_e4m3_to_double(int(code) & 0xFF))


def _as_bytes(x: np.ndarray, name: str) -> np.ndarray:
    if x.dtype != np.uint8 or x.ndim != 2:
        raise TypeError(f"{name} must be a 2-D uint8 array of E4M3 codes")
    if x.shape[1] > 1 and x.strides[1] != 1:
        raise ValueError(f"{name} must have a unit stride along K")
    return x


def gemm_fp8(A: np.ndarray, B: np.ndarray, scale_a: float = 1.0, scale_b: float = 1.0,
             threads: int = 0) -> np.ndarray:
    """C = RNE_bf16(sa·sb·A·Bᵀ) for E4M3 codes A (M×K), B (N×K); sa, sb are float32 values."""
    A = _as_bytes(A, "A")
    B = _as_bytes(B, "B")
    M, K = A.shape
    N = B.shape[0]
    C = np.zeros((M, N), dtype=np.uint16)
    scale = float(np.float32(scale_a)) * float(np.float32(scale_b))
    if M and N:
        _load().oracle_gemm_fp8e4m3(_ptr(A), _ptr(B), _ptr(C), M, N, K, max(A.strides[0], K), max(B.strides[0], K),
                                    N, scale, int(threads))
    return C


def gemm_fp8_entries(A: np.ndarray, B: np.ndarray, rows, cols, scale_a: float = 1.0, scale_b: float = 1.0,
                     threads: int = 0) -> np.ndarray:
    A = _as_bytes(A, "A")
    B = _as_bytes(B, "B")
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    cols = np.ascontiguousarray(np.asarray(cols, dtype=np.int64))
    out = np.zeros(rows.size, dtype=np.uint16)
    scale = float(np.float32(scale_a)) * float(np.float32(scale_b))
    if rows.size:
        _load().oracle_gemm_fp8e4m3_entries(_ptr(A), _ptr(B), _ptr(out), A.shape[1], A.strides[0], B.strides[0],
                                            scale, _ptr(rows), _ptr(cols), rows.size, int(threads))
    return out


# ---- MXFP8 GEMM ------------------------------------------------------------

def ue8m0_value(code: int) -> float:
    """Value of a UE8M0 scale byte: 2^(E-127), NaN for 255."""
    return float(_load().oracle_ue8m0_to_double(int(code) & 0xFF))


def _mx_args(A, B, SA, SB):
    A = _as_bytes(A, "A")
    B = _as_bytes(B, "B")
    M, K = A.shape
    N = B.shape[0]
    if K % 32:
        raise ValueError("K must be a multiple of the block size 32")
    for x, rows, name in ((SA, M, "SA"), (SB, N, "SB")):
        if x.dtype != np.uint8 or x.shape != (rows, K // 32) or (x.shape[1] > 1 and x.strides[1] != 1):
            raise TypeError(f"{name} must be a uint8 array of shape ({rows}, K/32) with unit stride")
    return A, B, M, N, K


def gemm_mxfp8(A: np.ndarray, B: np.ndarray, SA: np.ndarray, SB: np.ndarray, threads: int = 0) -> np.ndarray:
    """C = RNE_bf16(Σ_b SA·SB·Σ_block A·B) for E4M3 codes A (M×K), B (N×K) and
    UE8M0 block scales SA (M×K/32), SB (N×K/32)."""
    A, B, M, N, K = _mx_args(A, B, SA, SB)
    C = np.zeros((M, N), dtype=np.uint16)
    if M and N:
        _load().oracle_gemm_mxfp8(_ptr(A), _ptr(B), _ptr(SA), _ptr(SB), _ptr(C), M, N, K, max(A.strides[0], K),
                                  max(B.strides[0], K), max(SA.strides[0], K // 32), max(SB.strides[0], K // 32), N,
                                  int(threads))
    return C


def gemm_mxfp8_entries(A, B, SA, SB, rows, cols, threads: int = 0) -> np.ndarray:
    A, B, M, N, K = _mx_args(A, B, SA, SB)
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    cols = np.ascontiguousarray(np.asarray(cols, dtype=np.int64))
    out = np.zeros(rows.size, dtype=np.uint16)
    if rows.size:
        _load().oracle_gemm_mxfp8_entries(_ptr(A), _ptr(B), _ptr(SA), _ptr(SB), _ptr(out), K, A.strides[0],
                                          B.strides[0], max(SA.strides[0], K // 32), max(SB.strides[0], K // 32),
                                          _ptr(rows), _ptr(cols), rows.size, int(threads))
    return out


# ---- attention forward (GQA) ---------------------------------------------

def attention_fwd(Q: np.ndarray, K: np.ndarray, V: np.ndarray, causal: bool = False, rows=None,
                  threads: int = 0, with_lse: bool = False):
    """O = softmax(Q·Kᵀ/√D)·V per (batch, head), GQA head groups, bf16 bits in
    and out; Q [B, Hq, S, D], K and V [B, Hkv, S, D]. ``rows`` = (begin, end)
    of the flattened (b, h, i) rows to compute (others stay 0). With
    ``with_lse`` also returns the float64 log-sum-exp of each row's scaled
    scores, shape [B, Hq, S] (NaN where not computed)."""
    for name, x in (("Q", Q), ("K", K), ("V", V)):
        if x.dtype != np.uint16 or x.ndim != 4 or not x.flags.c_contiguous:
            raise TypeError(f"{name} must be a contiguous 4-D uint16 array of bf16 bits")
    B, Hq, S, D = Q.shape
    Hkv = K.shape[1]
    if K.shape != (B, Hkv, S, D) or V.shape != K.shape or Hq % Hkv:
        raise ValueError("shapes do not form a GQA attention")
    O = np.zeros_like(Q)
    lse = np.full((B, Hq, S), np.nan) if with_lse else None
    r0, r1 = (0, B * Hq * S) if rows is None else rows
    if r1 > r0:
        _load().oracle_attention_fwd(_ptr(Q), _ptr(K), _ptr(V), _ptr(O), _ptr(lse) if with_lse else None,
                                     B, Hq, Hkv, S, D, int(bool(causal)), int(r0), int(r1), int(threads))
    return (O, lse) if with_lse else O
