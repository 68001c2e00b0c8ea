"""Shared helpers of the GPU parity tests (host-side marshalling and the
tolerance written in the tests)."""
from __future__ import annotations

import numpy as np

import synth

SENTINEL = 0x7FBF   # a NaN bit pattern no GEMM result can produce from finite inputs


def to_device(bits: np.ndarray, rows_pad: int = 0, cols_pad: int = 0, fill: int = 0):
    """uint16 bf16 bits -> bf16 CUDA tensor; optional padded storage (a view
    into a larger allocation) to exercise leading dimensions > cols."""
    import torch
    r, c = bits.shape
    store = np.full((r + rows_pad, c + cols_pad), fill, dtype=np.uint16)
    store[:r, :c] = bits
    t = torch.from_numpy(store.view(np.int16)).to("cuda").view(torch.bfloat16)
    return t[:r, :c], t


def to_host(t) -> np.ndarray:
    import torch
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def tolerance(ref_bits: np.ndarray, K: int, sigma_a: float, sigma_b: float) -> np.ndarray:
    """Per-entry bound |C_gpu - C_ref| <= 2^-7·|C_ref| + 2^-12·sqrt(K)·σ_A·σ_B.

    2^-7·|C_ref| is at most one bf16 ulp of the value (a rounding-boundary
    flip between fp32 and exact accumulation); the absolute term covers fp32
    cancellation near zero (fp32 error ≈ 2^-24·sqrt(K)·σ_A·σ_B, far below it).
    σ are the generator's nominal standard deviations."""
    ref = synth.bf16_bits_to_f32(ref_bits).astype(np.float64)
    return 2.0 ** -7 * np.abs(ref) + 2.0 ** -12 * np.sqrt(max(K, 1)) * sigma_a * sigma_b


def assert_close(got_bits: np.ndarray, ref_bits: np.ndarray, K: int, sigma_a: float, sigma_b: float,
                 what: str = ""):
    got = synth.bf16_bits_to_f32(got_bits).astype(np.float64)
    ref = synth.bf16_bits_to_f32(ref_bits).astype(np.float64)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    err = np.abs(got - ref)
    tol = tolerance(ref_bits, K, sigma_a, sigma_b)
    bad = err > tol
    if bad.any():
        idx = np.argwhere(bad)[:5]
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} entries outside tolerance; first "
                             f"{idx.tolist()} got {got[bad][:5]} want {ref[bad][:5]}")


def assert_bitexact(got_bits: np.ndarray, ref_bits: np.ndarray, what: str = ""):
    """Bit-exact, except that +0 and -0 compare equal (the sign of an exact
    zero depends on where the accumulation starts, which the method leaves open)."""
    same = (got_bits == ref_bits) | (((got_bits & 0x7FFF) == 0) & ((ref_bits & 0x7FFF) == 0))
    if not same.all():
        idx = np.argwhere(~same)[:5]
        raise AssertionError(f"{what}: {int((~same).sum())} of {same.size} entries differ; first {idx.tolist()}: "
                             f"got {[hex(int(x)) for x in got_bits[~same][:5]]} "
                             f"want {[hex(int(x)) for x in ref_bits[~same][:5]]}")


def isnan_bf16(bits: np.ndarray) -> np.ndarray:
    """NaN bit patterns of bf16 (any payload)."""
    return ((bits & 0x7F80) == 0x7F80) & ((bits & 0x007F) != 0)


def assert_same_ieee(got: np.ndarray, want: np.ndarray, what: str = ""):
    """NaN in the same places (payloads may differ), every other entry bit-exact."""
    gn, wn = isnan_bf16(got), isnan_bf16(want)
    assert np.array_equal(gn, wn), f"{what}: NaN at {np.argwhere(gn != wn)[:5].tolist()}"
    assert np.array_equal(got[~gn], want[~wn]), f"{what}: differs at {np.argwhere((got != want) & ~gn)[:5].tolist()}"
