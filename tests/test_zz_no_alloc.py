"""The GEMM entry point that allocates nothing (hk_gemm_bf16_noalloc).

It exists for callers that cannot call cudaMalloc when they run a GEMM — for
example code running inside a memory pool that owns all device memory, or a
hook of an allocator that must not re-enter it. Its K-split scratch lives in
a fixed array inside the library. These tests call it through the C-ABI and
check it against the CPU oracle (bit for bit on integer data, within the
parity tolerance on normal data) and against the ordinary entry point
hk_gemm_bf16 on the same inputs, on calls in a row: every call finds the
previous call's leftovers in the shared array, including NaN partials from a
larger call with another split and another padded width.

This file is named so that pytest collects it last.
"""
from __future__ import annotations

import numpy as np
import pytest

import oracle
import synth
from gpu_util import assert_bitexact, assert_close, to_device, to_host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def hk():
    import torch
    if not torch.cuda.is_available():
        pytest.fail("no CUDA device")
    import dense_bf16_gemm_02_gb300 as pkg
    pkg.load()
    return pkg


def _noalloc(hk, A_bits, B_bits, split_k):
    """C from hk_gemm_bf16_noalloc (host bf16 bits); the status word must stay clear."""
    import torch
    M, K = A_bits.shape
    N = B_bits.shape[0]
    A, _ = to_device(A_bits)
    B, _ = to_device(B_bits)
    C = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    stream = int(torch.cuda.current_stream().cuda_stream)
    st = hk.hk_gemm_bf16_noalloc(A.data_ptr(), B.data_ptr(), C.data_ptr(), M, N, K, K, K, N, split_k, stream)
    assert st == hk.HK_OK, hk.hk_gemm_last_error_string()
    torch.cuda.synchronize()
    assert hk.hk_gemm_last_device_status(torch.cuda.current_device()) == hk.HK_OK
    return to_host(C)


def _ordinary(hk, A_bits, B_bits):
    import torch
    M, K = A_bits.shape
    N = B_bits.shape[0]
    A, _ = to_device(A_bits)
    B, _ = to_device(B_bits)
    C = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    st = hk.hk_gemm_bf16(A.data_ptr(), B.data_ptr(), C.data_ptr(), M, N, K, K, K, N,
                         int(torch.cuda.current_stream().cuda_stream))
    assert st == hk.HK_OK, hk.hk_gemm_last_error_string()
    torch.cuda.synchronize()
    return to_host(C)


def _poison_scratch(hk):
    """A forced-split call with NaN inputs: its fp32 partials (NaN) stay in the shared array."""
    M, N, K = 128, 4096, 4096
    nan = np.full((M, K), 0x7FC0, dtype=np.uint16)
    B = synth.int_bf16(N, K, 5)
    got = _noalloc(hk, nan, B, 8)
    assert np.all((got & 0x7F80) == 0x7F80) and np.all(got & 0x7F), "NaN inputs must give NaN"


@pytest.mark.parametrize("split_k", [0, 4])
def test_noalloc_matches_oracle_and_ordinary_entry_point_twice(hk, split_k):
    M, N, K = 64, 2048, 8192
    _poison_scratch(hk)
    for call in range(2):      # two calls in a row on the shared scratch, different inputs
        A = synth.normal_bf16(M, K, 700 + call)
        B = synth.normal_bf16(N, K, 800 + call)
        got = _noalloc(hk, A, B, split_k)
        assert_close(got, oracle.gemm(A, B), K, 1.0, 1.0, f"no-alloc vs oracle, call {call + 1}, split_k={split_k}")
        assert_close(got, _ordinary(hk, A, B), K, 1.0, 1.0, f"no-alloc vs hk_gemm_bf16, call {call + 1}")


def test_noalloc_integer_inputs_are_bit_exact(hk):
    _poison_scratch(hk)
    for call, (M, N, K, split) in enumerate([(100, 1000, 4096, 5), (37, 1496, 2056, 3), (130, 520, 1024, 2)]):
        A = synth.int_bf16(M, K, 900 + call)
        B = synth.int_bf16(N, K, 950 + call)
        got = _noalloc(hk, A, B, split)
        assert_bitexact(got, oracle.gemm(A, B), f"no-alloc integer call {call + 1} (split {split})")
        assert_bitexact(got, _ordinary(hk, A, B), f"no-alloc vs hk_gemm_bf16, call {call + 1}")


def test_noalloc_automatic_split_beyond_the_array_runs_unsplit(hk):
    """A shape whose automatic K split would need more scratch than the array
    holds (32 MiB) runs without a split; sampled entries against the oracle."""
    limit = 32 << 20
    shape = None
    for M, N, K in [(192, 8192, 16384), (512, 6144, 16384), (768, 4096, 16384), (256, 4096, 32768),
                    (128, 8192, 8192), (256, 8192, 16384)]:
        plan = hk.Plan(M, N, K)
        if plan.workspace_size > limit:
            shape = (M, N, K)
            plan.close()
            break
        plan.close()
    assert shape is not None, "no candidate shape splits K beyond the fixed array"
    M, N, K = shape
    A = synth.normal_bf16(M, K, 961)
    B = synth.normal_bf16(N, K, 962)
    got = _noalloc(hk, A, B, 0)
    r, c = synth.sample_positions(M, N, 963, count=2048)
    ref, _ = oracle.gemm_entries(A, B, r, c)
    assert_close(got[r, c], ref, K, 1.0, 1.0, f"no-alloc unsplit {M}x{N}x{K} samples")


def test_noalloc_large_skinny_call(hk):
    """128 x 28672 x 8192 (the HBM-bound projection shape), sampled entries against the oracle."""
    M, N, K = 128, 28672, 8192
    A = synth.normal_bf16(M, K, 971, 0.02)
    B = synth.normal_bf16(N, K, 972, 0.02)
    got = _noalloc(hk, A, B, 0)
    r, c = synth.sample_positions(M, N, 973, count=2048)
    ref, _ = oracle.gemm_entries(A, B, r, c)
    assert_close(got[r, c], ref, K, 0.02, 0.02, "no-alloc skinny samples")


def test_noalloc_rejects_scratch_beyond_its_maximum(hk):
    import torch
    M, N, K = 128, 8192, 8192          # 16 splits of 128 x 8192 fp32 partials = 64 MiB > 32 MiB
    A = torch.zeros((M, K), dtype=torch.bfloat16, device="cuda")
    B = torch.zeros((N, K), dtype=torch.bfloat16, device="cuda")
    C = torch.zeros((M, N), dtype=torch.bfloat16, device="cuda")
    st = hk.hk_gemm_bf16_noalloc(A.data_ptr(), B.data_ptr(), C.data_ptr(), M, N, K, K, K, N, 16, 0)
    assert st == hk.HK_ERR_WORKSPACE
    assert "scratch" in hk.hk_gemm_last_error_string()
