"""The GEMM entry point that allocates nothing (hk_gemm_bf16_noalloc).

It exists for callers that cannot call cudaMalloc when they run a GEMM — for
example code running inside a memory pool that owns all device memory, or a
hook of an allocator that must not re-enter it. Its K-split scratch lives in
a fixed array inside the library. These tests call it through the C-ABI and
compare it with the ordinary entry point hk_gemm_bf16 on the same inputs,
within the tolerance the parity tests use, on two calls in a row (the second
call finds the first call's leftovers in the shared array).

This file is named so that pytest collects it last.
"""
from __future__ import annotations

import numpy as np
import pytest

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


def _pair(hk, A_bits, B_bits, split_k):
    """(C from hk_gemm_bf16, C from hk_gemm_bf16_noalloc) for the same inputs."""
    import torch
    M, K = A_bits.shape
    N = B_bits.shape[0]
    A, _ = to_device(A_bits)
    B, _ = to_device(B_bits)
    C_ref = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    C_new = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    stream = int(torch.cuda.current_stream().cuda_stream)
    st = hk.hk_gemm_bf16(A.data_ptr(), B.data_ptr(), C_ref.data_ptr(), M, N, K, K, K, N, stream)
    assert st == hk.HK_OK, hk.hk_gemm_last_error_string()
    st = hk.hk_gemm_bf16_noalloc(A.data_ptr(), B.data_ptr(), C_new.data_ptr(), M, N, K, K, K, N, split_k, stream)
    assert st == hk.HK_OK, hk.hk_gemm_last_error_string()
    torch.cuda.synchronize()
    return to_host(C_ref), to_host(C_new)


@pytest.mark.parametrize("split_k", [0, 4])
def test_noalloc_matches_ordinary_entry_point_twice(hk, split_k):
    M, N, K = 64, 2048, 8192
    for call in range(2):      # two calls in a row on the shared scratch, different inputs
        A = synth.normal_bf16(M, K, 700 + call)
        B = synth.normal_bf16(N, K, 800 + call)
        ref, got = _pair(hk, A, B, split_k)
        assert_close(got, ref, K, 1.0, 1.0, f"no-alloc call {call + 1}, split_k={split_k}")


def test_noalloc_integer_inputs_are_bit_exact(hk):
    M, N, K = 100, 1000, 4096
    for call in range(2):
        A = synth.int_bf16(M, K, 900 + call)
        B = synth.int_bf16(N, K, 950 + call)
        ref, got = _pair(hk, A, B, 5)
        assert_bitexact(got, ref, f"no-alloc integer call {call + 1}")


def test_noalloc_rejects_scratch_beyond_its_maximum(hk):
    import torch
    M, N, K = 128, 8192, 8192          # 16 splits of 128 x 8192 fp32 partials = 64 MiB > 32 MiB
    A = torch.zeros((M, K), dtype=torch.bfloat16, device="cuda")
    B = torch.zeros((N, K), dtype=torch.bfloat16, device="cuda")
    C = torch.zeros((M, N), dtype=torch.bfloat16, device="cuda")
    st = hk.hk_gemm_bf16_noalloc(A.data_ptr(), B.data_ptr(), C.data_ptr(), M, N, K, K, K, N, 16, 0)
    assert st == hk.HK_ERR_WORKSPACE
    assert "scratch" in hk.hk_gemm_last_error_string()
