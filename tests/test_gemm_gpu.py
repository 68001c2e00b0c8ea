"""GPU parity: the CUDA GEMM through the C-ABI against the CPU oracle.

Floating-point inputs: every checked entry within
|C_gpu - C_ref| <= 2^-7·|C_ref| + 2^-12·sqrt(K)·σ_A·σ_B.
Integer-valued inputs ({-4..4}): every partial sum is an integer below 2^24,
so fp32 accumulation is exact in any order and the results are bit-exact.
"""
from __future__ import annotations

import functools

import numpy as np
import pytest

import oracle
import synth
from gpu_util import SENTINEL, assert_bitexact, assert_close, assert_same_ieee, isnan_bf16, to_device, to_host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def hk():
    import torch
    if not torch.cuda.is_available():
        pytest.fail("no CUDA device")
    import dense_bf16_gemm_02_gb300 as pkg
    pkg.load()
    return pkg


def run_gemm(hk, A_bits, B_bits, pad=(0, 0, 0, 0), stream=None):
    """GEMM through hk_gemm_bf16 with guard bands around C; returns C bits and
    checks the guard bands are untouched."""
    import torch
    M, K = A_bits.shape
    N = B_bits.shape[0]
    a_pad, b_pad, c_rows_pad, c_cols_pad = pad
    A, Astore = to_device(A_bits, cols_pad=a_pad)
    B, Bstore = to_device(B_bits, cols_pad=b_pad)
    ldc_cols = N + ((-N) % 8) + c_cols_pad
    C, Cstore = to_device(np.full((M, N), SENTINEL, dtype=np.uint16), rows_pad=c_rows_pad,
                          cols_pad=ldc_cols - N, fill=SENTINEL)
    lda, ldb = Astore.stride(0), Bstore.stride(0)
    st = hk.hk_gemm_bf16(A.data_ptr(), B.data_ptr(), C.data_ptr(), M, N, K, lda, ldb, Cstore.stride(0),
                         int(torch.cuda.current_stream().cuda_stream) if stream is None else stream)
    assert st == hk.HK_OK, hk.hk_gemm_last_error_string()
    torch.cuda.synchronize()
    assert hk.hk_gemm_last_device_status(torch.cuda.current_device()) == hk.HK_OK
    full = to_host(Cstore)
    guard = full.copy()
    guard[:M, :N] = SENTINEL
    assert np.all(guard == SENTINEL), "a write landed outside C"
    return full[:M, :N]


def _pad_k(K):
    return (-K) % 8


# ---------------------------------------------------------- small / ragged --

RAGGED = [(1, 1, 1), (7, 9, 5), (64, 64, 64), (128, 256, 64), (200, 136, 72), (256, 256, 256),
          (257, 255, 65), (320, 264, 200), (513, 1000, 300), (1000, 520, 1032), (130, 2050, 40),
          (1, 600, 129), (600, 1, 129), (300, 300, 8)]


@pytest.mark.parametrize("M,N,K", RAGGED)
def test_ragged_integer_bitexact(hk, M, N, K):
    A = synth.int_bf16(M, K, 1100 + M)
    B = synth.int_bf16(N, K, 2100 + N)
    pad = _pad_k(K)
    got = run_gemm(hk, A, B, pad=(pad, pad + 8, 3, 8))
    assert_bitexact(got, oracle.gemm(A, B), f"int {M}x{N}x{K}")


@pytest.mark.parametrize("M,N,K", RAGGED)
def test_ragged_normal(hk, M, N, K):
    A = synth.normal_bf16(M, K, 1000 + M)
    B = synth.normal_bf16(N, K, 2000 + N)
    pad = _pad_k(K)
    got = run_gemm(hk, A, B, pad=(pad, pad, 1, 0))
    assert_close(got, oracle.gemm(A, B), K, 1.0, 1.0, f"normal {M}x{N}x{K}")


def test_gemm_256_workload(hk):
    w = synth.WORKLOADS["gemm_256"]
    A, B = synth.operands(w)
    assert_close(run_gemm(hk, A, B), oracle.gemm(A, B), w.K, w.scale, w.scale, "256^3")
    Ai, Bi = synth.operands(w, integer=True)
    assert_bitexact(run_gemm(hk, Ai, Bi), oracle.gemm(Ai, Bi), "256^3 int")


def test_k_zero_gives_zeros(hk):
    import torch
    M, N = 300, 200
    C = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    A = torch.empty((M, 8), dtype=torch.bfloat16, device="cuda")
    B = torch.empty((N, 8), dtype=torch.bfloat16, device="cuda")
    st = hk.hk_gemm_bf16(A.data_ptr(), B.data_ptr(), C.data_ptr(), M, N, 0, 8, 8, N, 0)
    assert st == hk.HK_OK
    torch.cuda.synchronize()
    assert torch.all(C == 0)


def test_empty_outputs_launch_nothing(hk):
    assert hk.hk_gemm_bf16(0, 0, 0, 0, 64, 64, 64, 64, 64, 0) == hk.HK_OK
    assert hk.hk_gemm_bf16(0, 0, 0, 64, 0, 64, 64, 64, 64, 0) == hk.HK_OK


def test_misaligned_arguments_rejected(hk):
    import torch
    A = torch.zeros((64, 72), dtype=torch.bfloat16, device="cuda")
    C = torch.zeros((64, 64), dtype=torch.bfloat16, device="cuda")
    assert hk.hk_gemm_bf16(A.data_ptr() + 2, A.data_ptr(), C.data_ptr(), 64, 64, 64, 72, 72, 64, 0) == \
        hk.HK_ERR_MISALIGNED
    assert hk.hk_gemm_bf16(A.data_ptr(), A.data_ptr(), C.data_ptr(), 64, 64, 64, 68, 72, 64, 0) == \
        hk.HK_ERR_MISALIGNED


def test_deterministic(hk):
    A = synth.normal_bf16(1024, 2048, 5)
    B = synth.normal_bf16(768, 2048, 6)
    a = run_gemm(hk, A, B)
    b = run_gemm(hk, A, B)
    assert np.array_equal(a, b)


def test_torch_binding_and_plan(hk):
    import torch
    A = synth.normal_bf16(700, 520, 15)
    B = synth.normal_bf16(900, 520, 16)
    ref = oracle.gemm(A, B)
    At, _ = to_device(A)
    Bt, _ = to_device(B)
    assert_close(to_host(hk.gemm(At, Bt)), ref, 520, 1, 1, "gemm()")
    for group_m, max_clusters in [(1, 1), (3, 2), (8, 0), (100, 5)]:
        plan = hk.Plan(700, 900, 520, ldc=904, group_m=group_m, max_clusters=max_clusters)
        info = plan.info()
        assert info["kernels_per_run"] == 1 and plan.workspace_size == 0
        C = torch.empty((700, 904), dtype=torch.bfloat16, device="cuda")[:, :900]
        plan.run(At, Bt, C)
        torch.cuda.synchronize()
        assert plan.device_status() == hk.HK_OK
        assert_close(to_host(C), ref, 520, 1, 1, f"plan group_m={group_m} clusters={max_clusters}")
        plan.close()


def test_stream_argument(hk):
    import torch
    A = synth.int_bf16(384, 256, 1)
    B = synth.int_bf16(512, 256, 2)
    s = torch.cuda.Stream()
    At, _ = to_device(A)
    Bt, _ = to_device(B)
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        C = hk.gemm(At, Bt)
    s.synchronize()
    assert_bitexact(to_host(C), oracle.gemm(A, B), "side stream")


# (label, M, N, K, plan options, expected kernel id, expected stages or 0, expected K splits)
TIMEOUT_CASES = [
    ("pair bf16", 512, 512, 512, {"kernel": 1}, 1, 0, 1),
    ("single 128x256, 16-row A stages", 1, 512, 512, {"kernel": 2}, 2, 6, 1),
    ("single 128x256, 64-row A stages", 40, 512, 512, {"kernel": 2}, 2, 5, 1),
    ("single 128x64", 100, 512, 512, {"kernel": 5}, 5, 0, 1),
    ("single 128x256, split K", 64, 1024, 2048, {"kernel": 2, "split_k": 4}, 2, 0, 4),
    ("pair bf16, split K", 512, 512, 2048, {"kernel": 1, "split_k": 2}, 1, 0, 2),
    ("pair 256x128", 256, 640, 512, {"kernel": 6}, 6, 8, 1),
    ("pair 256x112", 256, 640, 512, {"kernel": 7}, 7, 9, 1),
    ("fp8 pair", 512, 512, 512, {"input_type": 1}, 1, 0, 1),
    ("fp8 single 128x192", 128, 600, 512, {"input_type": 1, "kernel": 3}, 3, 0, 1),
]


@pytest.mark.parametrize("case", TIMEOUT_CASES, ids=[c[0] for c in TIMEOUT_CASES])
def test_bounded_wait_reports_timeout_and_recovers(hk, case):
    """Fault injected on the host side of the protocol: the producer withholds
    one arrival, a bounded wait runs out, every role of the kernel drains and
    returns (pair and single-CTA kernels, short-A stages, split K with its
    dependent reduction, E4M3), the status word reports HK_ERR_TIMEOUT, and
    the context stays usable: the same plan without the fault is then exact."""
    import torch
    label, M, N, K, opts, kernel, stages, splits = case
    fp8 = opts.get("input_type", 0) == hk.HK_INPUT_E4M3
    if fp8:
        A, B = synth.int_e4m3(M, K, 3 + M), synth.int_e4m3(N, K, 4 + N)
        At, Bt = torch.from_numpy(A).to("cuda"), torch.from_numpy(B).to("cuda")
        want = oracle.gemm_fp8(A, B, 1.0, 1.0)
    else:
        A, B = synth.int_bf16(M, K, 3 + M), synth.int_bf16(N, K, 4 + N)
        At, _ = to_device(A)
        Bt, _ = to_device(B)
        want = oracle.gemm(A, B)
    C = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    plan = hk.Plan(M, N, K, timeout_ns=20_000_000, flags=hk.HK_FLAG_FAULT_DROP_ARRIVE, **opts)
    info = plan.info()
    assert info["kernel"] == kernel and info["split_k"] == splits, (label, info)
    if stages:
        assert info["stages"] == stages, (label, info)
    plan.run(At, Bt, C)
    torch.cuda.synchronize()
    assert plan.device_status() == hk.HK_ERR_TIMEOUT, label
    assert plan.device_status() == hk.HK_OK, label       # read-and-clear
    plan.close()
    good = hk.Plan(M, N, K, **opts)
    C.zero_()
    good.run(At, Bt, C)
    torch.cuda.synchronize()
    assert good.device_status() == hk.HK_OK, label
    good.close()
    assert_bitexact(to_host(C), want, f"{label}: after timeout")


# ------------------------------------------------------- full workloads --

@functools.lru_cache(maxsize=1)
def _operands(name, integer=False):
    return synth.operands(synth.WORKLOADS[name], integer=integer)


def _check_workload(hk, name, integer=False, via_plan=False):
    import torch
    w = synth.WORKLOADS[name]
    A, B = _operands(name, integer)
    At, _ = to_device(A)
    Bt, _ = to_device(B)
    if via_plan:   # a plan may split K (workspace allocated by Plan.run), as bench.py runs decode shapes
        plan = hk.Plan(w.M, w.N, w.K)
        C = plan.run(At, Bt, torch.empty((w.M, w.N), dtype=torch.bfloat16, device=At.device))
    else:
        C = hk.gemm(At, Bt)
    torch.cuda.synchronize()
    assert hk.hk_gemm_last_device_status(torch.cuda.current_device()) == hk.HK_OK
    got = to_host(C)
    del At, Bt, C
    check = assert_bitexact if integer else (
        lambda g, r, what: assert_close(g, r, w.K, w.scale, w.scale, what))
    if not w.sampled:
        check(got, oracle.gemm(A, B), name)
        return
    r, c = synth.sample_positions(w.M, w.N, 3000 + w.wid)
    ref, _ = oracle.gemm_entries(A, B, r, c)
    check(got[r, c], ref, name + " samples")
    rows = synth.full_rows(w.M, 3000 + w.wid)
    ref_rows, _ = oracle.gemm_rows(A, B, rows)
    check(got[rows], ref_rows, name + " rows")


def test_workload_4096(hk):
    _check_workload(hk, "gemm_4096")


def test_workload_8192(hk):
    _check_workload(hk, "gemm_8192")


def test_workload_8192_integer(hk):
    _check_workload(hk, "gemm_8192", integer=True)


def test_workload_16384(hk):
    _check_workload(hk, "gemm_16384")


def test_workload_projection(hk):
    _check_workload(hk, "proj_16384x28672x8192")


def test_workload_skinny(hk):
    _check_workload(hk, "skinny_128x28672x8192")


def test_workload_decode_one_token(hk):
    _check_workload(hk, "decode_1x28672x8192", via_plan=True)


def test_workload_decode_batch_64(hk):
    _check_workload(hk, "decode_64x8192x28672", via_plan=True)


def test_workload_decode_batch_256(hk):
    _check_workload(hk, "decode_256x8192x8192", via_plan=True)


# ------------------------------------------------------ kernel variants --

VARIANT_SHAPES = [(1, 1, 1), (100, 300, 70), (128, 1000, 520), (257, 130, 64), (700, 452, 1000)]


def run_plan(hk, A_bits, B_bits, **cfg):
    import torch
    cfg.setdefault("split_k", 1)
    M, K = A_bits.shape
    N = B_bits.shape[0]
    kp = (-K) % 8
    A, Astore = to_device(A_bits, cols_pad=kp)
    B, Bstore = to_device(B_bits, cols_pad=kp + 8)
    ldc = N + ((-N) % 8) + 8
    C, Cstore = to_device(np.full((M, N), SENTINEL, dtype=np.uint16), rows_pad=2, cols_pad=ldc - N,
                          fill=SENTINEL)
    plan = hk.Plan(M, N, K, lda=Astore.stride(0), ldb=Bstore.stride(0), ldc=Cstore.stride(0), **cfg)
    info = plan.info()
    st = plan.run_raw(A.data_ptr(), B.data_ptr(), C.data_ptr(), 0, 0,
                      int(torch.cuda.current_stream().cuda_stream))
    assert st == hk.HK_OK, hk.hk_gemm_last_error_string()
    torch.cuda.synchronize()
    assert plan.device_status() == hk.HK_OK
    plan.close()
    full = to_host(Cstore)
    guard = full.copy()
    guard[:M, :N] = SENTINEL
    assert np.all(guard == SENTINEL), "a write landed outside C"
    return full[:M, :N], info


@pytest.mark.parametrize("kernel", [1, 2, 3, 4, 5, 6, 7])
@pytest.mark.parametrize("M,N,K", VARIANT_SHAPES)
def test_kernel_variants_integer_bitexact(hk, kernel, M, N, K):
    A = synth.int_bf16(M, K, 1200 + M)
    B = synth.int_bf16(N, K, 2200 + N)
    got, info = run_plan(hk, A, B, kernel=kernel, max_clusters=3)
    assert info["kernel"] == kernel
    assert_bitexact(got, oracle.gemm(A, B), f"kernel {kernel} int {M}x{N}x{K}")


@pytest.mark.parametrize("kernel", [2, 3, 4, 5, 6, 7])
def test_kernel_variants_normal(hk, kernel):
    M, N, K = 200, 777, 1500
    A = synth.normal_bf16(M, K, 31)
    B = synth.normal_bf16(N, K, 32)
    got, info = run_plan(hk, A, B, kernel=kernel)
    assert_close(got, oracle.gemm(A, B), K, 1, 1, f"kernel {kernel}")


def test_automatic_kernel_choice(hk):
    assert hk.Plan(128, 28672, 8192).info()["kernel"] == 3      # 150 tiles of 128x192 ~ one per SM
    assert hk.Plan(8192, 8192, 8192).info()["kernel"] == 1
    assert hk.Plan(385, 4096, 4096).info()["ctas_per_unit"] == 2  # above 384 rows: CTA pairs
    assert hk.Plan(129, 4096, 4096).info()["ctas_per_unit"] == 1  # a 129-row pair tile would be half empty
    assert hk.Plan(256, 8192, 8192).info()["kernel"] == 7       # 74 pairs of 256x112 (9 stages): one wave, no K split
    assert hk.Plan(384, 8192, 8192).info()["kernel"] == 3       # 3 x 43 tiles of 128x192 (measured best)
    assert hk.Plan(200, 4096, 4096, input_type=hk.HK_INPUT_E4M3).info()["kernel"] == 1   # E4M3: pairs above 128
    small = hk.Plan(64, 1024, 1024).info()
    assert small["kernel"] == 5 and small["ctas_per_unit"] == 1  # 16 tiles: narrowest tiles spread widest


# ----------------------------------------------------------------- split K --

def run_split(hk, A_bits, B_bits, ws_fill=0, runs=1, **cfg):
    """Plan with (possibly forced) K splits, run `runs` times on one workspace."""
    import torch
    M, K = A_bits.shape
    N = B_bits.shape[0]
    kp = (-K) % 8
    A, Astore = to_device(A_bits, cols_pad=kp)
    B, Bstore = to_device(B_bits, cols_pad=kp)
    ldc = N + ((-N) % 8)
    plan = hk.Plan(M, N, K, lda=Astore.stride(0), ldb=Bstore.stride(0), ldc=ldc, **cfg)
    info = plan.info()
    ws_bytes = plan.workspace_size
    ws = torch.full((max(ws_bytes, 1) + 255,), ws_fill, dtype=torch.uint8, device="cuda")
    ws_ptr = (ws.data_ptr() + 255) & ~255
    outs = []
    for _ in range(runs):
        C, Cstore = to_device(np.full((M, N), SENTINEL, dtype=np.uint16), rows_pad=2, cols_pad=ldc - N,
                              fill=SENTINEL)
        st = plan.run_raw(A.data_ptr(), B.data_ptr(), C.data_ptr(), ws_ptr, ws_bytes,
                          int(torch.cuda.current_stream().cuda_stream))
        assert st == hk.HK_OK, hk.hk_gemm_last_error_string()
        torch.cuda.synchronize()
        assert plan.device_status() == hk.HK_OK
        full = to_host(Cstore)
        guard = full.copy()
        guard[:M, :N] = SENTINEL
        assert np.all(guard == SENTINEL), "a write landed outside C"
        outs.append(full[:M, :N])
    plan.close()
    return outs, info


@pytest.mark.parametrize("kernel,splits,M,N,K", [
    (1, 2, 300, 200, 1000), (1, 5, 257, 520, 2049), (6, 3, 200, 700, 1000), (2, 3, 100, 700, 900), (3, 7, 64, 1000, 2000),
    (4, 16, 128, 300, 1030), (5, 4, 1, 77, 640), (3, 2, 200, 600, 128), (7, 3, 200, 1000, 1000),
    (7, 2, 260, 1120, 520)])
def test_split_k_integer_bitexact(hk, kernel, splits, M, N, K):
    A = synth.int_bf16(M, K, 1300 + M)
    B = synth.int_bf16(N, K, 2300 + N)
    (got,), info = run_split(hk, A, B, kernel=kernel, split_k=splits)
    assert info["split_k"] == splits and info["workspace_bytes"] > 0
    assert_bitexact(got, oracle.gemm(A, B), f"kernel {kernel} split {splits} {M}x{N}x{K}")


def test_split_k_normal_and_deterministic(hk):
    M, N, K = 96, 2000, 4096
    A = synth.normal_bf16(M, K, 41)
    B = synth.normal_bf16(N, K, 42)
    outs, info = run_split(hk, A, B, ws_fill=0xFF, runs=3, kernel=3, split_k=6)
    assert_close(outs[0], oracle.gemm(A, B), K, 1, 1, "split 6")
    assert np.array_equal(outs[0], outs[1]) and np.array_equal(outs[1], outs[2])


def test_split_k_automatic_for_small_m(hk):
    """64 x 2048 x 8192: 16-32 output tiles for 152 SMs, so the plan splits K."""
    A = synth.normal_bf16(64, 8192, 43)
    B = synth.normal_bf16(2048, 8192, 44)
    outs, info = run_split(hk, A, B)
    assert info["split_k"] > 1 and info["ctas_per_unit"] == 1
    r, c = synth.sample_positions(64, 2048, 45, count=2048)
    ref, _ = oracle.gemm_entries(A, B, r, c)
    assert_close(outs[0][r, c], ref, 8192, 1, 1, "auto split")
    assert hk.Plan(8192, 8192, 8192).info()["split_k"] == 1          # full waves: never split


def test_split_k_workspace_errors(hk):
    import torch
    plan = hk.Plan(64, 1024, 4096, split_k=4, kernel=4)
    need = plan.workspace_size
    assert need > 0
    A = torch.zeros((64, 4096), dtype=torch.bfloat16, device="cuda")
    B = torch.zeros((1024, 4096), dtype=torch.bfloat16, device="cuda")
    C = torch.zeros((64, 1024), dtype=torch.bfloat16, device="cuda")
    ws = torch.zeros(need + 512, dtype=torch.uint8, device="cuda")
    base = (ws.data_ptr() + 255) & ~255
    assert plan.run_raw(A.data_ptr(), B.data_ptr(), C.data_ptr(), 0, 0, 0) == hk.HK_ERR_WORKSPACE
    assert plan.run_raw(A.data_ptr(), B.data_ptr(), C.data_ptr(), base, need - 1, 0) == hk.HK_ERR_WORKSPACE
    assert plan.run_raw(A.data_ptr(), B.data_ptr(), C.data_ptr(), base + 16, need, 0) == hk.HK_ERR_WORKSPACE
    assert plan.run_raw(A.data_ptr(), B.data_ptr(), C.data_ptr(), base, need, 0) == hk.HK_OK
    torch.cuda.synchronize()
    assert plan.device_status() == hk.HK_OK
    plan.close()


# ---------------------------------------------------- tail round split --

@pytest.mark.parametrize("M,N,K", [(4096, 4096, 512), (256, 1024, 640), (512, 1000, 320), (2900, 700, 200),
                                   (8192, 8192, 128)])
def test_tail_split_integer_bitexact(hk, M, N, K):
    """Tiles of the last partial round run as two 256x128 halves."""
    A = synth.int_bf16(M, K, 1400 + M)
    B = synth.int_bf16(N, K, 2400 + N)
    got, info = run_plan(hk, A, B, kernel=1)
    assert info["kernel"] == 1 and info["tail_split_tiles"] > 0
    if M * N <= 4096 * 4096:
        assert_bitexact(got, oracle.gemm(A, B), f"tail split {M}x{N}x{K}")
    else:
        r, c = synth.sample_positions(M, N, 77, count=4096)
        ref, _ = oracle.gemm_entries(A, B, r, c)
        assert_bitexact(got[r, c], ref, f"tail split {M}x{N}x{K} samples")
    whole, info2 = run_plan(hk, A, B, kernel=1, flags=hk.HK_FLAG_NO_TAIL_SPLIT)
    assert info2["tail_split_tiles"] == 0
    assert_bitexact(got, whole, "split vs whole")


@pytest.mark.parametrize("M,N,K", [(256, 1024, 640), (600, 1000, 320), (130, 4100, 136)])
def test_tail_split_narrow_pair_integer_bitexact(hk, M, N, K):
    """The 256x128 pair's last partial round runs as 256x64 halves."""
    A = synth.int_bf16(M, K, 1450 + M)
    B = synth.int_bf16(N, K, 2450 + N)
    got, info = run_plan(hk, A, B, kernel=6)
    assert info["kernel"] == 6 and info["tile_n"] == 128 and info["tail_split_tiles"] > 0
    assert_bitexact(got, oracle.gemm(A, B), f"narrow pair tail split {M}x{N}x{K}")
    whole, info2 = run_plan(hk, A, B, kernel=6, flags=hk.HK_FLAG_NO_TAIL_SPLIT)
    assert info2["tail_split_tiles"] == 0
    assert_bitexact(got, whole, "split vs whole")


@pytest.mark.parametrize("M,N,K", [(256, 8192, 256), (300, 1000, 264), (200, 112, 64), (257, 230, 136),
                                   (512, 2240, 72)])
def test_pair_256x112_integer_bitexact(hk, M, N, K):
    """The 112-wide pair: a tile's last 16 columns go out by plain stores (all
    inside N, partly past it at N = 1000 and 230, or wholly past it), and a
    partial last round keeps whole tiles (no half-width units: N / 2 = 56 is no
    MMA width). N = 8192 is 74 tiles; 512 x 2240 is 40 tiles, whose last
    round on 12 pairs holds 4 (a half-splitting pair would split it)."""
    A = synth.int_bf16(M, K, 1470 + M)
    B = synth.int_bf16(N, K, 2470 + N)
    got, info = run_plan(hk, A, B, kernel=7)
    assert info["kernel"] == 7 and info["tile_n"] == 112 and info["tail_split_tiles"] == 0
    assert info["num_tiles"] == -(-M // 256) * -(-N // 112)
    assert_bitexact(got, oracle.gemm(A, B), f"pair 256x112 {M}x{N}x{K}")
    if N == 2240:
        few, info2 = run_plan(hk, A, B, kernel=7, max_clusters=12)
        assert info2["tail_split_tiles"] == 0
        assert_bitexact(few, got, "12 pairs vs all")


@pytest.mark.parametrize("M,N,K", [(257, 600, 128), (300, 1000, 264)])
def test_fused_epilogue_pair_256x112_integer_bitexact(hk, M, N, K):
    """Bias and ReLU, then a residual after the activation, on the 112-wide
    pair (the narrow last chunk of every tile included)."""
    A = synth.int_bf16(M, K, 1960 + M)
    B = synth.int_bf16(N, K, 2960 + N)
    bias = synth.int_bf16(1, N, 3960 + N)[0]
    R = synth.int_bf16(M, N, 4960 + N, -40, 40)
    got = run_epilogue(hk, A, B, bias, 1, split_k=1, kernel=7)
    assert_bitexact(got, oracle.gemm_epilogue(A, B, bias, 1), f"pair 112 relu + bias {M}x{N}x{K}")
    got = run_fused(hk, A, B, bias, R, 1, split_k=1, kernel=7)
    assert_bitexact(got, oracle.gemm_epilogue(A, B, bias, 1, residual=R), f"pair 112 residual {M}x{N}x{K}")


def test_tail_split_normal_matches_whole_tiles(hk):
    M, N, K = 1024, 2000, 1000          # 4 x 8 = 32 tiles: all run as halves
    A = synth.normal_bf16(M, K, 61)
    B = synth.normal_bf16(N, K, 62)
    got, info = run_plan(hk, A, B, kernel=1)
    assert info["tail_split_tiles"] > 0
    assert_close(got, oracle.gemm(A, B), K, 1, 1, "tail split normal")
    whole, _ = run_plan(hk, A, B, kernel=1, flags=2)
    assert_close(got, whole, K, 1, 1, "split vs whole")


# --------------------------------------------------------- fused epilogue --

def run_epilogue(hk, A_bits, B_bits, bias_bits, act, split_k=None, kernel=0):
    import torch
    M, K = A_bits.shape
    N = B_bits.shape[0]
    kp = (-K) % 8
    A, Astore = to_device(A_bits, cols_pad=kp)
    B, Bstore = to_device(B_bits, cols_pad=kp)
    ldc = N + ((-N) % 8)
    C, Cstore = to_device(np.full((M, N), SENTINEL, dtype=np.uint16), rows_pad=1, cols_pad=ldc - N,
                          fill=SENTINEL)
    bias_t = None
    if bias_bits is not None:
        bias_t = torch.from_numpy(np.ascontiguousarray(bias_bits).view(np.int16)).to("cuda")
    bptr = bias_t.data_ptr() if bias_t is not None else 0
    stream = int(torch.cuda.current_stream().cuda_stream)
    if split_k is None:
        st = hk.hk_gemm_bf16_epilogue(A.data_ptr(), B.data_ptr(), C.data_ptr(), bptr, M, N, K, Astore.stride(0),
                                      Bstore.stride(0), Cstore.stride(0), act, stream)
    else:
        plan = hk.Plan(M, N, K, lda=Astore.stride(0), ldb=Bstore.stride(0), ldc=Cstore.stride(0),
                       split_k=split_k, kernel=kernel, activation=act)
        ws = torch.zeros(max(plan.workspace_size, 1) + 256, dtype=torch.uint8, device="cuda")
        st = plan.run_epilogue_raw(A.data_ptr(), B.data_ptr(), C.data_ptr(), bptr, (ws.data_ptr() + 255) & ~255,
                                   plan.workspace_size, stream)
    assert st == hk.HK_OK, hk.hk_gemm_last_error_string()
    torch.cuda.synchronize()
    full = to_host(Cstore)
    guard = full.copy()
    guard[:M, :N] = SENTINEL
    assert np.all(guard == SENTINEL), "a write landed outside C"
    return full[:M, :N]


@pytest.mark.parametrize("act", [0, 1, 2, 3])
@pytest.mark.parametrize("with_bias", [False, True])
@pytest.mark.parametrize("M,N,K", [(300, 517, 200), (64, 1000, 640), (1024, 768, 1536)])
def test_epilogue_normal(hk, act, with_bias, M, N, K):
    A = synth.normal_bf16(M, K, 1500 + M)
    B = synth.normal_bf16(N, K, 2500 + N)
    bias = synth.normal_bf16(1, N, 3500 + N, 4.0)[0] if with_bias else None
    got = run_epilogue(hk, A, B, bias, act)
    ref = oracle.gemm_epilogue(A, B, bias, act)
    assert_close(got, ref, K, 1, 1, f"act {act} bias {with_bias} {M}x{N}x{K}")


@pytest.mark.parametrize("M,N,K", [(257, 300, 128), (128, 2050, 96)])
def test_epilogue_relu_integer_bitexact(hk, M, N, K):
    A = synth.int_bf16(M, K, 1600 + M)
    B = synth.int_bf16(N, K, 2600 + N)
    bias = synth.int_bf16(1, N, 3600 + N)[0]
    got = run_epilogue(hk, A, B, bias, 1)
    assert_bitexact(got, oracle.gemm_epilogue(A, B, bias, 1), "relu + bias integer")


@pytest.mark.parametrize("act", [1, 2, 3])
def test_epilogue_in_split_k_reduction(hk, act):
    M, N, K = 64, 1200, 4096
    A = synth.normal_bf16(M, K, 71)
    B = synth.normal_bf16(N, K, 72)
    bias = synth.normal_bf16(1, N, 73, 2.0)[0]
    got = run_epilogue(hk, A, B, bias, act, split_k=4, kernel=4)
    assert_close(got, oracle.gemm_epilogue(A, B, bias, act), K, 1, 1, f"split-K act {act}")


def test_epilogue_argument_errors(hk):
    import torch
    A = torch.zeros((64, 64), dtype=torch.bfloat16, device="cuda")
    C = torch.zeros((64, 64), dtype=torch.bfloat16, device="cuda")
    bias = torch.zeros(80, dtype=torch.bfloat16, device="cuda")
    assert hk.hk_gemm_bf16_epilogue(A.data_ptr(), A.data_ptr(), C.data_ptr(), bias.data_ptr() + 2, 64, 64, 64,
                                    64, 64, 64, 1, 0) == hk.HK_ERR_MISALIGNED
    assert hk.hk_gemm_bf16_epilogue(A.data_ptr(), A.data_ptr(), C.data_ptr(), bias.data_ptr(), 64, 64, 64,
                                    64, 64, 64, 7, 0) == hk.HK_ERR_INVALID_ARG


# ------------------------------------------------------- plan caches --

def test_one_shot_cache_with_changing_pointers_and_many_shapes(hk):
    """The one-shot call caches plans (32 shapes, least recently used) and each
    plan the tensor maps of its last pointers: calls that alternate buffers of
    one shape, and more shapes than the cache holds (evictions), stay exact."""
    import torch
    M, N, K = 300, 520, 136
    bufs = []
    for i in range(3):
        A, B = synth.int_bf16(M, K, 5100 + i), synth.int_bf16(N, K, 5200 + i)
        bufs.append((A, B, to_device(A)[0], to_device(B)[0]))
    Cs = [torch.empty((M, N), dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    stream = int(torch.cuda.current_stream().cuda_stream)
    for it in range(6):
        A, B, At, Bt = bufs[it % 3]
        C = Cs[it % 2]
        assert hk.hk_gemm_bf16(At.data_ptr(), Bt.data_ptr(), C.data_ptr(), M, N, K, K, K, N, stream) == hk.HK_OK
        torch.cuda.synchronize()
        assert_bitexact(to_host(C), oracle.gemm(A, B), f"alternating buffers, call {it}")
    for i in range(40):                      # 40 distinct shapes: the cache evicts
        m, n, k = 16 + 8 * i, 40 + 8 * (i % 7), 24 + 8 * (i % 5)
        A, B = synth.int_bf16(m, k, 5300 + i), synth.int_bf16(n, k, 5400 + i)
        At, _ = to_device(A)
        Bt, _ = to_device(B)
        C = torch.empty((m, n), dtype=torch.bfloat16, device="cuda")
        assert hk.hk_gemm_bf16(At.data_ptr(), Bt.data_ptr(), C.data_ptr(), m, n, k, k, k, n, stream) == hk.HK_OK
        torch.cuda.synchronize()
        assert_bitexact(to_host(C), oracle.gemm(A, B), f"shape {m}x{n}x{k}")
    assert hk.hk_gemm_last_device_status(torch.cuda.current_device()) == hk.HK_OK


def test_plan_run_with_changing_pointers(hk):
    import torch
    M, N, K = 260, 300, 200
    plan = hk.Plan(M, N, K, lda=K + 8, ldb=K + 8, ldc=N + 4)
    for it in range(4):
        A, B = synth.int_bf16(M, K, 5500 + it), synth.int_bf16(N, K, 5600 + it)
        At, _ = to_device(A, cols_pad=8)
        Bt, _ = to_device(B, cols_pad=8)
        C, Cstore = to_device(np.zeros((M, N), dtype=np.uint16), cols_pad=4)
        st = plan.run_raw(At.data_ptr(), Bt.data_ptr(), C.data_ptr(), 0, 0, int(torch.cuda.current_stream().cuda_stream))
        assert st == hk.HK_OK, hk.hk_gemm_last_error_string()
        torch.cuda.synchronize()
        assert_bitexact(to_host(Cstore)[:M, :N], oracle.gemm(A, B), f"plan run {it}")
    assert plan.device_status() == hk.HK_OK
    plan.close()


# ------------------------------------- programmatic dependent launches --

def test_dependent_chain_on_one_stream(hk):
    """Every GEMM is launched as a programmatic dependent of the kernel before it:
    its prologue may overlap that kernel, but its loads of A/B and its stores of C
    must wait for it. A chain on one stream with no host synchronisation: each
    GEMM reads the previous one's C (read after write), and the last one writes
    over the first one's A (write after read); pair and single-CTA kernels, and a
    K split whose reduction is itself a dependent launch. Integer data: exact."""
    import torch
    stream = int(torch.cuda.current_stream().cuda_stream)
    M, K = 512, 256
    A0 = synth.int_bf16(M, K, 5701, -1, 1)   # every partial sum of the chain stays an integer below 2^24
    Bs = [synth.int_bf16(K, K, 5710 + i, -1, 1) for i in range(3)]
    A0d, _ = to_device(A0)
    Bd = [to_device(b)[0] for b in Bs]
    C1 = torch.empty((M, K), dtype=torch.bfloat16, device="cuda")
    C2 = torch.empty((64, K), dtype=torch.bfloat16, device="cuda")
    # C1 = A0·B0ᵀ (pair kernel); C2 = C1[:64]·B1ᵀ (single-CTA, K split through a plan);
    # A0[:64] = C2·B2ᵀ (overwrites rows of A0, which the first GEMM read)
    assert hk.hk_gemm_bf16(A0d.data_ptr(), Bd[0].data_ptr(), C1.data_ptr(), M, K, K, K, K, K, stream) == hk.HK_OK
    plan = hk.Plan(64, K, K, split_k=2, kernel=4)
    ws = torch.empty(plan.workspace_size + 256, dtype=torch.uint8, device="cuda")
    assert plan.run_raw(C1.data_ptr(), Bd[1].data_ptr(), C2.data_ptr(), (ws.data_ptr() + 255) & ~255,
                        plan.workspace_size, stream) == hk.HK_OK
    assert hk.hk_gemm_bf16(C2.data_ptr(), Bd[2].data_ptr(), A0d.data_ptr(), 64, K, K, K, K, K, stream) == hk.HK_OK
    torch.cuda.synchronize()
    assert hk.hk_gemm_last_device_status(torch.cuda.current_device()) == hk.HK_OK
    c1 = oracle.gemm(A0, Bs[0])
    c2 = oracle.gemm(np.ascontiguousarray(c1[:64]), Bs[1])
    a_new = oracle.gemm(c2, Bs[2])
    assert_bitexact(to_host(C1), c1, "first GEMM")
    assert_bitexact(to_host(C2), c2, "second GEMM (reads the first's C)")
    got_a = to_host(A0d)
    assert_bitexact(got_a[:64], a_new, "third GEMM (writes the first's A)")
    assert_bitexact(got_a[64:], A0[64:], "rows of A the chain does not write")
    plan.close()


# ------------------------------------------------- fused residual add --

def run_fused(hk, A_bits, B_bits, bias_bits, R_bits, act, split_k=None, kernel=0, in_place=False, ldr_pad=0):
    """C = bf16(act(A·Bᵀ + bias) + R) through hk_gemm_bf16_fused (or a plan with a
    forced kernel and K split); R in its own padded storage, or C itself."""
    import torch
    M, K = A_bits.shape
    N = B_bits.shape[0]
    kp = (-K) % 8
    A, Astore = to_device(A_bits, cols_pad=kp)
    B, Bstore = to_device(B_bits, cols_pad=kp)
    ldc = N + ((-N) % 8)
    if in_place:
        C, Cstore = to_device(R_bits, rows_pad=1, cols_pad=ldc - N, fill=SENTINEL)
        Rptr, ldr = C.data_ptr(), Cstore.stride(0)
    else:
        C, Cstore = to_device(np.full((M, N), SENTINEL, dtype=np.uint16), rows_pad=1, cols_pad=ldc - N,
                              fill=SENTINEL)
        ldr_cols = N + ((-N) % 8) + ldr_pad
        Rt, Rstore = to_device(R_bits, cols_pad=ldr_cols - N, fill=SENTINEL)
        Rptr, ldr = Rt.data_ptr(), Rstore.stride(0)
    bias_t = None
    if bias_bits is not None:
        bias_t = torch.from_numpy(np.ascontiguousarray(bias_bits).view(np.int16)).to("cuda")
    bptr = bias_t.data_ptr() if bias_t is not None else 0
    stream = int(torch.cuda.current_stream().cuda_stream)
    if split_k is None:
        st = hk.hk_gemm_bf16_fused(A.data_ptr(), B.data_ptr(), C.data_ptr(), bptr, Rptr, M, N, K, Astore.stride(0),
                                   Bstore.stride(0), Cstore.stride(0), ldr, act, stream)
    else:
        plan = hk.Plan(M, N, K, lda=Astore.stride(0), ldb=Bstore.stride(0), ldc=Cstore.stride(0),
                       split_k=split_k, kernel=kernel, activation=act)
        assert plan.info()["split_k"] == split_k
        ws = torch.zeros(max(plan.workspace_size, 1) + 256, dtype=torch.uint8, device="cuda")
        st = plan.run_fused_raw(A.data_ptr(), B.data_ptr(), C.data_ptr(), bptr, Rptr, ldr,
                                (ws.data_ptr() + 255) & ~255, plan.workspace_size, stream)
    assert st == hk.HK_OK, hk.hk_gemm_last_error_string()
    torch.cuda.synchronize()
    assert hk.hk_gemm_last_device_status(torch.cuda.current_device()) == hk.HK_OK
    full = to_host(Cstore)
    guard = full.copy()
    guard[:M, :N] = SENTINEL
    assert np.all(guard == SENTINEL), "a write landed outside C"
    return full[:M, :N]


@pytest.mark.parametrize("act,with_bias", [(0, False), (0, True), (2, True), (3, False)])
@pytest.mark.parametrize("M,N,K", [(300, 517, 200), (64, 1000, 640), (1024, 768, 1536), (7, 333, 96)])
def test_residual_normal(hk, act, with_bias, M, N, K):
    A = synth.normal_bf16(M, K, 1700 + M)
    B = synth.normal_bf16(N, K, 2700 + N)
    bias = synth.normal_bf16(1, N, 3700 + N, 2.0)[0] if with_bias else None
    R = synth.normal_bf16(M, N, 4700 + M + N, 4.0)
    got = run_fused(hk, A, B, bias, R, act)
    ref = oracle.gemm_epilogue(A, B, bias, act, residual=R)
    assert_close(got, ref, K, 1, 1, f"residual act {act} bias {with_bias} {M}x{N}x{K}")


@pytest.mark.parametrize("M,N,K", [(257, 300, 128), (128, 2050, 96), (520, 1030, 264)])
def test_residual_relu_integer_bitexact(hk, M, N, K):
    """Integer data: every fp32 step is exact, so act(dot + bias) + R matches bit for bit."""
    A = synth.int_bf16(M, K, 1800 + M)
    B = synth.int_bf16(N, K, 2800 + N)
    bias = synth.int_bf16(1, N, 3800 + N)[0]
    R = synth.int_bf16(M, N, 4800 + N, -60, 60)
    got = run_fused(hk, A, B, bias, R, 1)
    assert_bitexact(got, oracle.gemm_epilogue(A, B, bias, 1, residual=R), "relu + bias + residual integer")


@pytest.mark.parametrize("M,N,K", [(300, 517, 200), (130, 264, 72)])
def test_residual_in_place(hk, M, N, K):
    """R = C (same pointer and leading dimension): C ← act(A·Bᵀ + bias) + C."""
    A = synth.int_bf16(M, K, 1900 + M)
    B = synth.int_bf16(N, K, 2900 + N)
    bias = synth.int_bf16(1, N, 3900 + N)[0]
    R = synth.int_bf16(M, N, 4900 + N, -30, 30)
    got = run_fused(hk, A, B, bias, R, 0, in_place=True)
    assert_bitexact(got, oracle.gemm_epilogue(A, B, bias, 0, residual=R), "in-place residual")


def test_residual_padded_leading_dimension(hk):
    M, N, K = 200, 120, 64
    A, B = synth.int_bf16(M, K, 61), synth.int_bf16(N, K, 62)
    R = synth.int_bf16(M, N, 63, -9, 9)
    got = run_fused(hk, A, B, None, R, 0, ldr_pad=40)
    assert_bitexact(got, oracle.gemm_epilogue(A, B, None, 0, residual=R), "ldr > N")


@pytest.mark.parametrize("M,N,K", [(257, 600, 128), (520, 1030, 264)])
def test_fused_epilogue_narrow_pair_integer_bitexact(hk, M, N, K):
    """The 256x128 pair kernel, its 256x64 tail halves included (10 and 27
    tiles: every tile runs as two halves), with bias and ReLU, then with a
    residual added after the activation."""
    A = synth.int_bf16(M, K, 1950 + M)
    B = synth.int_bf16(N, K, 2950 + N)
    bias = synth.int_bf16(1, N, 3950 + N)[0]
    R = synth.int_bf16(M, N, 4950 + N, -40, 40)
    got = run_epilogue(hk, A, B, bias, 1, split_k=1, kernel=6)
    assert_bitexact(got, oracle.gemm_epilogue(A, B, bias, 1), f"narrow pair relu + bias {M}x{N}x{K}")
    got = run_fused(hk, A, B, bias, R, 1, split_k=1, kernel=6)
    assert_bitexact(got, oracle.gemm_epilogue(A, B, bias, 1, residual=R), f"narrow pair residual {M}x{N}x{K}")


@pytest.mark.parametrize("kernel,splits", [(4, 4), (1, 3), (2, 2), (6, 3), (7, 2)])
def test_residual_in_split_k_reduction(hk, kernel, splits):
    """A K split adds bias, activation and R in its reduction kernel."""
    M, N, K = (300 if kernel in (1, 6, 7) else 64), 1200, 2048
    A = synth.int_bf16(M, K, 81)
    B = synth.int_bf16(N, K, 82)
    bias = synth.int_bf16(1, N, 83)[0]
    R = synth.int_bf16(M, N, 84, -50, 50)
    got = run_fused(hk, A, B, bias, R, 1, split_k=splits, kernel=kernel)
    assert_bitexact(got, oracle.gemm_epilogue(A, B, bias, 1, residual=R), f"split-K residual {kernel}/{splits}")
    An, Bn = synth.normal_bf16(M, K, 85), synth.normal_bf16(N, K, 86)
    Rn = synth.normal_bf16(M, N, 87, 3.0)
    got = run_fused(hk, An, Bn, None, Rn, 2, split_k=splits, kernel=kernel)
    assert_close(got, oracle.gemm_epilogue(An, Bn, None, 2, residual=Rn), K, 1, 1, "split-K residual normal")


def test_residual_fp8_plan(hk):
    """An E4M3 plan: alpha, then the residual."""
    import torch
    M, N, K = 260, 300, 256
    A8, B8 = synth.int_e4m3(M, K, 91), synth.int_e4m3(N, K, 92)
    R = synth.int_bf16(M, N, 93, -20, 20)
    ldc = N + ((-N) % 8)
    a = torch.from_numpy(A8).to("cuda")
    b = torch.from_numpy(B8).to("cuda")
    C, Cstore = to_device(np.zeros((M, N), dtype=np.uint16), cols_pad=ldc - N)
    Rt, Rstore = to_device(R, cols_pad=ldc - N)
    plan = hk.Plan(M, N, K, lda=K, ldb=K, ldc=ldc, input_type=hk.HK_INPUT_E4M3, alpha=2.0)
    st = plan.run_fused_raw(a.data_ptr(), b.data_ptr(), C.data_ptr(), 0, Rt.data_ptr(), Rstore.stride(0), 0, 0,
                            int(torch.cuda.current_stream().cuda_stream))
    assert st == hk.HK_OK, hk.hk_gemm_last_error_string()
    torch.cuda.synchronize()
    got = to_host(Cstore)[:M, :N]
    table = np.array([oracle.e4m3_value(c) for c in range(256)])
    prod = 2.0 * (table[A8] @ table[B8].T)                     # exact: small integers
    want = synth.f32_to_bf16_bits((prod + synth.bf16_bits_to_f32(R)).astype(np.float32))
    assert_bitexact(got, want, "fp8 + residual")


def test_residual_argument_errors(hk):
    import torch
    A = torch.zeros((64, 64), dtype=torch.bfloat16, device="cuda")
    C = torch.zeros((64, 64), dtype=torch.bfloat16, device="cuda")
    R = torch.zeros((64, 80), dtype=torch.bfloat16, device="cuda")
    f = hk.hk_gemm_bf16_fused
    assert f(A.data_ptr(), A.data_ptr(), C.data_ptr(), 0, R.data_ptr() + 2, 64, 64, 64, 64, 64, 64, 80, 0, 0) \
        == hk.HK_ERR_MISALIGNED
    assert f(A.data_ptr(), A.data_ptr(), C.data_ptr(), 0, R.data_ptr(), 64, 64, 64, 64, 64, 64, 68, 0, 0) \
        == hk.HK_ERR_MISALIGNED
    assert f(A.data_ptr(), A.data_ptr(), C.data_ptr(), 0, R.data_ptr(), 64, 64, 64, 64, 64, 64, 56, 0, 0) \
        == hk.HK_ERR_INVALID_ARG
    # R == C needs ldr == ldc; a partial overlap with C is rejected
    Cw = torch.zeros((64, 80), dtype=torch.bfloat16, device="cuda")
    assert f(A.data_ptr(), A.data_ptr(), Cw.data_ptr(), 0, Cw.data_ptr(), 64, 64, 64, 64, 64, 80, 72, 0, 0) \
        == hk.HK_ERR_INVALID_ARG
    assert f(A.data_ptr(), A.data_ptr(), Cw.data_ptr(), 0, Cw.data_ptr() + 16, 64, 64, 64, 64, 64, 80, 80, 0, 0) \
        == hk.HK_ERR_INVALID_ARG
    assert f(A.data_ptr(), A.data_ptr(), C.data_ptr(), 0, R.data_ptr(), 64, 64, 64, 64, 64, 64, 80, 9, 0) \
        == hk.HK_ERR_INVALID_ARG
    torch.cuda.synchronize()


# ------------------------------------------------------------ FP8 (E4M3) --

def run_fp8(hk, A_codes, B_codes, sa=1.0, sb=1.0):
    import torch
    M, K = A_codes.shape
    N = B_codes.shape[0]
    kp = (-K) % 16
    def dev(x, pad):
        st = np.zeros((x.shape[0], x.shape[1] + pad), dtype=np.uint8)
        st[:, :x.shape[1]] = x
        return torch.from_numpy(st).to("cuda")
    A, B = dev(A_codes, kp), dev(B_codes, kp + 16)
    ldc = N + ((-N) % 8)
    C, Cstore = to_device(np.full((M, N), SENTINEL, dtype=np.uint16), rows_pad=1, cols_pad=ldc - N, fill=SENTINEL)
    st = hk.hk_gemm_fp8_e4m3(A.data_ptr(), B.data_ptr(), C.data_ptr(), M, N, K, A.stride(0), B.stride(0),
                             Cstore.stride(0), sa, sb, int(torch.cuda.current_stream().cuda_stream))
    assert st == hk.HK_OK, hk.hk_gemm_last_error_string()
    torch.cuda.synchronize()
    assert hk.hk_gemm_last_device_status(torch.cuda.current_device()) == hk.HK_OK
    full = to_host(Cstore)
    guard = full.copy()
    guard[:M, :N] = SENTINEL
    assert np.all(guard == SENTINEL), "a write landed outside C"
    return full[:M, :N]


@pytest.mark.parametrize("M,N,K", [(1, 1, 1), (256, 256, 128), (300, 517, 200), (64, 1000, 640), (1000, 1300, 1000),
                                   (2048, 2048, 2048)])
def test_fp8_integer_bitexact(hk, M, N, K):
    A = synth.int_e4m3(M, K, 1700 + M)
    B = synth.int_e4m3(N, K, 2700 + N)
    got = run_fp8(hk, A, B, 0.5, 0.25)
    assert_bitexact(got, oracle.gemm_fp8(A, B, 0.5, 0.25), f"fp8 int {M}x{N}x{K}")


@pytest.mark.parametrize("M,N,K", [(256, 256, 256), (300, 517, 200), (128, 4096, 4096), (1500, 700, 1900)])
def test_fp8_normal(hk, M, N, K):
    A = synth.normal_e4m3(M, K, 1800 + M)
    B = synth.normal_e4m3(N, K, 2800 + N)
    sa, sb = synth.FP8_SCALES
    got = run_fp8(hk, A, B, sa, sb)
    assert_close(got, oracle.gemm_fp8(A, B, sa, sb), K, sa, sb, f"fp8 {M}x{N}x{K}")


def test_fp8_workload_8192(hk):
    w = synth.FP8_WORKLOADS["fp8_gemm_8192"]
    A, B = synth.operands_fp8(w)
    sa, sb = synth.FP8_SCALES
    got = run_fp8(hk, A, B, sa, sb)
    r, c = synth.sample_positions(w.M, w.N, 3000 + w.wid)
    ref = oracle.gemm_fp8_entries(A, B, r, c, sa, sb)
    assert_close(got[r, c], ref, w.K, sa, sb, "fp8 8192^3 samples")


def test_fp8_argument_errors(hk):
    import torch
    A = torch.zeros((64, 64), dtype=torch.uint8, device="cuda")
    C = torch.zeros((64, 64), dtype=torch.bfloat16, device="cuda")
    assert hk.hk_gemm_fp8_e4m3(A.data_ptr(), A.data_ptr(), C.data_ptr(), 64, 64, 40, 40, 64, 64, 1.0, 1.0, 0) == \
        hk.HK_ERR_MISALIGNED
    assert hk.hk_gemm_fp8_e4m3(A.data_ptr(), A.data_ptr(), C.data_ptr(), 64, 64, 64, 64, 64, 64,
                               float("inf"), 1.0, 0) == hk.HK_ERR_INVALID_ARG


# ------------------------------------------------ graphs and concurrency --

def test_cuda_graph_capture_and_replay(hk):
    """After its first call on a device, hk_gemm_bf16 enqueues only a kernel
    launch, so a sequence of GEMMs can be captured into a CUDA graph and
    replayed."""
    import torch
    A = synth.int_bf16(512, 640, 11)
    B = synth.int_bf16(768, 640, 12)
    At, _ = to_device(A)
    Bt, _ = to_device(B)
    C = torch.empty((512, 768), dtype=torch.bfloat16, device="cuda")
    hk.gemm(At, Bt, out=C)                  # first call: per-device set-up outside the capture
    torch.cuda.synchronize()
    C.zero_()
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for _ in range(3):
            hk.gemm(At, Bt, out=C)
    torch.cuda.synchronize()
    C.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert_bitexact(to_host(C), oracle.gemm(A, B), "graph replay")
    assert hk.hk_gemm_last_device_status(torch.cuda.current_device()) == hk.HK_OK


def test_concurrent_streams_with_different_plans(hk):
    """Persistent GEMMs of different shapes on two streams at once: no
    kernel waits on another, so they can share the SMs in any order."""
    import torch
    shapes = [(2048, 2048, 1024), (128, 8192, 2048)]
    ops, outs, refs = [], [], []
    for i, (M, N, K) in enumerate(shapes):
        A = synth.int_bf16(M, K, 20 + i)
        B = synth.int_bf16(N, K, 30 + i)
        ops.append((to_device(A)[0], to_device(B)[0]))
        refs.append(oracle.gemm(A, B))
    streams = [torch.cuda.Stream() for _ in shapes]
    torch.cuda.synchronize()
    for rep in range(4):
        for (At, Bt), s in zip(ops, streams):
            with torch.cuda.stream(s):
                outs.append(hk.gemm(At, Bt))
    torch.cuda.synchronize()
    for i, C in enumerate(outs):
        assert_bitexact(to_host(C), refs[i % 2], f"stream {i % 2} rep {i // 2}")
    assert hk.hk_gemm_last_device_status(torch.cuda.current_device()) == hk.HK_OK


# ------------------------------------------------ special values (IEEE) --

def _exact_bf16(x: np.ndarray) -> np.ndarray:
    """float64 values that bf16 holds exactly (incl. ±Inf, NaN, subnormals) -> bf16 bits."""
    x = np.asarray(x, dtype=np.float64)
    f = np.ascontiguousarray(x.astype(np.float32))
    finite = np.isfinite(x)
    assert np.array_equal(f[finite].astype(np.float64), x[finite]), "value not exact in fp32"
    u = f.view(np.uint32)
    assert not np.any(u[finite] & np.uint32(0xFFFF)), "value not exact in bf16"
    return (u >> np.uint32(16)).astype(np.uint16)


def _gemm_bits(hk, A, B):
    At, _ = to_device(A)
    Bt, _ = to_device(B)
    C = hk.gemm(At, Bt)
    import torch
    torch.cuda.synchronize()
    assert hk.hk_gemm_last_device_status(torch.cuda.current_device()) == hk.HK_OK
    return to_host(C)


@pytest.mark.parametrize("M", [64, 300], ids=["single_cta", "cta_pair"])
def test_subnormal_inputs_are_not_flushed(hk, M):
    """A holds bf16 subnormals m·2^-133 (|m| ≤ 127), B holds k·2^100: every
    product m·k·2^-33 is normal and every sum is exact in fp32, so C matches
    the IEEE oracle bit for bit only if no subnormal input is flushed."""
    N, K = 200, 256
    g = np.random.Generator(np.random.PCG64(7100 + M))
    a = g.integers(-127, 128, size=(M, K)).astype(np.float64) * 2.0 ** -133
    b = g.integers(-4, 5, size=(N, K)).astype(np.float64) * 2.0 ** 100
    A, B = _exact_bf16(a), _exact_bf16(b)
    assert np.all((A & 0x7F80) == 0)                  # every input of A is subnormal or zero
    want = oracle.gemm(A, B)
    assert np.count_nonzero(want) > 0.9 * want.size
    assert_bitexact(_gemm_bits(hk, A, B), want, f"subnormal A, M={M}")


@pytest.mark.parametrize("M", [64, 300], ids=["single_cta", "cta_pair"])
def test_inf_and_nan_propagate_like_ieee(hk, M):
    """±Inf and NaN operands: Inf·k gives ±Inf, Inf·0 and Inf − Inf give NaN,
    NaN poisons its row (and a NaN in B its column); the other entries stay
    exact (integer data)."""
    N, K = 200, 256
    g = np.random.Generator(np.random.PCG64(7200 + M))
    a = g.integers(-4, 5, size=(M, K)).astype(np.float64)
    b = g.integers(-4, 5, size=(N, K)).astype(np.float64)
    a[1, 5] = np.inf
    a[2, 7] = -np.inf
    a[3, 9] = np.nan
    a[4, 11], a[4, 12] = np.inf, -np.inf
    b[6, 20] = np.inf
    b[7, 21] = np.nan
    A, B = _exact_bf16(a), _exact_bf16(b)
    want = oracle.gemm(A, B)
    nan = isnan_bf16(want)
    assert nan.any() and np.any(want == 0x7F80) and np.any(want == 0xFF80) and (~nan).sum() > 0.9 * want.size
    assert_same_ieee(_gemm_bits(hk, A, B), want, f"Inf/NaN, M={M}")


@pytest.mark.parametrize("M", [64, 300], ids=["single_cta", "cta_pair"])
def test_overflow_at_the_bf16_rounding(hk, M):
    """Sums that are finite in fp32 but round past the largest bf16
    ((2 − 2^-7)·2^127) become ±Inf, including the exact tie
    (2 − 2^-8)·2^127 (ties to even: the largest bf16 has an odd mantissa);
    the largest bf16 itself and 2^127 stay finite; 2^128 overflows."""
    N, K = 64, 8
    big = (2.0 - 2.0 ** -7) * 2.0 ** 126
    a = np.zeros((M, K))
    a[0, :2] = [2.0 ** 127, big]        # sum with B row 0: (2 - 2^-8)·2^127, a tie -> +Inf
    a[1, :2] = [big, big]               # (2 - 2^-7)·2^127: the largest bf16
    a[2, :2] = [2.0 ** 127, 2.0 ** 127]  # 2^128: overflows
    a[3, :2] = [-2.0 ** 127, -big]      # the negative tie -> -Inf
    a[4:, :] = np.random.Generator(np.random.PCG64(7300 + M)).integers(-4, 5, size=(M - 4, K))
    b = np.random.Generator(np.random.PCG64(7400 + M)).integers(-4, 5, size=(N, K)).astype(np.float64)
    b[0, :2] = [1.0, 1.0]
    b[1, :2] = [1.0, 0.0]               # row 0 of A: 2^127, finite
    b[2, :2] = [0.5, 0.5]               # halves: all of rows 0-3 finite
    b[:3, 2:] = 0.0
    A, B = _exact_bf16(a), _exact_bf16(b)
    want = oracle.gemm(A, B)
    assert want[0, 0] == 0x7F80 and want[1, 0] == 0x7F7F and want[2, 0] == 0x7F80 and want[3, 0] == 0xFF80
    assert want[0, 1] == 0x7F00 and want[2, 2] == 0x7F00
    assert_same_ieee(_gemm_bits(hk, A, B), want, f"overflow, M={M}")


@pytest.mark.parametrize("M", [64, 300], ids=["single_cta", "cta_pair"])
def test_fp8_subnormal_and_nan_codes(hk, M):
    """E4M3 subnormal operands (±m/8·2^-6) against small integers: every sum
    is exact in fp32, so C matches the oracle bit for bit only if no
    subnormal is flushed. The NaN codes S.1111.111 in A and in B poison
    their row and column; the other entries stay exact."""
    N, K = 200, 256
    g = np.random.Generator(np.random.PCG64(7500 + M))
    A = (g.integers(0, 8, size=(M, K)) | (g.integers(0, 2, size=(M, K)) << 7)).astype(np.uint8)
    B = synth.int_e4m3(N, K, 7600 + M)
    want = oracle.gemm_fp8(A, B, 1.0, 1.0)
    assert np.count_nonzero(want) > 0.9 * want.size
    assert_bitexact(run_fp8(hk, A, B, 1.0, 1.0), want, f"fp8 subnormal A, M={M}")
    A2 = synth.int_e4m3(M, K, 7700 + M)
    A2[1, 3], A2[2, 5] = 0x7F, 0xFF
    B2 = B.copy()
    B2[4, 7] = 0x7F
    want = oracle.gemm_fp8(A2, B2, 1.0, 1.0)
    assert isnan_bf16(want).any()
    assert_same_ieee(run_fp8(hk, A2, B2, 1.0, 1.0), want, f"fp8 NaN codes, M={M}")
