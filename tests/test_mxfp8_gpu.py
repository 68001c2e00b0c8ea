"""GPU parity of the MXFP8 GEMM (hk_gemm_mxfp8) against the oracle.

Integer E4M3 data with scales 2^-1 .. 2^1 keep every partial sum an exact
multiple of 2^-2 far below 2^24, so fp32 accumulation in any order is exact
and the result must match the oracle bit for bit. Normal data with wider
scales is compared within 2^-7·|C| (one bf16 rounding step) plus 2^-16 times
the sum of the absolute scaled products (far above fp32 accumulation error).
"""
from __future__ import annotations

import numpy as np
import pytest

import synth
from gpu_util import assert_bitexact, assert_same_ieee, isnan_bf16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def hk():
    import torch
    if not torch.cuda.is_available():
        pytest.fail("no CUDA device")
    import dense_bf16_gemm_02_gb300 as pkg
    pkg.load()
    return pkg


@pytest.fixture(scope="module")
def oracle():
    import oracle as o
    o.build()
    return o


def run_mx(hk, A, B, SA, SB, ws_extra=0):
    import torch
    M, K = A.shape
    N = B.shape[0]
    dev = lambda x: torch.from_numpy(np.ascontiguousarray(x)).to("cuda")
    a, b, sa, sb = dev(A), dev(B), dev(SA), dev(SB)
    ldc = max(8, N + (-N) % 8)
    c = torch.full((M, ldc), float("nan"), dtype=torch.bfloat16, device="cuda")
    nbytes = hk.hk_gemm_mxfp8_workspace_size(M, N, K)
    ws = torch.empty(max(nbytes + ws_extra, 256), dtype=torch.uint8, device="cuda")
    st = hk.hk_gemm_mxfp8(a.data_ptr(), b.data_ptr(), sa.data_ptr(), sb.data_ptr(), c.data_ptr(), M, N, K, K, K,
                          K // 32, K // 32, ldc, ws.data_ptr(), nbytes + ws_extra, 0)
    assert st == hk.HK_OK, hk.hk_gemm_last_error_string()
    torch.cuda.synchronize()
    assert hk.hk_gemm_last_device_status(0) == hk.HK_OK
    out = c.view(torch.int16).cpu().numpy().view(np.uint16)
    assert np.all(out[:, N:] == np.uint16(0x7FC0)), "padding columns of C were written"
    return out[:, :N]


def abs_scaled(A, B, SA, SB):
    """Σ_b 2^(SA+SB-254)·Σ_{k∈b}|a·b| in float64 (tolerance scale)."""
    fa = np.abs(np.vectorize(lambda c: synth_e4m3(c))(A))
    fb = np.abs(np.vectorize(lambda c: synth_e4m3(c))(B))
    K = A.shape[1]
    out = np.zeros((A.shape[0], B.shape[0]))
    for blk in range(K // 32):
        sl = slice(32 * blk, 32 * blk + 32)
        out += np.exp2(SA[:, blk:blk + 1].astype(np.float64) - 127) * np.exp2(SB[:, blk].astype(np.float64) - 127)[None, :] \
            * (fa[:, sl] @ fb[:, sl].T)
    return out


_E4M3 = None


def synth_e4m3(code):
    global _E4M3
    if _E4M3 is None:
        import oracle
        _E4M3 = np.array([oracle.e4m3_value(c) for c in range(256)])
    return _E4M3[int(code)]


SHAPES = [(256, 384, 256), (300, 500, 320), (1, 200, 64), (100, 1000, 512), (129, 193, 32), (200, 190, 160),
          (1024, 1152, 1024)]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_mx_integer_inputs_bit_exact(hk, oracle, shape):
    M, N, K = shape
    A, B = synth.int_e4m3(M, K, 1300 + M), synth.int_e4m3(N, K, 1400 + N)
    SA, SB = synth.mx_scales(M, K // 32, 1500, 126, 128), synth.mx_scales(N, K // 32, 1600, 126, 128)
    got = run_mx(hk, A, B, SA, SB)
    assert_bitexact(got, oracle.gemm_mxfp8(A, B, SA, SB), f"mxfp8 integer {shape}")


@pytest.mark.parametrize("shape", [(256, 384, 256), (300, 500, 320), (100, 1000, 512)], ids=lambda s: "x".join(map(str, s)))
def test_mx_normal_inputs(hk, oracle, shape):
    M, N, K = shape
    A, B = synth.normal_e4m3(M, K, 1700 + M), synth.normal_e4m3(N, K, 1800 + N)
    SA, SB = synth.mx_scales(M, K // 32, 1900, 120, 134), synth.mx_scales(N, K // 32, 2000, 120, 134)
    got = synth.bf16_bits_to_f32(run_mx(hk, A, B, SA, SB)).astype(np.float64)
    want = synth.bf16_bits_to_f32(oracle.gemm_mxfp8(A, B, SA, SB)).astype(np.float64)
    tol = 2.0 ** -7 * np.abs(want) + 2.0 ** -16 * abs_scaled(A, B, SA, SB)
    bad = np.abs(got - want) > tol
    assert not bad.any(), f"{int(bad.sum())} entries outside tolerance, first {np.argwhere(bad)[:3].tolist()}"


def test_mx_scales_matter_per_block(hk, oracle):
    """A block's scale moves only the products of that block: raising the A
    scales of block 3 by 4 (×16) must match the oracle exactly."""
    M, N, K = 128, 192, 256
    A, B = synth.int_e4m3(M, K, 2100), synth.int_e4m3(N, K, 2200)
    SA = np.full((M, K // 32), 127, np.uint8)
    SB = np.full((N, K // 32), 127, np.uint8)
    SA[:, 3] = 131
    SB[::3, 5] = 125
    assert_bitexact(run_mx(hk, A, B, SA, SB), oracle.gemm_mxfp8(A, B, SA, SB), "mxfp8 per-block scales")


def test_mx_workload_sampled(hk, oracle):
    w = synth.MX_WORKLOADS["mxfp8_gemm_8192"]
    A, B, SA, SB = synth.operands_mx(w)
    got = run_mx(hk, A, B, SA, SB)
    r, c = synth.sample_positions(w.M, w.N, 3000 + w.wid, count=2048, tile_m=128, tile_n=256)
    want = oracle.gemm_mxfp8_entries(A, B, SA, SB, r, c)
    g = synth.bf16_bits_to_f32(got[r, c]).astype(np.float64)
    ref = synth.bf16_bits_to_f32(want).astype(np.float64)
    # |scaled terms| ≤ 2^6 per product, K = 8192 terms, N(0,1) data: 2^-16·Σ|..| bounded by 2^-16·2^6·K·E|ab|
    tol = 2.0 ** -7 * np.abs(ref) + 2.0 ** -16 * 64 * w.K * 0.7
    bad = np.abs(g - ref) > tol
    assert not bad.any(), f"{int(bad.sum())} sampled entries outside tolerance"


@pytest.mark.parametrize("lds,offset", [((12, 16), (0, 0)), ((13, 8), (0, 0)), ((8, 8), (1, 3))],
                         ids=["padded_words", "odd_stride", "odd_offset"])
def test_mx_strided_scales(hk, oracle, lds, offset):
    """Scale arrays with row strides above K/32 and at odd byte offsets: the
    arrangement reads them with 4-byte loads only when every row's scales of a
    stage are an aligned word, else byte by byte; both must give the oracle's
    result exactly (integer data)."""
    import torch
    M, N, K = 300, 260, 256
    kb = K // 32
    A, B = synth.int_e4m3(M, K, 2300), synth.int_e4m3(N, K, 2400)
    SA, SB = synth.mx_scales(M, kb, 2500, 126, 128), synth.mx_scales(N, kb, 2600, 126, 128)

    def placed(S, ld, off):
        buf = torch.full((S.shape[0] * ld + off + 16,), 255, dtype=torch.uint8)   # 255 (NaN) in the padding
        view = buf[off:off + S.shape[0] * ld].view(S.shape[0], ld)
        view[:, :kb] = torch.from_numpy(S)
        return buf.to("cuda"), off

    (sa_buf, oa), (sb_buf, ob) = placed(SA, lds[0], offset[0]), placed(SB, lds[1], offset[1])
    dev = lambda x: torch.from_numpy(np.ascontiguousarray(x)).to("cuda")
    a, b = dev(A), dev(B)
    ldc = N + (-N) % 8
    c = torch.full((M, ldc), float("nan"), dtype=torch.bfloat16, device="cuda")
    nbytes = hk.hk_gemm_mxfp8_workspace_size(M, N, K)
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    st = hk.hk_gemm_mxfp8(a.data_ptr(), b.data_ptr(), sa_buf.data_ptr() + oa, sb_buf.data_ptr() + ob, c.data_ptr(),
                          M, N, K, K, K, lds[0], lds[1], ldc, ws.data_ptr(), nbytes, 0)
    assert st == hk.HK_OK, hk.hk_gemm_last_error_string()
    torch.cuda.synchronize()
    assert hk.hk_gemm_last_device_status(0) == hk.HK_OK
    got = c.view(torch.int16).cpu().numpy().view(np.uint16)[:, :N]
    assert_bitexact(got, oracle.gemm_mxfp8(A, B, SA, SB), f"mxfp8 strided scales {lds} {offset}")


def test_mx_argument_errors(hk):
    import torch
    x = torch.zeros(4096, dtype=torch.uint8, device="cuda")
    p = x.data_ptr()
    assert hk.hk_gemm_mxfp8(p, p, p, p, p, 64, 64, 48, 48, 48, 2, 2, 64, p, 4096, 0) == hk.HK_ERR_INVALID_ARG
    need = hk.hk_gemm_mxfp8_workspace_size(64, 64, 64)
    assert need > 0
    assert hk.hk_gemm_mxfp8(p, p, p, p, p, 64, 64, 64, 64, 64, 2, 2, 64, p, need - 1, 0) == hk.HK_ERR_WORKSPACE
    assert hk.hk_gemm_mxfp8(p, p, p, p, p, 64, 64, 64, 64, 64, 1, 2, 64, p, need, 0) == hk.HK_ERR_INVALID_ARG


@pytest.mark.parametrize("M", [300, 100], ids=["pair_256x256", "single_128x192"])
def test_mx_bounded_wait_reports_timeout_and_recovers(hk, oracle, M):
    """Fault set on the host: the producer withholds one arrival, so the scale
    copier's wait on that stage (and the MMA thread's behind it) runs out
    after 20 ms; every role drains and returns, the status word reports
    HK_ERR_TIMEOUT once, and the next call on the same context is exact.
    Unknown flag bits are rejected."""
    import torch
    N, K = 260, 256
    kb = K // 32
    A, B = synth.int_e4m3(M, K, 2700 + M), synth.int_e4m3(N, K, 2800)
    SA, SB = synth.mx_scales(M, kb, 2900, 126, 128), synth.mx_scales(N, kb, 3000, 126, 128)
    dev = lambda x: torch.from_numpy(np.ascontiguousarray(x)).to("cuda")
    a, b, sa, sb = dev(A), dev(B), dev(SA), dev(SB)
    ldc = N + (-N) % 8
    c = torch.zeros((M, ldc), dtype=torch.bfloat16, device="cuda")
    nbytes = hk.hk_gemm_mxfp8_workspace_size(M, N, K)
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")

    def call(flags, timeout_ns):
        return hk.hk_gemm_mxfp8_ex(a.data_ptr(), b.data_ptr(), sa.data_ptr(), sb.data_ptr(), c.data_ptr(), M, N, K,
                                   K, K, kb, kb, ldc, ws.data_ptr(), nbytes, flags, timeout_ns, 0)

    assert call(hk.HK_FLAG_FAULT_DROP_ARRIVE, 20_000_000) == hk.HK_OK, hk.hk_gemm_last_error_string()
    torch.cuda.synchronize()
    assert hk.hk_gemm_last_device_status(0) == hk.HK_ERR_TIMEOUT
    assert hk.hk_gemm_last_device_status(0) == hk.HK_OK   # read-and-clear
    assert call(0, 0) == hk.HK_OK, hk.hk_gemm_last_error_string()
    torch.cuda.synchronize()
    assert hk.hk_gemm_last_device_status(0) == hk.HK_OK
    got = c.view(torch.int16).cpu().numpy().view(np.uint16)[:, :N]
    assert_bitexact(got, oracle.gemm_mxfp8(A, B, SA, SB), f"mxfp8 {M}x{N}x{K} after timeout")
    assert call(0x4, 0) == hk.HK_ERR_INVALID_ARG


@pytest.mark.parametrize("M", [100, 300], ids=["single_128x192", "pair_256x256"])
def test_mx_subnormal_and_nan_codes(hk, oracle, M):
    """E4M3 subnormal operands against small integers with scales 2^-1..2^1:
    exact in fp32, so bit-exact only if nothing is flushed. E4M3 NaN codes
    in A and B, and the UE8M0 NaN scale (255) on one block of a row of A and
    of a row of B, give NaN where IEEE arithmetic on the decoded values does
    (a NaN scale poisons its whole row or column); the rest stays exact."""
    N, K = 200, 128
    kb = K // 32
    g = np.random.Generator(np.random.PCG64(7800 + M))
    A = (g.integers(0, 8, size=(M, K)) | (g.integers(0, 2, size=(M, K)) << 7)).astype(np.uint8)
    B = synth.int_e4m3(N, K, 7900 + M)
    SA, SB = synth.mx_scales(M, kb, 8000 + M, 126, 128), synth.mx_scales(N, kb, 8100, 126, 128)
    want = oracle.gemm_mxfp8(A, B, SA, SB)
    assert np.count_nonzero(want) > 0.9 * want.size
    assert_bitexact(run_mx(hk, A, B, SA, SB), want, f"mxfp8 subnormal A, M={M}")
    A2, B2 = synth.int_e4m3(M, K, 8200 + M), B.copy()
    A2[1, 3] = 0x7F
    B2[4, 40] = 0xFF
    SA2, SB2 = SA.copy(), SB.copy()
    SA2[5, 2] = 255
    SB2[6, 1] = 255
    want = oracle.gemm_mxfp8(A2, B2, SA2, SB2)
    assert isnan_bf16(want[5]).all() and isnan_bf16(want[:, 6]).all()
    assert_same_ieee(run_mx(hk, A2, B2, SA2, SB2), want, f"mxfp8 NaN codes and scale, M={M}")
