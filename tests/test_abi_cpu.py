"""The C-ABI library without a GPU: it loads, exports every entry point the
header declares, and rejects invalid arguments on the host before any CUDA
call is made. No computation is attempted here."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "hk_gemm.h")


@pytest.fixture(scope="module")
def lib():
    from dense_bf16_gemm_02_gb300 import build
    build.build()
    from dense_bf16_gemm_02_gb300 import hk_gemm
    return hk_gemm.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(hk_\w+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for want in ("hk_gemm_bf16", "hk_gemm_plan_create", "hk_gemm_plan_run", "hk_gemm_plan_workspace_size",
                 "hk_gemm_plan_destroy", "hk_status_string"):
        assert want in names


def test_every_declared_symbol_is_exported(lib):
    from dense_bf16_gemm_02_gb300 import hk_gemm
    out = subprocess.run(["nm", "-D", "--defined-only", hk_gemm.LIB_PATH], capture_output=True, text=True,
                         check=True).stdout
    exported = set(re.findall(r"\sT\s(\w+)", out))
    missing = [n for n in declared_functions() if n not in exported]
    assert not missing, missing
    for n in declared_functions():
        assert hasattr(lib, n)
    assert set(hk_gemm.EXPORTED) <= set(declared_functions())


def test_status_strings(lib):
    for code in range(8):
        s = lib.hk_status_string(code).decode()
        assert s.startswith("HK_")
    assert b"unknown" in lib.hk_status_string(99)


def test_host_validation_without_gpu(lib):
    from dense_bf16_gemm_02_gb300 import hk_gemm as h
    P = 1 << 20  # a 16-byte aligned fake address; never dereferenced on these paths
    # empty problems return HK_OK without touching the device
    assert lib.hk_gemm_bf16(None, None, None, 0, 5, 5, 8, 8, 8, None) == h.HK_OK
    assert lib.hk_gemm_bf16(None, None, None, 5, 0, 5, 8, 8, 8, None) == h.HK_OK
    # negative sizes / small leading dimensions
    assert lib.hk_gemm_bf16(P, P, P, -1, 8, 8, 8, 8, 8, None) == h.HK_ERR_INVALID_ARG
    assert lib.hk_gemm_bf16(P, P, P, 8, 8, 16, 8, 16, 8, None) == h.HK_ERR_INVALID_ARG
    assert lib.hk_gemm_bf16(P, P, P, 8, 16, 8, 8, 8, 8, None) == h.HK_ERR_INVALID_ARG
    assert lib.hk_gemm_bf16(P, P, P, 1 << 31, 8, 8, 8, 8, 8, None) == h.HK_ERR_INVALID_ARG
    # leading dimensions not multiples of 8, unaligned pointers, null pointers
    assert lib.hk_gemm_bf16(P, P, P, 8, 8, 12, 12, 16, 8, None) == h.HK_ERR_MISALIGNED
    assert lib.hk_gemm_bf16(P + 2, P, P, 8, 8, 8, 8, 8, 8, None) == h.HK_ERR_MISALIGNED
    assert lib.hk_gemm_bf16(P, P, P + 8, 8, 8, 8, 8, 8, 8, None) == h.HK_ERR_MISALIGNED
    assert lib.hk_gemm_bf16(None, P, P, 8, 8, 8, 8, 8, 8, None) == h.HK_ERR_INVALID_ARG
    assert lib.hk_gemm_bf16(P, P, None, 8, 8, 8, 8, 8, 8, None) == h.HK_ERR_INVALID_ARG
    assert b"leading" in lib.hk_gemm_last_error_string() or b"null" in lib.hk_gemm_last_error_string()
    # plan creation with invalid shapes fails on the host
    handle = ctypes.c_void_p()
    assert lib.hk_gemm_plan_create(ctypes.byref(handle), -5, 8, 8, 8, 8, 8, 0, None) == h.HK_ERR_INVALID_ARG
    assert not handle.value
    assert lib.hk_gemm_plan_create(None, 8, 8, 8, 8, 8, 8, 0, None) == h.HK_ERR_INVALID_ARG
    assert lib.hk_gemm_plan_run(None, P, P, P, None, 0, None) == h.HK_ERR_INVALID_ARG
    lib.hk_gemm_plan_destroy(None)


def test_attention_host_validation_without_gpu(lib):
    from dense_bf16_gemm_02_gb300 import hk_gemm as h
    P = 1 << 20
    att = lib.hk_attention_fwd
    # empty problems: nothing launched
    assert att(None, None, None, None, None, 0, 8, 2, 128, 128, 0, None) == h.HK_OK
    assert att(None, None, None, None, None, 2, 8, 2, 0, 64, 1, None) == h.HK_OK
    # head dimension, head grouping, negative sizes, size limit
    assert att(P, P, P, P, None, 1, 8, 2, 128, 96, 0, None) == h.HK_ERR_INVALID_ARG
    assert b"head dimension" in lib.hk_gemm_last_error_string()
    assert att(P, P, P, P, None, 1, 8, 3, 128, 128, 0, None) == h.HK_ERR_INVALID_ARG
    assert att(P, P, P, P, None, 1, 8, 0, 128, 128, 0, None) == h.HK_ERR_INVALID_ARG
    assert att(P, P, P, P, None, -1, 8, 2, 128, 128, 0, None) == h.HK_ERR_INVALID_ARG
    assert att(P, P, P, P, None, 1 << 16, 64, 8, 1 << 16, 128, 0, None) == h.HK_ERR_INVALID_ARG
    # null and misaligned pointers
    assert att(None, P, P, P, None, 1, 8, 2, 128, 128, 0, None) == h.HK_ERR_INVALID_ARG
    assert att(P, P, P + 8, P, None, 1, 8, 2, 128, 128, 0, None) == h.HK_ERR_MISALIGNED
    assert att(P, P, P, P, P + 2, 1, 8, 2, 128, 128, 0, None) == h.HK_ERR_MISALIGNED


def test_product_path_has_no_oracle_or_fallback():
    """The CUDA package never imports the oracle and has no CPU path."""
    pkg = os.path.join(ROOT, "dense_bf16_gemm_02_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                text = open(os.path.join(dirpath, f)).read()
                assert not re.search(r"^\s*(import|from)\s+oracle\b", text, re.M), f
                assert "torch.matmul" not in text and "cublas" not in text.lower(), f


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    from dense_bf16_gemm_02_gb300 import hk_gemm
    monkeypatch.setattr(hk_gemm, "_lib", None)
    monkeypatch.setattr(hk_gemm, "LIB_PATH", str(tmp_path / "absent.so"))
    with pytest.raises(RuntimeError, match="missing"):
        hk_gemm.load()


def test_mxfp8_host_validation_without_gpu(lib):
    """Argument checks of the block-scaled entry points run on the host,
    before any device call; the workspace size is a host computation."""
    from dense_bf16_gemm_02_gb300 import hk_gemm as h
    P = 1 << 20
    lib.hk_gemm_mxfp8_ex.argtypes = [ctypes.c_void_p] * 5 + [ctypes.c_int64] * 8 + [
        ctypes.c_void_p, ctypes.c_size_t, ctypes.c_uint32, ctypes.c_uint64, ctypes.c_void_p]
    lib.hk_gemm_mxfp8_ex.restype = ctypes.c_int32
    lib.hk_gemm_mxfp8_workspace_size.argtypes = [ctypes.c_int64] * 3
    lib.hk_gemm_mxfp8_workspace_size.restype = ctypes.c_size_t

    def mx(M=64, N=64, K=64, lda=64, ldb=64, ldsa=2, ldsb=2, ldc=64, a=P, sa=P, ws=P, wsb=1 << 20, flags=0):
        return lib.hk_gemm_mxfp8_ex(a, P, sa, P, P, M, N, K, lda, ldb, ldsa, ldsb, ldc, ws, wsb, flags, 0, None)

    assert mx(flags=0x4) == h.HK_ERR_INVALID_ARG and b"flags" in lib.hk_gemm_last_error_string()
    assert mx(K=48, lda=48, ldb=48) == h.HK_ERR_INVALID_ARG               # K not a multiple of 32
    assert mx(K=32, lda=40, ldb=40) == h.HK_ERR_MISALIGNED                 # FP8 ld not a multiple of 16
    assert mx(ldsa=1) == h.HK_ERR_INVALID_ARG                              # scale ld below K/32
    assert mx(M=0) == h.HK_OK and mx(N=0) == h.HK_OK                       # nothing to do
    assert mx(a=0) == h.HK_ERR_INVALID_ARG                                 # null operand
    assert mx(sa=0) == h.HK_ERR_INVALID_ARG                                # null scales
    need = lib.hk_gemm_mxfp8_workspace_size(64, 64, 64)
    assert need > 0 and need % 256 == 0
    assert mx(wsb=need - 1) == h.HK_ERR_WORKSPACE
    assert mx(ws=P + 128, wsb=need) == h.HK_ERR_WORKSPACE                  # not 256-byte aligned
    assert lib.hk_gemm_mxfp8_workspace_size(0, 64, 64) == 0
    # more K blocks or more tiles never need less workspace
    sizes = [lib.hk_gemm_mxfp8_workspace_size(m, n, k) for m, n, k in
             [(64, 64, 128), (64, 64, 256), (64, 512, 256), (300, 512, 256), (8192, 8192, 8192)]]
    assert sizes == sorted(sizes) and sizes[0] < sizes[-1]


def test_no_multicast_bulk_copies():
    """No TMA or bulk copy in the library's sources carries a multicast
    qualifier: every load reads this GPU's memory into the issuing CTA only
    (a pair's loads of one stage complete on the leader CTA's barrier, without
    multicast). The one multicast form that stays is tcgen05.commit's
    `.multicast::cluster`, an mbarrier arrival on the two CTAs of one pair, not
    a copy. The rule is checked on the code of every source under csrc/ and
    include/ (comments excluded)."""
    bad = []
    for d in ("dense_bf16_gemm_02_gb300/csrc", "include"):
        for f in sorted(os.listdir(os.path.join(ROOT, d))):
            if not f.endswith((".cu", ".cuh", ".h")):
                continue
            text = open(os.path.join(ROOT, d, f), encoding="utf-8").read()
            code = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
            code = re.sub(r"//[^\n]*", " ", code)
            for m in re.finditer(r'"[^"\n]*multicast[^"\n]*"', code):
                lit = m.group(0)
                if "cp.async.bulk" in lit or "cp.reduce.async.bulk" in lit or not lit.lstrip('"').startswith(
                        "tcgen05.commit"):
                    bad.append(f"{d}/{f}: {lit}")
    assert not bad, bad
