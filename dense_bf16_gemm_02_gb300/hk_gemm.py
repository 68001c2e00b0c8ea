"""Thin ctypes binding of the C-ABI in ``include/hk_gemm.h``.

Argument marshalling only: every step of the GEMM runs in the CUDA library.
The functions keep the C names; ``gemm`` and ``Plan`` are conveniences over
them for torch tensors. There is no fallback: if the compiled library is
missing, loading fails loudly.
"""
from __future__ import annotations

import ctypes
import os
import threading

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "_build", "libhk_gemm.so")

HK_OK = 0
HK_ERR_INVALID_ARG = 1
HK_ERR_MISALIGNED = 2
HK_ERR_UNSUPPORTED_DEVICE = 3
HK_ERR_LAUNCH = 4
HK_ERR_TIMEOUT = 5
HK_ERR_WORKSPACE = 6
HK_ERR_CUDA = 7

HK_KERNEL_AUTO = 0
HK_KERNEL_PAIR_256x256 = 1
HK_KERNEL_SINGLE_128x256 = 2
HK_KERNEL_SINGLE_128x192 = 3
HK_KERNEL_SINGLE_128x128 = 4
HK_KERNEL_SINGLE_128x64 = 5
HK_KERNEL_PAIR_256x128 = 6
HK_KERNEL_PAIR_256x112 = 7
KERNELS = (HK_KERNEL_PAIR_256x256, HK_KERNEL_SINGLE_128x256, HK_KERNEL_SINGLE_128x192,
           HK_KERNEL_SINGLE_128x128, HK_KERNEL_SINGLE_128x64, HK_KERNEL_PAIR_256x128, HK_KERNEL_PAIR_256x112)

HK_ACT_NONE = 0
HK_ACT_RELU = 1
HK_ACT_GELU = 2
HK_ACT_SILU = 3

HK_INPUT_BF16 = 0
HK_INPUT_E4M3 = 1

HK_FLAG_NONE = 0x0
HK_FLAG_FAULT_DROP_ARRIVE = 0x1
HK_FLAG_NO_TAIL_SPLIT = 0x2

EXPORTED = (
    "hk_gemm_bf16", "hk_gemm_plan_create", "hk_gemm_plan_workspace_size", "hk_gemm_plan_get_info",
    "hk_gemm_plan_run", "hk_gemm_plan_device_status", "hk_gemm_last_device_status",
    "hk_gemm_plan_destroy", "hk_status_string", "hk_gemm_last_error_string", "hk_gemm_bf16_noalloc",
    "hk_gemm_bf16_epilogue", "hk_gemm_plan_run_epilogue", "hk_gemm_bf16_fused", "hk_gemm_plan_run_fused",
    "hk_gemm_fp8_e4m3",
    "hk_attention_fwd", "hk_attention_fwd_ex", "hk_gemm_mxfp8", "hk_gemm_mxfp8_ex", "hk_gemm_mxfp8_workspace_size",
)


class hk_gemm_config(ctypes.Structure):
    _fields_ = [("group_m", ctypes.c_int32), ("max_clusters", ctypes.c_int32),
                ("split_k", ctypes.c_int32), ("kernel", ctypes.c_int32),
                ("timeout_ns", ctypes.c_uint64), ("flags", ctypes.c_uint32),
                ("activation", ctypes.c_uint32), ("input_type", ctypes.c_int32), ("alpha", ctypes.c_float)]


class hk_gemm_plan_info(ctypes.Structure):
    _fields_ = [("M", ctypes.c_int64), ("N", ctypes.c_int64), ("K", ctypes.c_int64),
                ("kernel", ctypes.c_int32), ("ctas_per_unit", ctypes.c_int32),
                ("tile_m", ctypes.c_int32), ("tile_n", ctypes.c_int32), ("tile_k", ctypes.c_int32),
                ("stages", ctypes.c_int32), ("num_tiles", ctypes.c_int32),
                ("grid_ctas", ctypes.c_int32), ("group_m", ctypes.c_int32),
                ("split_k", ctypes.c_int32), ("kernels_per_run", ctypes.c_int32),
                ("smem_bytes", ctypes.c_int32), ("workspace_bytes", ctypes.c_size_t),
                ("tail_split_tiles", ctypes.c_int32), ("reserved", ctypes.c_int32)]

    def as_dict(self) -> dict:
        return {name: getattr(self, name) for name, _ in self._fields_}


class HKError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        lib = load()
        super().__init__(f"{where}: {lib.hk_status_string(status).decode()} "
                         f"({lib.hk_gemm_last_error_string().decode()})")


_lib = None
_lock = threading.Lock()


def load() -> ctypes.CDLL:
    """Load the compiled library (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"the CUDA library {LIB_PATH} is missing: run "
                               "`python -c 'import __graft_entry__ as g; g.build()'` first")
        lib = ctypes.CDLL(LIB_PATH)
        P, I64, I32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
        lib.hk_gemm_bf16.argtypes = [P, P, P, I64, I64, I64, I64, I64, I64, P]
        lib.hk_gemm_bf16.restype = I32
        lib.hk_gemm_plan_create.argtypes = [ctypes.POINTER(P), I64, I64, I64, I64, I64, I64, I32,
                                            ctypes.POINTER(hk_gemm_config)]
        lib.hk_gemm_plan_create.restype = I32
        lib.hk_gemm_plan_workspace_size.argtypes = [P]
        lib.hk_gemm_plan_workspace_size.restype = ctypes.c_size_t
        lib.hk_gemm_plan_get_info.argtypes = [P, ctypes.POINTER(hk_gemm_plan_info)]
        lib.hk_gemm_plan_get_info.restype = I32
        lib.hk_gemm_plan_run.argtypes = [P, P, P, P, P, ctypes.c_size_t, P]
        lib.hk_gemm_plan_run.restype = I32
        lib.hk_gemm_plan_device_status.argtypes = [P]
        lib.hk_gemm_plan_device_status.restype = I32
        lib.hk_gemm_last_device_status.argtypes = [I32]
        lib.hk_gemm_last_device_status.restype = I32
        lib.hk_gemm_plan_destroy.argtypes = [P]
        lib.hk_gemm_plan_destroy.restype = None
        lib.hk_status_string.argtypes = [I32]
        lib.hk_status_string.restype = ctypes.c_char_p
        lib.hk_gemm_last_error_string.argtypes = []
        lib.hk_gemm_last_error_string.restype = ctypes.c_char_p
        lib.hk_gemm_bf16_epilogue.argtypes = [P, P, P, P, I64, I64, I64, I64, I64, I64, ctypes.c_int32, P]
        lib.hk_gemm_bf16_epilogue.restype = I32
        lib.hk_gemm_plan_run_epilogue.argtypes = [P, P, P, P, P, P, ctypes.c_size_t, P]
        lib.hk_gemm_plan_run_epilogue.restype = I32
        lib.hk_gemm_bf16_fused.argtypes = [P, P, P, P, P, I64, I64, I64, I64, I64, I64, I64, ctypes.c_int32, P]
        lib.hk_gemm_bf16_fused.restype = I32
        lib.hk_gemm_plan_run_fused.argtypes = [P, P, P, P, P, P, I64, P, ctypes.c_size_t, P]
        lib.hk_gemm_plan_run_fused.restype = I32
        lib.hk_gemm_fp8_e4m3.argtypes = [P, P, P, I64, I64, I64, I64, I64, I64, ctypes.c_float, ctypes.c_float, P]
        lib.hk_gemm_fp8_e4m3.restype = I32
        lib.hk_gemm_bf16_noalloc.argtypes = [P, P, P, I64, I64, I64, I64, I64, I64, ctypes.c_int32, P]
        lib.hk_gemm_bf16_noalloc.restype = I32
        lib.hk_gemm_mxfp8.argtypes = [P, P, P, P, P, I64, I64, I64, I64, I64, I64, I64, I64, P, ctypes.c_size_t, P]
        lib.hk_gemm_mxfp8.restype = I32
        lib.hk_gemm_mxfp8_ex.argtypes = [P, P, P, P, P, I64, I64, I64, I64, I64, I64, I64, I64, P, ctypes.c_size_t,
                                         ctypes.c_uint32, ctypes.c_uint64, P]
        lib.hk_gemm_mxfp8_ex.restype = I32
        lib.hk_gemm_mxfp8_workspace_size.argtypes = [I64, I64, I64]
        lib.hk_gemm_mxfp8_workspace_size.restype = ctypes.c_size_t
        lib.hk_attention_fwd.argtypes = [P, P, P, P, P, I64, I64, I64, I64, I64, I32, P]
        lib.hk_attention_fwd.restype = I32
        lib.hk_attention_fwd_ex.argtypes = [P, P, P, P, P, I64, I64, I64, I64, I64, I32, ctypes.c_uint32,
                                            ctypes.c_uint64, P]
        lib.hk_attention_fwd_ex.restype = I32
        _lib = lib
        return lib


# ------------------------------------------------------------ raw C names --

def hk_gemm_bf16(A: int, B: int, C: int, M: int, N: int, K: int, lda: int, ldb: int, ldc: int,
                 stream: int = 0) -> int:
    return load().hk_gemm_bf16(A, B, C, M, N, K, lda, ldb, ldc, stream)


def hk_gemm_bf16_epilogue(A: int, B: int, C: int, bias: int, M: int, N: int, K: int, lda: int, ldb: int,
                          ldc: int, activation: int = 0, stream: int = 0) -> int:
    """C = bf16(act(A·Bᵀ + bias)) (bias: device pointer or 0)."""
    return load().hk_gemm_bf16_epilogue(A, B, C, bias or None, M, N, K, lda, ldb, ldc, activation, stream)


def hk_gemm_bf16_fused(A: int, B: int, C: int, bias: int, R: int, M: int, N: int, K: int, lda: int, ldb: int,
                       ldc: int, ldr: int, activation: int = 0, stream: int = 0) -> int:
    """C = bf16(act(A·Bᵀ + bias) + R) (bias, R: device pointers or 0; R may be C with ldr == ldc)."""
    return load().hk_gemm_bf16_fused(A, B, C, bias or None, R or None, M, N, K, lda, ldb, ldc, ldr, activation,
                                     stream)


def hk_gemm_fp8_e4m3(A: int, B: int, C: int, M: int, N: int, K: int, lda: int, ldb: int, ldc: int,
                     scale_a: float = 1.0, scale_b: float = 1.0, stream: int = 0) -> int:
    """C (bf16) = (scale_a·scale_b)·A·Bᵀ for E4M3 operands A (M×K), B (N×K)."""
    return load().hk_gemm_fp8_e4m3(A, B, C, M, N, K, lda, ldb, ldc, scale_a, scale_b, stream)


def hk_gemm_bf16_noalloc(A: int, B: int, C: int, M: int, N: int, K: int, lda: int, ldb: int, ldc: int,
                         split_k: int = 0, stream: int = 0) -> int:
    """The GEMM that allocates nothing (scratch in a fixed array of the library)."""
    return load().hk_gemm_bf16_noalloc(A, B, C, M, N, K, lda, ldb, ldc, split_k, stream)


def hk_gemm_mxfp8(A: int, B: int, SFA: int, SFB: int, C: int, M: int, N: int, K: int, lda: int, ldb: int,
                  ldsfa: int, ldsfb: int, ldc: int, workspace: int, workspace_bytes: int, stream: int = 0) -> int:
    """C (bf16) = block-scaled A·Bᵀ: E4M3 A (M×K), B (N×K), UE8M0 scales per 32 K elements."""
    return load().hk_gemm_mxfp8(A, B, SFA, SFB, C, M, N, K, lda, ldb, ldsfa, ldsfb, ldc, workspace or None,
                                workspace_bytes, stream)


def hk_gemm_mxfp8_ex(A: int, B: int, SFA: int, SFB: int, C: int, M: int, N: int, K: int, lda: int, ldb: int,
                     ldsfa: int, ldsfb: int, ldc: int, workspace: int, workspace_bytes: int, flags: int = 0,
                     timeout_ns: int = 0, stream: int = 0) -> int:
    return load().hk_gemm_mxfp8_ex(A, B, SFA, SFB, C, M, N, K, lda, ldb, ldsfa, ldsfb, ldc, workspace or None,
                                   workspace_bytes, flags, timeout_ns, stream)


def hk_gemm_mxfp8_workspace_size(M: int, N: int, K: int) -> int:
    return int(load().hk_gemm_mxfp8_workspace_size(M, N, K))


def hk_attention_fwd(Q: int, K: int, V: int, O: int, lse: int, B: int, Hq: int, Hkv: int, S: int, D: int,
                     causal: int = 0, stream: int = 0) -> int:
    """O = softmax(Q·Kᵀ/√D)·V (GQA; Q, O [B,Hq,S,D], K, V [B,Hkv,S,D] bf16; lse fp32 [B,Hq,S] or 0)."""
    return load().hk_attention_fwd(Q, K, V, O, lse or None, B, Hq, Hkv, S, D, int(causal), stream)


def hk_attention_fwd_ex(Q: int, K: int, V: int, O: int, lse: int, B: int, Hq: int, Hkv: int, S: int, D: int,
                        causal: int = 0, flags: int = 0, timeout_ns: int = 0, stream: int = 0) -> int:
    return load().hk_attention_fwd_ex(Q, K, V, O, lse or None, B, Hq, Hkv, S, D, int(causal), flags,
                                      timeout_ns, stream)


def hk_gemm_last_device_status(device: int) -> int:
    return load().hk_gemm_last_device_status(device)


def hk_status_string(status: int) -> str:
    return load().hk_status_string(status).decode()


def hk_gemm_last_error_string() -> str:
    return load().hk_gemm_last_error_string().decode()


# ------------------------------------------------------- torch helpers --

def _check_operand(t, name):
    import torch
    if not isinstance(t, torch.Tensor) or t.dtype != torch.bfloat16 or not t.is_cuda or t.dim() != 2:
        raise TypeError(f"{name} must be a 2-D bfloat16 CUDA tensor")
    if t.size(1) > 1 and t.stride(1) != 1:
        raise ValueError(f"{name} must be contiguous along its last dimension")


def _stream_handle(stream) -> int:
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream)


def gemm(A, B, out=None, stream=None):
    """C = A·Bᵀ for bf16 CUDA tensors A (M×K) and B (N×K); returns C (M×N)."""
    import torch
    _check_operand(A, "A")
    _check_operand(B, "B")
    M, K = A.shape
    N, K2 = B.shape
    if K != K2:
        raise ValueError(f"A is {M}x{K} but B is {N}x{K2}")
    if out is None:
        # rows padded to a multiple of 8 elements (the TMA stride rule); a view is returned
        ldc_pad = max(8, N + (-N) % 8)
        out = torch.empty((M, ldc_pad), dtype=torch.bfloat16, device=A.device)[:, :N]
    else:
        _check_operand(out, "out")
        if tuple(out.shape) != (M, N):
            raise ValueError("out has the wrong shape")
    lda = max(A.stride(0), K) if M > 1 else max(K + (-K) % 8, 8)
    ldb = max(B.stride(0), K) if N > 1 else max(K + (-K) % 8, 8)
    ldc = max(out.stride(0), N) if M > 1 else max(N + (-N) % 8, 8)
    st = hk_gemm_bf16(A.data_ptr(), B.data_ptr(), out.data_ptr(), M, N, K, lda, ldb, ldc,
                      _stream_handle(stream))
    if st != HK_OK:
        raise HKError(st, "hk_gemm_bf16")
    return out


def attention(q, k, v, causal: bool = False, return_lse: bool = False, out=None, stream=None):
    """softmax(q·kᵀ/√D)·v for contiguous bf16 CUDA tensors q [B, Hq, S, D] and
    k, v [B, Hkv, S, D] (Hkv divides Hq; D 64 or 128). Returns o [B, Hq, S, D]
    (and the fp32 log-sum-exp [B, Hq, S] with ``return_lse``)."""
    import torch
    for t, name in ((q, "q"), (k, "k"), (v, "v")):
        if (not isinstance(t, torch.Tensor) or t.dtype != torch.bfloat16 or not t.is_cuda or t.dim() != 4
                or not t.is_contiguous()):
            raise TypeError(f"{name} must be a contiguous 4-D bfloat16 CUDA tensor")
    B, Hq, S, D = q.shape
    Hkv = k.shape[1]
    if tuple(k.shape) != (B, Hkv, S, D) or tuple(v.shape) != tuple(k.shape):
        raise ValueError("k and v must be [B, Hkv, S, D] with q's B, S and D")
    if out is None:
        out = torch.empty_like(q)
    lse = torch.empty((B, Hq, S), dtype=torch.float32, device=q.device) if return_lse else None
    st = hk_attention_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                          lse.data_ptr() if lse is not None else 0, B, Hq, Hkv, S, D, int(causal),
                          _stream_handle(stream))
    if st != HK_OK:
        raise HKError(st, "hk_attention_fwd")
    return (out, lse) if return_lse else out


class Plan:
    """A plan for one GEMM shape (wraps hk_gemm_plan_*)."""

    def __init__(self, M, N, K, lda=None, ldb=None, ldc=None, device=0, group_m=0, max_clusters=0,
                 split_k=0, timeout_ns=0, flags=0, kernel=0, activation=0, input_type=0, alpha=0.0):
        lib = load()
        self._lib = lib
        self.M, self.N, self.K = M, N, K
        cfg = hk_gemm_config(group_m=group_m, max_clusters=max_clusters, split_k=split_k,
                             timeout_ns=timeout_ns, flags=flags, kernel=kernel, activation=activation,
                             input_type=input_type, alpha=alpha)
        handle = ctypes.c_void_p()
        st = lib.hk_gemm_plan_create(ctypes.byref(handle), M, N, K, lda if lda is not None else K,
                                     ldb if ldb is not None else K, ldc if ldc is not None else N,
                                     device, ctypes.byref(cfg))
        if st != HK_OK:
            raise HKError(st, "hk_gemm_plan_create")
        self._h = handle

    @property
    def workspace_size(self) -> int:
        return int(self._lib.hk_gemm_plan_workspace_size(self._h))

    def info(self) -> dict:
        inf = hk_gemm_plan_info()
        st = self._lib.hk_gemm_plan_get_info(self._h, ctypes.byref(inf))
        if st != HK_OK:
            raise HKError(st, "hk_gemm_plan_get_info")
        return inf.as_dict()

    def run_raw(self, A: int, B: int, C: int, workspace: int = 0, workspace_bytes: int = 0,
                stream: int = 0) -> int:
        return self._lib.hk_gemm_plan_run(self._h, A, B, C, workspace, workspace_bytes, stream)

    def run(self, A, B, C, workspace=None, stream=None):
        """Run on torch tensors. Without an explicit workspace, one is
        allocated once (through torch) and kept with the plan."""
        import torch
        if workspace is None and self.workspace_size > 0:
            if getattr(self, "_ws", None) is None:
                self._ws = torch.empty(self.workspace_size + 256, dtype=torch.uint8, device=A.device)
            ws = (self._ws.data_ptr() + 255) & ~255
            wsb = self.workspace_size
        else:
            ws = 0 if workspace is None else workspace.data_ptr()
            wsb = 0 if workspace is None else workspace.numel() * workspace.element_size()
        st = self.run_raw(A.data_ptr(), B.data_ptr(), C.data_ptr(), ws, wsb, _stream_handle(stream))
        if st != HK_OK:
            raise HKError(st, "hk_gemm_plan_run")
        return C

    def run_epilogue_raw(self, A: int, B: int, C: int, bias: int = 0, workspace: int = 0, workspace_bytes: int = 0,
                         stream: int = 0) -> int:
        return self._lib.hk_gemm_plan_run_epilogue(self._h, A, B, C, bias or None, workspace, workspace_bytes,
                                                   stream)

    def run_fused_raw(self, A: int, B: int, C: int, bias: int = 0, R: int = 0, ldr: int = 0, workspace: int = 0,
                      workspace_bytes: int = 0, stream: int = 0) -> int:
        return self._lib.hk_gemm_plan_run_fused(self._h, A, B, C, bias or None, R or None, ldr, workspace,
                                                workspace_bytes, stream)

    def device_status(self) -> int:
        return int(self._lib.hk_gemm_plan_device_status(self._h))

    def close(self):
        if getattr(self, "_h", None):
            self._lib.hk_gemm_plan_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
