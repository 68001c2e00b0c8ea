"""GB300-native dense BF16 GEMM (C = A·Bᵀ, bf16 in, fp32 accumulate, bf16 out),
with its fused-epilogue (bias, activation, residual) and FP8 forms and the
attention forward (MHA / GQA) built on the same tensor-core primitives.

The compute path is the CUDA library built from ``csrc/`` for sm_103a and
reached through the C-ABI of ``include/hk_gemm.h``; this package is its
Python binding.
"""
from .hk_gemm import (HK_ACT_GELU, HK_ACT_NONE, HK_ACT_RELU, HK_ACT_SILU, HK_ERR_INVALID_ARG, HK_ERR_MISALIGNED,
                      HK_ERR_TIMEOUT, HK_ERR_UNSUPPORTED_DEVICE, HK_ERR_WORKSPACE, HK_FLAG_FAULT_DROP_ARRIVE,
                      HK_FLAG_NO_TAIL_SPLIT, HK_INPUT_BF16, HK_INPUT_E4M3, HK_OK, HKError, Plan, attention, gemm,
                      hk_attention_fwd, hk_attention_fwd_ex, hk_gemm_bf16, hk_gemm_bf16_epilogue, hk_gemm_bf16_fused,
                      hk_gemm_bf16_noalloc, hk_gemm_fp8_e4m3, hk_gemm_last_device_status, hk_gemm_last_error_string,
                      hk_gemm_mxfp8, hk_gemm_mxfp8_ex, hk_gemm_mxfp8_workspace_size, hk_status_string, load)

__all__ = ["attention", "gemm", "Plan", "HKError", "load",
           "hk_gemm_bf16", "hk_gemm_bf16_epilogue", "hk_gemm_bf16_fused", "hk_gemm_bf16_noalloc", "hk_gemm_fp8_e4m3",
           "hk_gemm_mxfp8", "hk_gemm_mxfp8_ex", "hk_gemm_mxfp8_workspace_size", "hk_attention_fwd",
           "hk_attention_fwd_ex", "hk_gemm_last_device_status", "hk_status_string", "hk_gemm_last_error_string",
           "HK_ACT_NONE", "HK_ACT_RELU", "HK_ACT_GELU", "HK_ACT_SILU", "HK_INPUT_BF16", "HK_INPUT_E4M3",
           "HK_OK", "HK_ERR_INVALID_ARG", "HK_ERR_MISALIGNED", "HK_ERR_TIMEOUT", "HK_ERR_WORKSPACE",
           "HK_ERR_UNSUPPORTED_DEVICE", "HK_FLAG_FAULT_DROP_ARRIVE", "HK_FLAG_NO_TAIL_SPLIT"]
