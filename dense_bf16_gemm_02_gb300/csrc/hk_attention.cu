// Host side of hk_attention_fwd (include/hk_gemm.h): argument checks, the
// three 3-D TMA tensor maps over Q, K and V, and the launch of the
// attention-forward kernel.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <mutex>

#include "../../include/hk_gemm.h"
#include "attn_kernel.cuh"
#include "host_internal.h"

namespace {

hk_status fail(hk_status s, const char* fmt, ...) __attribute__((format(printf, 2, 3)));
hk_status fail(hk_status s, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    return hk_host::set_error(s, buf);
}

hk_status cuda_fail(hk_status s, const char* what, cudaError_t e) {
    return fail(s, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

constexpr uint64_t kDefaultTimeoutNs = 1000000000ull;   // 1 s per bounded wait
constexpr int kMaxDevices = 64;

// Per-device one-time kernel set-up (the dynamic shared-memory opt-in).
std::mutex g_setup_mutex;
bool g_setup[kMaxDevices] = {};

template <int kD>
hk_status setup_kernel() {
    cudaError_t e = cudaFuncSetAttribute(hk::attn::attn_fwd_kernel<kD>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         hk::attn::AttnGeometry<kD>::kSmemBytes);
    if (e != cudaSuccess) return cuda_fail(HK_ERR_CUDA, "configuring the attention kernel", e);
    return HK_OK;
}

// 3-D bf16 tensor map over a contiguous [heads, S, D] array with a box of
// 64 columns × 128 rows × 1 head and 128-byte swizzling; rows past S read as 0.
hk_status encode_heads(PFN_cuTensorMapEncodeTiled_v12000 enc, CUtensorMap* map, const void* ptr, int64_t heads,
                       int64_t S, int64_t D, const char* name) {
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(S), static_cast<cuuint64_t>(heads)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * 2, static_cast<cuuint64_t>(S * D) * 2};
    cuuint32_t box[3] = {64, 128, 1};
    cuuint32_t elem_strides[3] = {1, 1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box,
                     elem_strides, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return fail(HK_ERR_INVALID_ARG, "encoding the tensor map of %s failed (CUresult %d)", name, (int)r);
    return HK_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" hk_status hk_attention_fwd_ex(const void* Q, const void* K, const void* V, void* O, float* lse,
                                         int64_t B, int64_t Hq, int64_t Hkv, int64_t S, int64_t D, int32_t causal,
                                         uint32_t flags, uint64_t timeout_ns, void* stream) {
    if (B < 0 || Hq < 0 || Hkv < 0 || S < 0) return fail(HK_ERR_INVALID_ARG, "negative size");
    if (D != 64 && D != 128) return fail(HK_ERR_INVALID_ARG, "head dimension %lld (supported: 64, 128)", (long long)D);
    if (Hkv == 0 ? Hq != 0 : (Hq % Hkv) != 0)
        return fail(HK_ERR_INVALID_ARG, "Hq=%lld is not a multiple of Hkv=%lld", (long long)Hq, (long long)Hkv);
    const int64_t lim = (int64_t(1) << 31) - 1;
    if (B * Hq > lim || S > lim || B * Hq * ((S + 255) / 256) > lim || B * Hq * S > lim)
        return fail(HK_ERR_INVALID_ARG, "problem too large (B*Hq*S must stay below 2^31)");
    if (B == 0 || Hq == 0 || S == 0) return HK_OK;
    if (!Q || !K || !V || !O) return fail(HK_ERR_INVALID_ARG, "null operand pointer");
    if (!aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned16(O))
        return fail(HK_ERR_MISALIGNED, "Q, K, V and O must be 16-byte aligned");
    if (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)) return fail(HK_ERR_MISALIGNED, "lse must be 4-byte aligned");

    int device = 0;
    cudaError_t e = cudaGetDevice(&device);
    if (e != cudaSuccess) return cuda_fail(HK_ERR_CUDA, "cudaGetDevice", e);
    if (device < 0 || device >= kMaxDevices) return fail(HK_ERR_INVALID_ARG, "device %d out of range", device);
    int sm_count = 0;
    hk_status s = hk_host::check_device(device, &sm_count);
    if (s != HK_OK) return s;
    {
        std::lock_guard<std::mutex> lock(g_setup_mutex);
        if (!g_setup[device]) {
            if ((s = setup_kernel<64>()) != HK_OK || (s = setup_kernel<128>()) != HK_OK) return s;
            g_setup[device] = true;
        }
    }
    uint32_t* status = nullptr;
    if ((s = hk_host::status_word(device, &status)) != HK_OK) return s;
    PFN_cuTensorMapEncodeTiled_v12000 enc = nullptr;
    if ((s = hk_host::tensor_map_encoder(&enc)) != HK_OK) return s;

    CUtensorMap tq, tk, tv;
    if ((s = encode_heads(enc, &tq, Q, B * Hq, S, D, "Q")) != HK_OK) return s;
    if ((s = encode_heads(enc, &tk, K, B * Hkv, S, D, "K")) != HK_OK) return s;
    if ((s = encode_heads(enc, &tv, V, B * Hkv, S, D, "V")) != HK_OK) return s;

    hk::attn::AttnParams p = {};
    p.B = static_cast<int32_t>(B);
    p.Hq = static_cast<int32_t>(Hq);
    p.Hkv = static_cast<int32_t>(Hkv);
    p.S = static_cast<int32_t>(S);
    p.causal = causal ? 1 : 0;
    p.q_pairs = static_cast<int32_t>((S + 255) / 256);
    p.n_items = static_cast<int32_t>(B * Hq * p.q_pairs);
    p.kv_blocks = static_cast<int32_t>((S + 127) / 128);
    p.scale_log2 = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(D)));
    p.O = static_cast<uint16_t*>(O);
    p.lse = lse;
    p.status = status;
    p.launch_id = hk_host::next_launch_id();
    p.flags = flags;
    p.timeout_ns = timeout_ns ? timeout_ns : kDefaultTimeoutNs;

    // persistent: one CTA per SM (at most one per work item), each walking its items
    const unsigned grid = static_cast<unsigned>(std::min<int64_t>(B * Hq * p.q_pairs, sm_count));
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (D == 64) {
        hk::attn::attn_fwd_kernel<64><<<grid, hk::attn::AttnGeometry<64>::kThreads, hk::attn::AttnGeometry<64>::kSmemBytes, st>>>(
            tq, tk, tv, p);
    } else {
        hk::attn::attn_fwd_kernel<128><<<grid, hk::attn::AttnGeometry<128>::kThreads, hk::attn::AttnGeometry<128>::kSmemBytes, st>>>(
            tq, tk, tv, p);
    }
    e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(HK_ERR_LAUNCH, "launching the attention kernel", e);
    return HK_OK;
}

extern "C" hk_status hk_attention_fwd(const void* Q, const void* K, const void* V, void* O, float* lse, int64_t B,
                                      int64_t Hq, int64_t Hkv, int64_t S, int64_t D, int32_t causal, void* stream) {
    return hk_attention_fwd_ex(Q, K, V, O, lse, B, Hq, Hkv, S, D, causal, 0u, 0u, stream);
}
