// Host side of the C-ABI declared in include/hk_gemm.h: argument checks,
// plans, TMA tensor-map encoding, the device status word and the cluster
// launch of the persistent GEMM kernel.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <cmath>
#include <cstdlib>
#include <cstring>
#include <memory>
#include <mutex>
#include <new>
#include <string>

#include "../../include/hk_gemm.h"
#include "gemm_kernel.cuh"
#include "host_internal.h"

namespace {

thread_local std::string g_last_error;

hk_status fail(hk_status s, const char* fmt, ...) __attribute__((format(printf, 2, 3)));
hk_status fail(hk_status s, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return s;
}

hk_status cuda_fail(hk_status s, const char* what, cudaError_t e) {
    return fail(s, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

#ifndef HK_PAIR_ATOMS
#define HK_PAIR_ATOMS 1   // K atoms per stage of the bf16 pair kernel (1: 64 K elements, 6 stages; 2: 128, 3 stages)
#endif
#ifndef HK_PDL
#define HK_PDL 1   // launch every GEMM as a programmatic dependent of the previous kernel on its stream
#endif
#ifndef HK_MX_PAIR_ATOMS
// K atoms per stage of the block-scaled pair kernel: two (256 K elements, 3 stages)
// measured no faster than one (626K vs 621K kernel cycles at 8192^3)
#define HK_MX_PAIR_ATOMS 1
#endif
#ifndef HK_FP8_PAIR_ATOMS
#define HK_FP8_PAIR_ATOMS 1
#endif

constexpr int kMaxDevices = 64;
constexpr uint64_t kDefaultTimeoutNs = 1000000000ull;   // 1 s per bounded wait
constexpr int kDefaultGroupM = 8;

// -------------------------------------------------------------- variants --

using KernelFn = void (*)(CUtensorMap, CUtensorMap, CUtensorMap, CUtensorMap, hk::GemmParams);

struct Variant {
    int id;            // value of hk_gemm_config.kernel
    int cg;            // CTAs per work unit (1 or 2)
    int tile_m, tile_n;
    int stages, smem_bytes;
    bool fp8;          // E4M3 operands (else bf16)
    bool mx;           // block-scaled E4M3 (MXFP8); never chosen automatically
    int a_rows_max;    // rows of A a stage holds (16 or 64 for the decode kernels, else 128)
    int k_elems;       // K elements per pipeline stage
    int atoms;         // 128-byte K atoms per stage (TMA boxes per operand and stage)
    int sf_bytes;      // MXFP8: bytes of scale blocks per K block and CTA
    bool halves;       // the tail split may run its tiles as two half-width units
    KernelFn fn;
    const char* name;
};

template <int kCG, int kTileN, bool kFp8, bool kMx = false, int kARows = hk::kCtaM, int kAtoms = 1>
constexpr Variant make_variant(int id, const char* name) {
    using G = hk::Geometry<kCG, kTileN, kFp8, kMx, kARows, kAtoms>;
    return Variant{id, kCG, G::kTileM, G::kTileN, G::kStages, G::kSmemBytes, kFp8, kMx, G::kARowsMax, G::kKElems,
                   kAtoms, G::kSfBytes, G::kHalves, &hk::gemm_bf16_kernel<kCG, kTileN, kFp8, kMx, kARows, kAtoms>,
                   name};
}

const Variant kVariants[] = {
    // decode (M <= 16, M <= 64): single-CTA tiles with 16- or 64-row A stages, so more
    // stages of B are in flight; listed before the 128-row forms (shortest first) so that
    // they win the time model's ties
    make_variant<1, 256, false, false, 16>(HK_KERNEL_SINGLE_128x256, "single 128x256, 16-row A"),
    make_variant<1, 192, false, false, 16>(HK_KERNEL_SINGLE_128x192, "single 128x192, 16-row A"),
    make_variant<1, 128, false, false, 16>(HK_KERNEL_SINGLE_128x128, "single 128x128, 16-row A"),
    make_variant<1, 64, false, false, 16>(HK_KERNEL_SINGLE_128x64, "single 128x64, 16-row A"),
    make_variant<1, 256, false, false, 64>(HK_KERNEL_SINGLE_128x256, "single 128x256, 64-row A"),
    make_variant<1, 192, false, false, 64>(HK_KERNEL_SINGLE_128x192, "single 128x192, 64-row A"),
    make_variant<1, 128, false, false, 64>(HK_KERNEL_SINGLE_128x128, "single 128x128, 64-row A"),
    make_variant<1, 64, false, false, 64>(HK_KERNEL_SINGLE_128x64, "single 128x64, 64-row A"),
    make_variant<2, 256, false, false, hk::kCtaM, HK_PAIR_ATOMS>(HK_KERNEL_PAIR_256x256, "pair 256x256"),
    make_variant<2, 128, false, false>(HK_KERNEL_PAIR_256x128, "pair 256x128"),
    // 8192 columns make 74 tiles of 112 for the 76 pairs of a GB300 (64 of 128)
    make_variant<2, 112, false, false>(HK_KERNEL_PAIR_256x112, "pair 256x112"),
    make_variant<1, 256, false>(HK_KERNEL_SINGLE_128x256, "single 128x256"),
    make_variant<1, 192, false>(HK_KERNEL_SINGLE_128x192, "single 128x192"),
    make_variant<1, 128, false>(HK_KERNEL_SINGLE_128x128, "single 128x128"),
    make_variant<1, 64, false>(HK_KERNEL_SINGLE_128x64, "single 128x64"),
    make_variant<2, 256, true, false, hk::kCtaM, HK_FP8_PAIR_ATOMS>(HK_KERNEL_PAIR_256x256, "fp8 pair 256x256"),
    make_variant<1, 256, true>(HK_KERNEL_SINGLE_128x256, "fp8 single 128x256"),
    make_variant<1, 192, true>(HK_KERNEL_SINGLE_128x192, "fp8 single 128x192"),
    make_variant<1, 128, true>(HK_KERNEL_SINGLE_128x128, "fp8 single 128x128"),
    make_variant<1, 64, true>(HK_KERNEL_SINGLE_128x64, "fp8 single 128x64"),
    make_variant<1, 192, true, true>(HK_KERNEL_SINGLE_128x192, "mxfp8 single 128x192"),
    make_variant<2, 256, true, true, hk::kCtaM, HK_MX_PAIR_ATOMS>(HK_KERNEL_PAIR_256x256, "mxfp8 pair 256x256"),
};
// N of the MXFP8 tiles: one CTA 128x192 (two TMEM accumulators), a pair
// 256x256 (one accumulator, see Geometry::kAccBufs)
constexpr int kMxTileNSingle = 192;
constexpr int kMxTileNPair = 256;
using GeomMxSingle = hk::Geometry<1, kMxTileNSingle, true, true>;
using GeomMxPair = hk::Geometry<2, kMxTileNPair, true, true, hk::kCtaM, HK_MX_PAIR_ATOMS>;
static_assert(GeomMxSingle::kSfbAtoms == GeomMxPair::kSfbAtoms, "one scale layout");
static_assert(GeomMxPair::kAccBufs == 1 && GeomMxSingle::kAccBufs == 2, "MXFP8 accumulator buffering");
constexpr int kMxSfbAtoms = GeomMxPair::kSfbAtoms;
constexpr int kNumVariants = sizeof(kVariants) / sizeof(kVariants[0]);

const Variant* find_variant(int id, bool fp8, bool mx = false) {
    for (const Variant& v : kVariants)
        if (v.id == id && v.fp8 == fp8 && v.mx == mx) return &v;
    return nullptr;
}

// ----------------------------------------------------------- device info --

struct DeviceInfo {
    bool probed = false;
    bool supported = false;
    int sm_count = 0;
    int max_units[kNumVariants] = {};   // co-resident work units (pairs or CTAs) per variant
    std::string why;
};

std::mutex g_dev_mutex;
DeviceInfo g_dev[kMaxDevices];

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

hk_status device_info(int device, const DeviceInfo** out) {
    if (device < 0 || device >= kMaxDevices) return fail(HK_ERR_INVALID_ARG, "device %d out of range", device);
    std::lock_guard<std::mutex> lock(g_dev_mutex);
    DeviceInfo& d = g_dev[device];
    if (!d.probed) {
        int major = 0, minor = 0;
        cudaError_t e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, device);
        if (e == cudaSuccess) e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, device);
        if (e == cudaSuccess) e = cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, device);
        if (e != cudaSuccess) return cuda_fail(HK_ERR_CUDA, "querying the device", e);
        if (major != 10 || minor != 3) {
            d.probed = true;
            d.supported = false;
            d.why = "compute capability " + std::to_string(major) + "." + std::to_string(minor) +
                    " (this library is built for 10.3, sm_103a)";
        } else {
            int prev = -1;
            cudaGetDevice(&prev);
            if (prev != device) cudaSetDevice(device);
            for (int i = 0; i < kNumVariants && e == cudaSuccess; ++i) {
                const Variant& v = kVariants[i];
                e = cudaFuncSetAttribute(v.fn, cudaFuncAttributeMaxDynamicSharedMemorySize, v.smem_bytes);
                if (e != cudaSuccess) break;
                if (v.cg == 2) {
                    cudaLaunchConfig_t cfg = {};
                    cudaLaunchAttribute attr[1];
                    attr[0].id = cudaLaunchAttributeClusterDimension;
                    attr[0].val.clusterDim.x = 2;
                    attr[0].val.clusterDim.y = 1;
                    attr[0].val.clusterDim.z = 1;
                    cfg.gridDim = dim3(2 * d.sm_count, 1, 1);
                    cfg.blockDim = dim3(hk::kThreads, 1, 1);
                    cfg.dynamicSmemBytes = v.smem_bytes;
                    cfg.attrs = attr;
                    cfg.numAttrs = 1;
                    e = cudaOccupancyMaxActiveClusters(&d.max_units[i], v.fn, &cfg);
                } else {
                    int per_sm = 0;
                    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, v.fn, hk::kThreads, v.smem_bytes);
                    d.max_units[i] = per_sm * d.sm_count;
                }
            }
            if (prev >= 0 && prev != device) cudaSetDevice(prev);
            if (e != cudaSuccess) return cuda_fail(HK_ERR_CUDA, "configuring the GEMM kernels", e);
            d.probed = true;
            d.supported = d.max_units[0] > 0;   // the bf16 pair kernel
            if (!d.supported) d.why = "no 2-CTA cluster of the GEMM kernel fits on the device";
        }
    }
    if (!d.supported) return fail(HK_ERR_UNSUPPORTED_DEVICE, "device %d: %s", device, d.why.c_str());
    *out = &d;
    return HK_OK;
}

hk_status get_encoder() {
    std::call_once(g_encode_once, [] {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    });
    if (!g_encode) return fail(HK_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
    return HK_OK;
}

// 2-D bf16 tensor map over a row-major (rows × cols, leading dimension ld)
// matrix with box (box_cols × box_rows).
hk_status encode_2d(CUtensorMap* map, const void* ptr, int64_t rows, int64_t cols, int64_t ld,
                    uint32_t box_cols, uint32_t box_rows, CUtensorMapSwizzle swizzle, const char* name,
                    bool bytes = false) {
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * (bytes ? 1u : 2u)};
    cuuint32_t box[2] = {box_cols, box_rows};
    cuuint32_t elem_strides[2] = {1, 1};
    CUresult r = g_encode(map, bytes ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                          const_cast<void*>(ptr), dims, strides, box,
                          elem_strides, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(HK_ERR_INVALID_ARG, "encoding the tensor map of %s failed (CUresult %d)", name, (int)r);
    return HK_OK;
}

// Launch ids are unique in the process: the kernel uses them to recognise
// its own abort flag and its own split-K arrival counters.
std::atomic<uint32_t> g_next_launch{1};

uint32_t next_launch_id() {
    uint32_t id = g_next_launch.fetch_add(1, std::memory_order_relaxed);
    if (id == 0) id = g_next_launch.fetch_add(1, std::memory_order_relaxed);
    return id;
}

// Per-device context of the one-shot entry point: its status word.
struct StatusWord {
    uint32_t* dev = nullptr;                 // [0] error bits, [1] aborted launch id
};

std::mutex g_ctx_mutex;
StatusWord* g_ctx[kMaxDevices] = {};

hk_status alloc_status(StatusWord* w) {
    cudaError_t e = cudaMalloc(&w->dev, 4 * sizeof(uint32_t));
    if (e == cudaSuccess) e = cudaMemset(w->dev, 0, 4 * sizeof(uint32_t));
    if (e != cudaSuccess) return cuda_fail(HK_ERR_CUDA, "allocating the device status word", e);
    return HK_OK;
}

hk_status read_status(StatusWord* w, int device) {
    int prev = -1;
    cudaGetDevice(&prev);
    if (prev != device) cudaSetDevice(device);
    uint32_t h[2] = {0, 0};
    cudaError_t e = cudaDeviceSynchronize();
    if (e == cudaSuccess) e = cudaMemcpy(h, w->dev, sizeof h, cudaMemcpyDeviceToHost);
    if (e == cudaSuccess && h[0] != 0) e = cudaMemset(w->dev, 0, sizeof(uint32_t));
    if (prev >= 0 && prev != device) cudaSetDevice(prev);
    if (e != cudaSuccess) return cuda_fail(HK_ERR_CUDA, "reading the device status word", e);
    if (h[0] != 0)
        return fail(HK_ERR_TIMEOUT, "a bounded wait in the GEMM kernel ran out (error bits 0x%x)", h[0]);
    return HK_OK;
}

// ------------------------------------------------------------ validation --

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

hk_status check_shape(int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb, int64_t ldc) {
    const int64_t lim = (int64_t(1) << 31) - 1;
    if (M < 0 || N < 0 || K < 0) return fail(HK_ERR_INVALID_ARG, "negative size (M=%lld N=%lld K=%lld)", (long long)M, (long long)N, (long long)K);
    if (M > lim || N > lim || K > lim) return fail(HK_ERR_INVALID_ARG, "size above 2^31-1");
    if (lda < (K > 0 ? K : 1) || ldb < (K > 0 ? K : 1) || ldc < (N > 0 ? N : 1))
        return fail(HK_ERR_INVALID_ARG, "leading dimension too small (lda=%lld ldb=%lld ldc=%lld)", (long long)lda,
                    (long long)ldb, (long long)ldc);
    if (lda > lim || ldb > lim || ldc > lim) return fail(HK_ERR_INVALID_ARG, "leading dimension above 2^31-1");
    if ((lda % 8) || (ldb % 8) || (ldc % 8))
        return fail(HK_ERR_MISALIGNED, "leading dimensions must be multiples of 8 elements (lda=%lld ldb=%lld ldc=%lld)",
                    (long long)lda, (long long)ldb, (long long)ldc);
    return HK_OK;
}

hk_status check_pointers(const void* A, const void* B, const void* C, int64_t K) {
    if (!C || (K > 0 && (!A || !B))) return fail(HK_ERR_INVALID_ARG, "null operand pointer");
    if (!aligned16(C) || (K > 0 && (!aligned16(A) || !aligned16(B))))
        return fail(HK_ERR_MISALIGNED, "operand pointers must be 16-byte aligned");
    return HK_OK;
}

// The residual of a fused epilogue: NULL, or an M×N bf16 matrix, 16-byte
// aligned with ldr a multiple of 8 and at least N, that is C itself (same
// pointer and leading dimension: an in-place update) or does not overlap C.
hk_status check_residual(const void* R, int64_t ldr, const void* C, int64_t M, int64_t N, int64_t ldc) {
    if (!R) return HK_OK;
    if (ldr < (N > 0 ? N : 1) || ldr > (int64_t(1) << 31) - 1)
        return fail(HK_ERR_INVALID_ARG, "residual leading dimension %lld outside [N, 2^31)", (long long)ldr);
    if (!aligned16(R) || (ldr % 8))
        return fail(HK_ERR_MISALIGNED, "the residual must be 16-byte aligned with ldr a multiple of 8 (ldr=%lld)",
                    (long long)ldr);
    if (R == C) {
        if (ldr != ldc) return fail(HK_ERR_INVALID_ARG, "a residual that is C must have ldr == ldc");
        return HK_OK;
    }
    const uintptr_t r0 = reinterpret_cast<uintptr_t>(R), c0 = reinterpret_cast<uintptr_t>(C);
    const uintptr_t r1 = r0 + 2u * static_cast<uintptr_t>((M - 1) * ldr + N);
    const uintptr_t c1 = c0 + 2u * static_cast<uintptr_t>((M - 1) * ldc + N);
    if (r0 < c1 && c0 < r1) return fail(HK_ERR_INVALID_ARG, "the residual overlaps C without being C");
    return HK_OK;
}

struct DeviceGuard {
    int prev = -1;
    explicit DeviceGuard(int device) {
        if (cudaGetDevice(&prev) != cudaSuccess) prev = -1;
        if (prev != device) cudaSetDevice(device);
    }
    ~DeviceGuard() {
        int cur = -1;
        if (prev >= 0 && cudaGetDevice(&cur) == cudaSuccess && cur != prev) cudaSetDevice(prev);
    }
};

}  // namespace

// ------------------------------------------------------------------ plans --

// Tensor maps of one set of operand pointers (encoding them costs host time
// on every call otherwise; a plan keeps the last set it ran with).
struct TensorMaps {
    bool valid = false;
    const void* a = nullptr;
    const void* b = nullptr;
    const void* c = nullptr;
    const void* scales = nullptr;   // MXFP8: the arranged scale blocks
    size_t scale_bytes = 0;
    CUtensorMap ta, tb, tc, tbh;
};

struct hk_gemm_plan {
    int64_t M, N, K, lda, ldb, ldc;
    int device;
    const Variant* variant;
    int sm_count;
    size_t ws_bytes;            // split K: fp32 partial matrices [splits][M][n_pad]
    hk::GemmParams params;      // everything but status/launch id
    int grid_ctas;
    hk_gemm_config cfg;
    StatusWord status;
    bool owns_status;
    // the tensor maps of the last run's pointers (runs may come from several threads)
    mutable std::mutex tmap_mutex;
    mutable TensorMaps tmaps;
};

namespace {

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Rows of A one CTA loads per stage: 128, or M rounded up to 8 when M is
// smaller (single-CTA kernels); rows of the smem tile beyond them only feed
// output rows that are never stored.
int a_rows_for(const Variant& v, int64_t M) {
    if (v.cg == 2 || M >= hk::kCtaM) return hk::kCtaM;
    return static_cast<int>(std::max<int64_t>(8, ceil_div(M, 8) * 8));
}

// Kernel choice by a small time model. Automatic choice among single-CTA
// kernels (128-row tiles, four widths) for M <= kMaxRowsSingle (bf16; 128 for
// E4M3) and CTA pairs (256-row tiles: 256, or for bf16 128 or 112 wide) for M > 128;
// between the two limits both compete. K is split only when one wave of
// tiles leaves work-unit slots idle and a workspace may be used. Estimated
// time of a candidate (µs):
//   GEMM   = the p-norm (kBoundNorm) of three bounds, so that two bounds near
//            each other cost more than either (their overlap is imperfect):
//              streaming: waves × (bytes one CTA moves per unit ÷ per-SM rate
//                         + pipeline fill); the rate is what the ring keeps in
//                         flight ÷ the load latency, at most a cap (one for
//                         single-CTA kernels, one per SM of a pair); A's bytes
//                         count kABytesWeight (A is shared by every unit of a
//                         row of tiles and comes from L2),
//              HBM:       (A, B, and C or the fp32 partials) ÷ HBM rate,
//              issue:     waves × K stages per unit × the larger of the tensor
//                         time of a stage and the issuing thread's floor per
//                         stage (narrow tiles are bound by the latter);
//   reduce = (split partials, counted twice: the GEMM writes them and the
//            reduction reads them back, + C written) ÷ HBM rate + launch, when
//            K is split (it runs after the GEMM, so its time adds).
// The constants were fitted to warm back-to-back timings of every (kernel,
// split) on 32 shapes from 1×1024×8192 to 2048×2048×8192 (GB300), with the
// tensor time of a K step fixed at its measured value: the choice is within
// 4.5 % of the best measured candidate on each shape, 0.6 % on average.
constexpr int kMaxSplits = 16;
constexpr int kMinKBlocksPerSplit = 8;
constexpr int64_t kMaxRowsSingle = 384;      // bf16: single-CTA kernels up to here
constexpr double kSmBytesPerUs = 106e3;      // one SM's streaming rate cap, single-CTA kernels (bytes/µs)
constexpr double kSmBytesPerUsPair = 75.7e3; // the same per SM of a CTA pair
constexpr double kLoadLatencyUs = 2.07;      // TMA load latency under load
constexpr double kHbmBytesPerUs = 6.01e6;    // HBM rate the streaming kernels reach (bytes/µs)
constexpr double kABytesWeight = 0.365;      // A's bytes (L2-resident, shared by a row of tiles) against B's
constexpr double kKStepUs = 0.27;            // tensor time of a 64-deep K step of a 256-wide tile per SM
constexpr double kIssueFloorUs = 0.206;      // the MMA-issuing thread's minimum per stage (waits, commit)
constexpr double kFillUs = 0.455;            // filling the ring at the start of a unit
constexpr double kLaunchUs = 4.55;           // the reduction: dependent launch, wait for the GEMM, tail
constexpr double kBoundNorm = 7.34;          // exponent of the p-norm that combines the three bounds

double estimate_us(const Variant& v, int64_t M, int64_t N, int64_t K, int64_t slots, int splits) {
    const int64_t tiles = ceil_div(M, v.tile_m) * ceil_div(N, v.tile_n);
    const int64_t units = tiles * splits;
    const double waves = double(ceil_div(units, slots));
    const double kb = double(ceil_div(ceil_div(K, v.k_elems), splits));
    const double elem = v.fp8 ? 1.0 : 2.0;
    const double stage_a = double(a_rows_for(v, M)) * hk::kRowBytes * v.atoms;
    const double stage_b = double(v.tile_n / v.cg) * hk::kRowBytes * v.atoms;
    const double cap = v.cg == 2 ? kSmBytesPerUsPair : kSmBytesPerUs;
    const double sm_rate = std::min(cap, (stage_a + stage_b) * v.stages / kLoadLatencyUs);
    const double t_stream = waves * ((stage_a * kABytesWeight + stage_b) * kb / sm_rate + kFillUs);
    const double n_pad = double(ceil_div(N, v.tile_n) * v.tile_n);
    const double partials = splits > 1 ? 4.0 * splits * M * n_pad : 0.0;
    const double operands = elem * (double(N) * K + double(M) * K);
    const double t_hbm = (operands + (splits > 1 ? partials : 2.0 * M * N)) / kHbmBytesPerUs;
    const double t_mma = waves * kb * std::max(kKStepUs * v.atoms * (double(v.tile_n) / 256.0), kIssueFloorUs);
    const double t_reduce = splits > 1 ? (2.0 * partials + 2.0 * M * N) / kHbmBytesPerUs + kLaunchUs : 0.0;
    const double t_gemm = std::pow(std::pow(t_stream, kBoundNorm) + std::pow(t_hbm, kBoundNorm) +
                                       std::pow(t_mma, kBoundNorm),
                                   1.0 / kBoundNorm);
    return t_gemm + t_reduce;
}

void choose_plan(int64_t M, int64_t N, int64_t K, const DeviceInfo* di, int max_units_cap, bool allow_split,
                 int forced_kernel, int forced_splits, bool fp8, const Variant** out_v, int* out_s) {
    const Variant* best_v = nullptr;
    int best_s = 1;
    double best_t = 0.0;
    for (int i = 0; i < kNumVariants; ++i) {
        const Variant& v = kVariants[i];
        if (v.fp8 != fp8 || v.mx) continue;
        if (a_rows_for(v, M) > v.a_rows_max) continue;   // short A stages serve only M up to their rows
        const bool single_ok = M <= (fp8 ? int64_t(hk::kCtaM) : kMaxRowsSingle);
        const bool pair_ok = M > hk::kCtaM;
        if (forced_kernel != HK_KERNEL_AUTO ? v.id != forced_kernel : !(v.cg == 2 ? pair_ok : single_ok)) continue;
        const int64_t k_blocks = ceil_div(K, v.k_elems);
        int64_t slots = di->max_units[i];
        if (max_units_cap > 0 && max_units_cap < slots) slots = max_units_cap;
        const int64_t tiles = ceil_div(M, v.tile_m) * ceil_div(N, v.tile_n);
        int s_lo = 1, s_hi = 1;
        if (forced_splits > 0) {
            s_lo = s_hi = forced_splits;
        } else if (allow_split && tiles < slots && k_blocks >= 2 * kMinKBlocksPerSplit) {
            s_hi = static_cast<int>(std::min<int64_t>(kMaxSplits, k_blocks / kMinKBlocksPerSplit));
        }
        for (int sp = s_lo; sp <= s_hi; ++sp) {
            const double t = estimate_us(v, M, N, K, slots, sp);
            if (!best_v || t < best_t) {   // on a tie the earlier candidate (fewer splits) stays
                best_v = &v;
                best_s = sp;
                best_t = t;
            }
        }
    }
    *out_v = best_v ? best_v : find_variant(HK_KERNEL_PAIR_256x256, fp8);
    *out_s = best_v ? best_s : 1;
}

hk_status fill_plan(hk_gemm_plan* p, int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb, int64_t ldc,
                    int device, const hk_gemm_config* config, const DeviceInfo* di, bool allow_split,
                    bool fp8 = false, float alpha = 1.0f) {
    p->M = M; p->N = N; p->K = K; p->lda = lda; p->ldb = ldb; p->ldc = ldc;
    p->device = device;
    std::memset(&p->cfg, 0, sizeof p->cfg);
    if (config) p->cfg = *config;
    if (p->cfg.group_m < 0 || p->cfg.max_clusters < 0 || p->cfg.split_k < 0)
        return fail(HK_ERR_INVALID_ARG, "negative config field");
    if (p->cfg.activation > HK_ACT_SILU) return fail(HK_ERR_INVALID_ARG, "unknown activation %u", p->cfg.activation);
    if (p->cfg.input_type != HK_INPUT_BF16 && p->cfg.input_type != HK_INPUT_E4M3)
        return fail(HK_ERR_INVALID_ARG, "unknown input type %d", (int)p->cfg.input_type);
    if (config) {   // a plan's own element type and scale
        fp8 = p->cfg.input_type == HK_INPUT_E4M3;
        if (p->cfg.alpha != 0.0f) alpha = p->cfg.alpha;
        if (!std::isfinite(alpha)) return fail(HK_ERR_INVALID_ARG, "alpha must be finite");
        if (fp8 && ((lda % 16) || (ldb % 16)))
            return fail(HK_ERR_MISALIGNED, "FP8 leading dimensions must be multiples of 16 elements");
    }
    if (p->cfg.kernel != HK_KERNEL_AUTO && !find_variant(p->cfg.kernel, fp8))
        return fail(HK_ERR_INVALID_ARG, "unknown kernel id %d", (int)p->cfg.kernel);
    const int64_t k_blocks_all = ceil_div(K, fp8 ? 128 : hk::kTileK);
    if (p->cfg.split_k > 1 && (p->cfg.split_k > k_blocks_all || p->cfg.split_k > 4096))
        return fail(HK_ERR_INVALID_ARG, "split_k %d exceeds the %lld K blocks of %d", (int)p->cfg.split_k,
                    (long long)k_blocks_all, fp8 ? 128 : hk::kTileK);
    const Variant* v = nullptr;
    int splits = 1;
    choose_plan(M, N, K, di, p->cfg.max_clusters, allow_split, p->cfg.kernel, p->cfg.split_k, fp8, &v, &splits);
    p->variant = v;
    p->sm_count = di->sm_count;
    const int vi = static_cast<int>(v - kVariants);
    const int group_m = p->cfg.group_m > 0 ? p->cfg.group_m : kDefaultGroupM;
    hk::GemmParams& g = p->params;
    std::memset(&g, 0, sizeof g);
    g.M = static_cast<int32_t>(M);
    g.N = static_cast<int32_t>(N);
    g.K = static_cast<int32_t>(K);
    g.tiles_m = static_cast<int32_t>(ceil_div(M, v->tile_m));
    g.tiles_n = static_cast<int32_t>(ceil_div(N, v->tile_n));
    g.k_blocks = static_cast<int32_t>(ceil_div(K, v->k_elems));
    if (splits > 1 && splits > g.k_blocks)   // every split must own at least one K stage
        return fail(HK_ERR_INVALID_ARG, "split_k %d exceeds the %d K stages of %d elements of kernel %s", splits,
                    (int)g.k_blocks, v->k_elems, v->name);
    g.alpha = alpha;
    const int64_t tiles = int64_t(g.tiles_m) * g.tiles_n;
    if (tiles > (int64_t(1) << 30)) return fail(HK_ERR_INVALID_ARG, "too many output tiles");
    g.num_tiles = static_cast<int32_t>(tiles);
    g.splits = splits;
    if (int64_t(splits) * tiles > (int64_t(1) << 30)) return fail(HK_ERR_INVALID_ARG, "too many work units");
    g.a_rows = a_rows_for(*v, M);
    g.expect_bytes = static_cast<uint32_t>(v->cg * (g.a_rows + v->tile_n / v->cg) * hk::kRowBytes * v->atoms);
    g.n_pad = int64_t(g.tiles_n) * v->tile_n;
    p->ws_bytes = splits > 1 ? static_cast<size_t>(splits) * static_cast<size_t>(M) * g.n_pad * 4 : 0;
    g.group_m = group_m;
    g.n_tma = static_cast<int32_t>(N & ~int64_t(7));
    g.ldc = ldc;
    g.flags = p->cfg.flags;
    g.act = static_cast<int32_t>(p->cfg.activation);
    g.timeout_ns = p->cfg.timeout_ns ? p->cfg.timeout_ns : kDefaultTimeoutNs;
    int units = di->max_units[vi];
    if (units <= 0) return fail(HK_ERR_UNSUPPORTED_DEVICE, "kernel %s does not fit on the device", v->name);
    if (p->cfg.max_clusters > 0 && p->cfg.max_clusters < units) units = p->cfg.max_clusters;
    // Last partial round of a pair kernel: when its R tiles fill at most half
    // of the units, each runs as two half-width units (256 x 128), so the
    // round takes about half as long. No workspace is involved.
    g.tail_start = -1;
    g.total_units = g.num_tiles * splits;
    if (v->cg == 2 && v->halves && splits == 1 && g.num_tiles > 0 && !(p->cfg.flags & HK_FLAG_NO_TAIL_SPLIT)) {
        const int64_t rounds = ceil_div(g.num_tiles, units);
        const int64_t last = g.num_tiles - (rounds - 1) * units;
        if (2 * last <= units) {
            g.tail_start = static_cast<int32_t>(g.num_tiles - last);
            g.total_units = static_cast<int32_t>(g.num_tiles + last);
        }
    }
    g.expect_bytes_half = static_cast<uint32_t>(v->cg * (g.a_rows + v->tile_n / v->cg / 2) * hk::kRowBytes * v->atoms);
    if (units > g.total_units) units = g.total_units;
    p->grid_ctas = v->cg * units;
    if (const char* log = std::getenv("HK_LOG"); log && log[0] == '1')
        std::fprintf(stderr, "hk_gemm plan: M=%lld N=%lld K=%lld kernel=%s splits=%d tail_tiles=%d grid=%d ctas "
                     "group_m=%d workspace=%zu B\n", (long long)M, (long long)N, (long long)K, v->name, splits,
                     g.tail_start >= 0 ? g.num_tiles - g.tail_start : 0, p->grid_ctas, group_m, p->ws_bytes);
    return HK_OK;
}

// Encode the four tensor maps of a run (A, B, C and the half-width B or the
// MXFP8 scale blocks) for these pointers.
hk_status encode_maps(const hk_gemm_plan* p, const void* A, const void* B, void* C, const void* mx_scales,
                      size_t mx_scale_bytes, TensorMaps* m) {
    hk_status s = get_encoder();
    if (s != HK_OK) return s;
    CUtensorMap& ta = m->ta;
    CUtensorMap& tb = m->tb;
    CUtensorMap& tc = m->tc;
    // A with K == 0 is never read; give the map a valid 1-column shape over C's memory
    const Variant* v = p->variant;
    const bool bytes = v->fp8;               // FP8 operands: 1-byte elements
    const void* a_ptr = p->K > 0 ? A : C;
    const void* b_ptr = p->K > 0 ? B : C;
    const int64_t kk = p->K > 0 ? p->K : (bytes ? 16 : 8);
    const int64_t lda = p->K > 0 ? p->lda : (bytes ? 2 * p->ldc : p->ldc);
    const int64_t ldb = p->K > 0 ? p->ldb : (bytes ? 2 * p->ldc : p->ldc);
    const uint32_t b_rows = static_cast<uint32_t>(v->tile_n / v->cg);
    const uint32_t a_box_rows = static_cast<uint32_t>(p->params.a_rows);
    const uint32_t box_k = static_cast<uint32_t>(v->k_elems / v->atoms);   // one 128-byte K atom per box
    if ((s = encode_2d(&ta, a_ptr, p->K > 0 ? p->M : 1, kk, lda, box_k, a_box_rows, CU_TENSOR_MAP_SWIZZLE_128B, "A", bytes)) != HK_OK) return s;
    if ((s = encode_2d(&tb, b_ptr, p->K > 0 ? p->N : 1, kk, ldb, box_k, b_rows, CU_TENSOR_MAP_SWIZZLE_128B, "B", bytes)) != HK_OK) return s;
    CUtensorMap& tbh = m->tbh;   // B in boxes of half the rows, for half-width units (MXFP8: the scale blocks)
    if (v->mx && mx_scales != nullptr) {
        // prearranged scale blocks as rows of 256 bytes, one 512-byte block = 2 rows
        if ((s = encode_2d(&tbh, mx_scales, static_cast<int64_t>(mx_scale_bytes / 256), 256, 256, 256, 2,
                           CU_TENSOR_MAP_SWIZZLE_NONE, "MXFP8 scales", true)) != HK_OK)
            return s;
    } else if ((s = encode_2d(&tbh, b_ptr, p->K > 0 ? p->N : 1, kk, ldb, box_k, b_rows / 2, CU_TENSOR_MAP_SWIZZLE_128B, "B", bytes)) != HK_OK) {
        return s;
    }
    // the map covers N rounded down to a multiple of 8 (see the epilogue); at
    // least 8 columns so that it stays valid when N < 8 (then it is unused)
    const int64_t n_tma = p->N & ~int64_t(7);
    if ((s = encode_2d(&tc, C, p->M, n_tma > 0 ? n_tma : 8, p->ldc, hk::kEpiCols, 32, CU_TENSOR_MAP_SWIZZLE_64B, "C")) != HK_OK) return s;
    m->a = A;
    m->b = B;
    m->c = C;
    m->scales = mx_scales;
    m->scale_bytes = mx_scale_bytes;
    m->valid = true;
    return HK_OK;
}

hk_status launch(const hk_gemm_plan* p, StatusWord* sw, const void* A, const void* B, void* C, void* workspace,
                 cudaStream_t stream, const void* bias = nullptr, const void* mx_scales = nullptr,
                 size_t mx_scale_bytes = 0, const void* residual = nullptr, int64_t ldr = 0) {
    if (p->M == 0 || p->N == 0) return HK_OK;
    const Variant* v = p->variant;
    TensorMaps maps;
    {
        std::lock_guard<std::mutex> lock(p->tmap_mutex);
        const TensorMaps& t = p->tmaps;
        if (t.valid && t.a == A && t.b == B && t.c == C && t.scales == mx_scales && t.scale_bytes == mx_scale_bytes)
            maps = t;
    }
    if (!maps.valid) {
        hk_status s = encode_maps(p, A, B, C, mx_scales, mx_scale_bytes, &maps);
        if (s != HK_OK) return s;
        std::lock_guard<std::mutex> lock(p->tmap_mutex);
        p->tmaps = maps;
    }
    const CUtensorMap& ta = maps.ta;
    const CUtensorMap& tb = maps.tb;
    const CUtensorMap& tc = maps.tc;
    const CUtensorMap& tbh = maps.tbh;

    hk::GemmParams g = p->params;
    g.c_ptr = static_cast<uint16_t*>(C);
    g.bias = static_cast<const uint16_t*>(bias);
    g.residual = static_cast<const uint16_t*>(residual);
    g.ldr = ldr;
    g.status = sw->dev;
    g.launch_id = next_launch_id();
    if (g.splits > 1) g.partials = static_cast<float*>(workspace);

    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    int nattr = 0;
    if (v->cg > 1) {
        attr[nattr].id = cudaLaunchAttributeClusterDimension;
        attr[nattr].val.clusterDim.x = static_cast<unsigned>(v->cg);
        attr[nattr].val.clusterDim.y = 1;
        attr[nattr].val.clusterDim.z = 1;
        ++nattr;
    }
    if (HK_PDL || mx_scales != nullptr) {
        // a programmatic dependent of the previous kernel on the stream (for the
        // block-scaled GEMM: of the scale arrangement): its prologue (barriers, TMEM,
        // tensor-map prefetch) overlaps that kernel's last CTAs; the producer and the
        // epilogue wait (griddepcontrol.wait) for that grid before any global access
        attr[nattr].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[nattr].val.programmaticStreamSerializationAllowed = 1;
        ++nattr;
    }
    cfg.gridDim = dim3(p->grid_ctas, 1, 1);
    cfg.blockDim = dim3(hk::kThreads, 1, 1);
    cfg.dynamicSmemBytes = v->smem_bytes;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = nattr;
    cudaError_t e = cudaLaunchKernelEx(&cfg, v->fn, ta, tb, tc, tbh, g);
    if (e != cudaSuccess) return cuda_fail(HK_ERR_LAUNCH, "launching the GEMM kernel", e);
    if (g.splits > 1) {
        // programmatic dependent launch: the reduction is scheduled while the GEMM
        // runs and waits (griddepcontrol.wait) for the GEMM's completion
        const int64_t groups = p->M * ceil_div(p->N, 8);
        const int64_t blocks = std::min<int64_t>(ceil_div(groups, 256), int64_t(p->sm_count) * 8);
        cudaLaunchConfig_t rc = {};
        cudaLaunchAttribute ra[1];
        ra[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        ra[0].val.programmaticStreamSerializationAllowed = 1;
        rc.gridDim = dim3(static_cast<unsigned>(blocks), 1, 1);
        rc.blockDim = dim3(256, 1, 1);
        rc.stream = stream;
        rc.attrs = ra;
        rc.numAttrs = 1;
        e = cudaLaunchKernelEx(&rc, hk::splitk_reduce_kernel, static_cast<const float*>(g.partials), g.splits, g.M,
                               g.N, g.n_pad, g.c_ptr, g.ldc, g.bias, g.act, g.alpha, g.residual, g.ldr);
        if (e != cudaSuccess) return cuda_fail(HK_ERR_LAUNCH, "launching the split-K reduction", e);
    }
    return HK_OK;
}

// Per-device status word of the one-shot entry points, created by the first call on the device.
hk_status context_status(int device, StatusWord** out) {
    std::lock_guard<std::mutex> lock(g_ctx_mutex);
    if (!g_ctx[device]) {
        StatusWord* w = new (std::nothrow) StatusWord();
        if (!w) return fail(HK_ERR_INVALID_ARG, "out of host memory");
        hk_status s = alloc_status(w);
        if (s != HK_OK) {
            delete w;
            return s;
        }
        g_ctx[device] = w;
    }
    *out = g_ctx[device];
    return HK_OK;
}

// ------------------------------------------------- one-shot plan cache --
//
// The one-shot entry points keep the plans they fill (argument checks done,
// kernel, split and schedule chosen by the time model) in a small
// least-recently-used cache keyed by everything that choice depends on; a
// repeated call is then a lookup, and the plan's tensor-map cache makes a
// call with the same pointers encode nothing. Entries are shared pointers:
// a call still running on an evicted plan keeps it alive.
struct OneShotKey {
    int device;
    int fp8;
    uint32_t act;
    uint32_t alpha_bits;
    int64_t M, N, K, lda, ldb, ldc;
    bool operator==(const OneShotKey& o) const {
        return device == o.device && fp8 == o.fp8 && act == o.act && alpha_bits == o.alpha_bits && M == o.M &&
               N == o.N && K == o.K && lda == o.lda && ldb == o.ldb && ldc == o.ldc;
    }
};

constexpr int kOneShotCacheSize = 32;

struct OneShotEntry {
    OneShotKey key;
    std::shared_ptr<hk_gemm_plan> plan;
    uint64_t last_use = 0;
};

std::mutex g_oneshot_mutex;
OneShotEntry g_oneshot[kOneShotCacheSize];
uint64_t g_oneshot_clock = 0;

hk_status one_shot_plan(int device, const DeviceInfo* di, int64_t M, int64_t N, int64_t K, int64_t lda,
                        int64_t ldb, int64_t ldc, bool fp8, uint32_t act, float alpha,
                        std::shared_ptr<hk_gemm_plan>* out) {
    OneShotKey key{device, fp8 ? 1 : 0, act, 0u, M, N, K, lda, ldb, ldc};
    std::memcpy(&key.alpha_bits, &alpha, sizeof alpha);
    {
        std::lock_guard<std::mutex> lock(g_oneshot_mutex);
        for (OneShotEntry& e : g_oneshot)
            if (e.plan && e.key == key) {
                e.last_use = ++g_oneshot_clock;
                *out = e.plan;
                return HK_OK;
            }
    }
    std::shared_ptr<hk_gemm_plan> p(new (std::nothrow) hk_gemm_plan());
    if (!p) return fail(HK_ERR_INVALID_ARG, "out of host memory");
    hk_gemm_config cfg;
    std::memset(&cfg, 0, sizeof cfg);
    cfg.activation = act;
    cfg.input_type = fp8 ? HK_INPUT_E4M3 : HK_INPUT_BF16;   // cfg.alpha stays 0: `alpha` below is used
    hk_status s = fill_plan(p.get(), M, N, K, lda, ldb, ldc, device, &cfg, di, false, fp8, alpha);
    if (s != HK_OK) return s;
    p->owns_status = false;
    std::lock_guard<std::mutex> lock(g_oneshot_mutex);
    OneShotEntry* victim = &g_oneshot[0];
    for (OneShotEntry& e : g_oneshot) {
        if (!e.plan) {
            victim = &e;
            break;
        }
        if (e.last_use < victim->last_use) victim = &e;
    }
    victim->key = key;
    victim->plan = p;
    victim->last_use = ++g_oneshot_clock;
    *out = p;
    return HK_OK;
}

// Device address of hk_gemm_bf16_noalloc's fixed array per device (looked
// up by its first call on the device); its first bytes are that entry
// point's status word.
std::mutex g_noalloc_mutex;
unsigned char* g_noalloc_ptr[kMaxDevices] = {};

// Status word of hk_gemm_bf16_noalloc's calls on `device`, or null when that
// entry point has not run there.
uint32_t* noalloc_status_word(int device) {
    std::lock_guard<std::mutex> lock(g_noalloc_mutex);
    return reinterpret_cast<uint32_t*>(g_noalloc_ptr[device]);
}

}  // namespace

namespace hk_host {

hk_status set_error(hk_status s, const char* msg) {
    g_last_error = msg;
    return s;
}

hk_status status_word(int device, uint32_t** out) {
    if (device < 0 || device >= kMaxDevices) return fail(HK_ERR_INVALID_ARG, "device %d out of range", device);
    StatusWord* w = nullptr;
    hk_status s = context_status(device, &w);
    if (s != HK_OK) return s;
    *out = w->dev;
    return HK_OK;
}

hk_status check_device(int device, int* sm_count) {
    const DeviceInfo* di = nullptr;
    hk_status s = device_info(device, &di);
    if (s != HK_OK) return s;
    *sm_count = di->sm_count;
    return HK_OK;
}

hk_status tensor_map_encoder(PFN_cuTensorMapEncodeTiled_v12000* out) {
    hk_status s = get_encoder();
    if (s != HK_OK) return s;
    *out = g_encode;
    return HK_OK;
}

uint32_t next_launch_id() { return ::next_launch_id(); }

}  // namespace hk_host

extern "C" {

const char* hk_status_string(hk_status s) {
    switch (s) {
        case HK_OK: return "HK_OK";
        case HK_ERR_INVALID_ARG: return "HK_ERR_INVALID_ARG: invalid size, leading dimension or pointer";
        case HK_ERR_MISALIGNED: return "HK_ERR_MISALIGNED: pointer not 16-byte aligned or leading dimension not a multiple of 8";
        case HK_ERR_UNSUPPORTED_DEVICE: return "HK_ERR_UNSUPPORTED_DEVICE: not a compute capability 10.3 GPU";
        case HK_ERR_LAUNCH: return "HK_ERR_LAUNCH: kernel launch failed";
        case HK_ERR_TIMEOUT: return "HK_ERR_TIMEOUT: a bounded wait in the kernel ran out";
        case HK_ERR_WORKSPACE: return "HK_ERR_WORKSPACE: workspace missing, too small or misaligned";
        case HK_ERR_CUDA: return "HK_ERR_CUDA: CUDA runtime error";
    }
    return "unknown hk_status";
}

const char* hk_gemm_last_error_string(void) { return g_last_error.c_str(); }

hk_status hk_gemm_plan_create(hk_gemm_plan** out, int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb,
                              int64_t ldc, int device, const hk_gemm_config* config) {
    if (!out) return fail(HK_ERR_INVALID_ARG, "out is NULL");
    *out = nullptr;
    hk_status s = check_shape(M, N, K, lda, ldb, ldc);
    if (s != HK_OK) return s;
    const DeviceInfo* di = nullptr;
    if ((s = device_info(device, &di)) != HK_OK) return s;
    hk_gemm_plan* p = new (std::nothrow) hk_gemm_plan();
    if (!p) return fail(HK_ERR_INVALID_ARG, "out of host memory");
    if ((s = fill_plan(p, M, N, K, lda, ldb, ldc, device, config, di, true)) != HK_OK) {
        delete p;
        return s;
    }
    {
        DeviceGuard guard(device);
        if ((s = alloc_status(&p->status)) != HK_OK) {
            delete p;
            return s;
        }
    }
    p->owns_status = true;
    *out = p;
    return HK_OK;
}

size_t hk_gemm_plan_workspace_size(const hk_gemm_plan* plan) { return plan ? plan->ws_bytes : 0; }

hk_status hk_gemm_plan_get_info(const hk_gemm_plan* p, hk_gemm_plan_info* info) {
    if (!p || !info) return fail(HK_ERR_INVALID_ARG, "NULL plan or info");
    std::memset(info, 0, sizeof *info);
    info->M = p->M; info->N = p->N; info->K = p->K;
    info->tile_m = p->variant->tile_m; info->tile_n = p->variant->tile_n; info->tile_k = p->variant->k_elems;
    info->stages = p->variant->stages;
    info->kernel = p->variant->id;
    info->ctas_per_unit = p->variant->cg;
    info->num_tiles = p->params.num_tiles;
    info->grid_ctas = (p->M == 0 || p->N == 0) ? 0 : p->grid_ctas;
    info->group_m = p->params.group_m;
    info->split_k = p->params.splits;
    info->kernels_per_run = (p->M == 0 || p->N == 0) ? 0 : (p->params.splits > 1 ? 2 : 1);
    info->smem_bytes = p->variant->smem_bytes;
    info->workspace_bytes = p->ws_bytes;
    info->tail_split_tiles = p->params.tail_start >= 0 ? p->params.num_tiles - p->params.tail_start : 0;
    return HK_OK;
}

hk_status hk_gemm_plan_run(const hk_gemm_plan* p, const void* A, const void* B, void* C, void* workspace,
                           size_t workspace_bytes, void* stream) {
    if (!p) return fail(HK_ERR_INVALID_ARG, "NULL plan");
    if (p->M == 0 || p->N == 0) return HK_OK;
    hk_status s = check_pointers(A, B, C, p->K);
    if (s != HK_OK) return s;
    if (p->ws_bytes > 0) {
        if (!workspace || workspace_bytes < p->ws_bytes)
            return fail(HK_ERR_WORKSPACE, "the plan needs %zu bytes of workspace, %zu given", p->ws_bytes,
                        workspace ? workspace_bytes : size_t(0));
        if (reinterpret_cast<uintptr_t>(workspace) & 255u)
            return fail(HK_ERR_WORKSPACE, "the workspace must be 256-byte aligned");
    }
    DeviceGuard guard(p->device);
    return launch(p, const_cast<StatusWord*>(&p->status), A, B, C, workspace, static_cast<cudaStream_t>(stream));
}

hk_status hk_gemm_plan_device_status(hk_gemm_plan* p) {
    if (!p) return fail(HK_ERR_INVALID_ARG, "NULL plan");
    return read_status(&p->status, p->device);
}

void hk_gemm_plan_destroy(hk_gemm_plan* p) {
    if (!p) return;
    if (p->owns_status && p->status.dev) {
        DeviceGuard guard(p->device);
        cudaFree(p->status.dev);
    }
    delete p;
}

hk_status hk_gemm_bf16(const void* A, const void* B, void* C, int64_t M, int64_t N, int64_t K, int64_t lda,
                       int64_t ldb, int64_t ldc, void* stream) {
    hk_status s = check_shape(M, N, K, lda, ldb, ldc);
    if (s != HK_OK) return s;
    if (M == 0 || N == 0) return HK_OK;
    if ((s = check_pointers(A, B, C, K)) != HK_OK) return s;
    int device = 0;
    cudaError_t e = cudaGetDevice(&device);
    if (e != cudaSuccess) return cuda_fail(HK_ERR_CUDA, "cudaGetDevice", e);
    const DeviceInfo* di = nullptr;
    if ((s = device_info(device, &di)) != HK_OK) return s;
    StatusWord* sw = nullptr;
    if ((s = context_status(device, &sw)) != HK_OK) return s;
    std::shared_ptr<hk_gemm_plan> plan;
    if ((s = one_shot_plan(device, di, M, N, K, lda, ldb, ldc, false, 0u, 1.0f, &plan)) != HK_OK) return s;
    return launch(plan.get(), sw, A, B, C, nullptr, static_cast<cudaStream_t>(stream));
}

hk_status hk_gemm_last_device_status(int device) {
    if (device < 0 || device >= kMaxDevices) return fail(HK_ERR_INVALID_ARG, "device %d out of range", device);
    StatusWord* sw = nullptr;
    {
        std::lock_guard<std::mutex> lock(g_ctx_mutex);
        sw = g_ctx[device];
    }
    hk_status s = sw ? read_status(sw, device) : HK_OK;
    // the calls of hk_gemm_bf16_noalloc keep their status word in the library's fixed array
    StatusWord fixed;
    fixed.dev = noalloc_status_word(device);
    if (fixed.dev) {
        const hk_status s2 = read_status(&fixed, device);   // read and cleared with no allocation
        if (s == HK_OK) s = s2;
    }
    return s;
}

hk_status hk_gemm_plan_run_epilogue(const hk_gemm_plan* p, const void* A, const void* B, void* C, const void* bias,
                                    void* workspace, size_t workspace_bytes, void* stream) {
    return hk_gemm_plan_run_fused(p, A, B, C, bias, nullptr, 0, workspace, workspace_bytes, stream);
}

hk_status hk_gemm_plan_run_fused(const hk_gemm_plan* p, const void* A, const void* B, void* C, const void* bias,
                                 const void* R, int64_t ldr, void* workspace, size_t workspace_bytes, void* stream) {
    if (!p) return fail(HK_ERR_INVALID_ARG, "NULL plan");
    if (p->M == 0 || p->N == 0) return HK_OK;
    hk_status s = check_pointers(A, B, C, p->K);
    if (s != HK_OK) return s;
    if (bias && (reinterpret_cast<uintptr_t>(bias) & 15u))
        return fail(HK_ERR_MISALIGNED, "the bias vector must be 16-byte aligned");
    if ((s = check_residual(R, ldr, C, p->M, p->N, p->ldc)) != HK_OK) return s;
    if (p->ws_bytes > 0) {
        if (!workspace || workspace_bytes < p->ws_bytes)
            return fail(HK_ERR_WORKSPACE, "the plan needs %zu bytes of workspace, %zu given", p->ws_bytes,
                        workspace ? workspace_bytes : size_t(0));
        if (reinterpret_cast<uintptr_t>(workspace) & 255u)
            return fail(HK_ERR_WORKSPACE, "the workspace must be 256-byte aligned");
    }
    DeviceGuard guard(p->device);
    return launch(p, const_cast<StatusWord*>(&p->status), A, B, C, workspace, static_cast<cudaStream_t>(stream),
                  bias, nullptr, 0, R, ldr);
}

hk_status hk_gemm_bf16_epilogue(const void* A, const void* B, void* C, const void* bias, int64_t M, int64_t N,
                                int64_t K, int64_t lda, int64_t ldb, int64_t ldc, int32_t activation, void* stream) {
    return hk_gemm_bf16_fused(A, B, C, bias, nullptr, M, N, K, lda, ldb, ldc, 0, activation, stream);
}

hk_status hk_gemm_bf16_fused(const void* A, const void* B, void* C, const void* bias, const void* R, int64_t M,
                             int64_t N, int64_t K, int64_t lda, int64_t ldb, int64_t ldc, int64_t ldr,
                             int32_t activation, void* stream) {
    hk_status s = check_shape(M, N, K, lda, ldb, ldc);
    if (s != HK_OK) return s;
    if (activation < 0 || activation > HK_ACT_SILU) return fail(HK_ERR_INVALID_ARG, "unknown activation %d", (int)activation);
    if (M == 0 || N == 0) return HK_OK;
    if ((s = check_pointers(A, B, C, K)) != HK_OK) return s;
    if (bias && (reinterpret_cast<uintptr_t>(bias) & 15u))
        return fail(HK_ERR_MISALIGNED, "the bias vector must be 16-byte aligned");
    if ((s = check_residual(R, ldr, C, M, N, ldc)) != HK_OK) return s;
    int device = 0;
    cudaError_t e = cudaGetDevice(&device);
    if (e != cudaSuccess) return cuda_fail(HK_ERR_CUDA, "cudaGetDevice", e);
    const DeviceInfo* di = nullptr;
    if ((s = device_info(device, &di)) != HK_OK) return s;
    StatusWord* sw = nullptr;
    if ((s = context_status(device, &sw)) != HK_OK) return s;
    std::shared_ptr<hk_gemm_plan> plan;
    if ((s = one_shot_plan(device, di, M, N, K, lda, ldb, ldc, false, static_cast<uint32_t>(activation), 1.0f,
                           &plan)) != HK_OK)
        return s;
    return launch(plan.get(), sw, A, B, C, nullptr, static_cast<cudaStream_t>(stream), bias, nullptr, 0, R, ldr);
}

hk_status hk_gemm_fp8_e4m3(const void* A, const void* B, void* C, int64_t M, int64_t N, int64_t K, int64_t lda,
                           int64_t ldb, int64_t ldc, float scale_a, float scale_b, void* stream) {
    // bf16 rules for C; for the 1-byte operands the TMA stride rule asks for
    // leading dimensions that are multiples of 16 elements
    hk_status s = check_shape(M, N, K, lda, ldb, ldc);
    if (s != HK_OK) return s;
    if ((lda % 16) || (ldb % 16))
        return fail(HK_ERR_MISALIGNED, "FP8 leading dimensions must be multiples of 16 elements (lda=%lld ldb=%lld)",
                    (long long)lda, (long long)ldb);
    if (!std::isfinite(scale_a) || !std::isfinite(scale_b))
        return fail(HK_ERR_INVALID_ARG, "FP8 scales must be finite");
    if (M == 0 || N == 0) return HK_OK;
    if ((s = check_pointers(A, B, C, K)) != HK_OK) return s;
    int device = 0;
    cudaError_t e = cudaGetDevice(&device);
    if (e != cudaSuccess) return cuda_fail(HK_ERR_CUDA, "cudaGetDevice", e);
    const DeviceInfo* di = nullptr;
    if ((s = device_info(device, &di)) != HK_OK) return s;
    StatusWord* sw = nullptr;
    if ((s = context_status(device, &sw)) != HK_OK) return s;
    const float alpha = static_cast<float>(static_cast<double>(scale_a) * static_cast<double>(scale_b));
    std::shared_ptr<hk_gemm_plan> plan;
    if ((s = one_shot_plan(device, di, M, N, K, lda, ldb, ldc, true, 0u, alpha, &plan)) != HK_OK) return s;
    return launch(plan.get(), sw, A, B, C, nullptr, static_cast<cudaStream_t>(stream));
}

// ---------------------------------------------------------------- MXFP8 --

namespace {

struct MxLayout {
    int64_t tiles_m, tiles_n, k_blocks;
    int tile_n;   // N of the tile the kernel for this M uses
    size_t a_bytes, b_offset, total;
};

// A scale blocks per 128-row group (a pair tile covers two groups, so their
// count is rounded up to even when the pair kernel runs: M > 128).
MxLayout mx_layout(int64_t M, int64_t N, int64_t K) {
    MxLayout l;
    l.tiles_m = M <= hk::kCtaM ? 1 : 2 * ceil_div(M, 2 * hk::kCtaM);
    l.tile_n = M <= hk::kCtaM ? kMxTileNSingle : kMxTileNPair;
    l.tiles_n = ceil_div(N, l.tile_n);
    // K blocks of 128: the pair kernel loads HK_MX_PAIR_ATOMS of them per stage, so
    // their count is rounded up to that multiple (the extra blocks hold scale 0)
    l.k_blocks = ceil_div(K, 128);
    if (M > hk::kCtaM) l.k_blocks = ceil_div(l.k_blocks, HK_MX_PAIR_ATOMS) * HK_MX_PAIR_ATOMS;
    l.a_bytes = static_cast<size_t>(l.tiles_m * l.k_blocks * 512);
    l.b_offset = (l.a_bytes + 255) & ~size_t(255);
    l.total = l.b_offset + static_cast<size_t>(l.tiles_n * l.k_blocks * 512 * kMxSfbAtoms);
    return l;
}

}  // namespace

size_t hk_gemm_mxfp8_workspace_size(int64_t M, int64_t N, int64_t K) {
    if (M <= 0 || N <= 0 || K <= 0) return 0;
    return mx_layout(M, N, K).total;
}

hk_status hk_gemm_mxfp8_ex(const void* A, const void* B, const void* SFA, const void* SFB, void* C, int64_t M,
                           int64_t N, int64_t K, int64_t lda, int64_t ldb, int64_t ldsfa, int64_t ldsfb, int64_t ldc,
                           void* workspace, size_t workspace_bytes, uint32_t flags, uint64_t timeout_ns,
                           void* stream) {
    if (flags & ~HK_FLAG_FAULT_DROP_ARRIVE) return fail(HK_ERR_INVALID_ARG, "unknown MXFP8 flags 0x%x", flags);
    hk_status s = check_shape(M, N, K, lda, ldb, ldc);
    if (s != HK_OK) return s;
    if (K % 32) return fail(HK_ERR_INVALID_ARG, "K=%lld is not a multiple of the scale block 32", (long long)K);
    if ((lda % 16) || (ldb % 16))
        return fail(HK_ERR_MISALIGNED, "FP8 leading dimensions must be multiples of 16 elements (lda=%lld ldb=%lld)",
                    (long long)lda, (long long)ldb);
    if (K > 0 && (ldsfa < K / 32 || ldsfb < K / 32))
        return fail(HK_ERR_INVALID_ARG, "scale leading dimensions must be at least K/32 (ldsfa=%lld ldsfb=%lld)",
                    (long long)ldsfa, (long long)ldsfb);
    if (M == 0 || N == 0) return HK_OK;
    if ((s = check_pointers(A, B, C, K)) != HK_OK) return s;
    if (K > 0 && (!SFA || !SFB)) return fail(HK_ERR_INVALID_ARG, "null scale pointer");
    const MxLayout lay = mx_layout(M, N, K);
    if (K > 0) {
        if (!workspace || workspace_bytes < lay.total)
            return fail(HK_ERR_WORKSPACE, "MXFP8 workspace of %zu bytes needed (got %zu)", lay.total, workspace_bytes);
        if (reinterpret_cast<uintptr_t>(workspace) & 255u)
            return fail(HK_ERR_WORKSPACE, "MXFP8 workspace must be 256-byte aligned");
    }
    int device = 0;
    cudaError_t e = cudaGetDevice(&device);
    if (e != cudaSuccess) return cuda_fail(HK_ERR_CUDA, "cudaGetDevice", e);
    const DeviceInfo* di = nullptr;
    if ((s = device_info(device, &di)) != HK_OK) return s;
    uint32_t* status = nullptr;
    if ((s = hk_host::status_word(device, &status)) != HK_OK) return s;
    StatusWord sw{status};
    // one CTA with 128x192 tiles for M <= 128, else CTA pairs with 256x256 tiles
    const bool pair = M > hk::kCtaM;
    const Variant* v = find_variant(pair ? HK_KERNEL_PAIR_256x256 : HK_KERNEL_SINGLE_128x192, true, true);
    if (v == nullptr || v->tile_n != lay.tile_n)
        return fail(HK_ERR_INVALID_ARG, "no MXFP8 kernel with the %d-column tiles of the scale layout", lay.tile_n);
    const int vi = static_cast<int>(v - kVariants);
    int units = di->max_units[vi];
    if (units <= 0) return fail(HK_ERR_UNSUPPORTED_DEVICE, "kernel %s does not fit on the device", v->name);
    hk_gemm_plan plan;
    plan.M = M; plan.N = N; plan.K = K; plan.lda = lda; plan.ldb = ldb; plan.ldc = ldc;
    plan.device = device;
    std::memset(&plan.cfg, 0, sizeof plan.cfg);
    plan.variant = v;
    plan.sm_count = di->sm_count;
    plan.ws_bytes = 0;
    plan.owns_status = false;
    hk::GemmParams& g = plan.params;
    std::memset(&g, 0, sizeof g);
    g.M = static_cast<int32_t>(M);
    g.N = static_cast<int32_t>(N);
    g.K = static_cast<int32_t>(K);
    g.tiles_m = static_cast<int32_t>(ceil_div(M, v->tile_m));
    g.tiles_n = static_cast<int32_t>(ceil_div(N, v->tile_n));
    g.k_blocks = static_cast<int32_t>(ceil_div(K, v->k_elems));
    g.alpha = 1.0f;
    const int64_t tiles = int64_t(g.tiles_m) * g.tiles_n;
    if (tiles > (int64_t(1) << 30)) return fail(HK_ERR_INVALID_ARG, "too many output tiles");
    g.num_tiles = static_cast<int32_t>(tiles);
    g.splits = 1;
    g.group_m = kDefaultGroupM;
    g.a_rows = a_rows_for(*v, M);
    // operand bytes of a stage (the scale blocks complete on their own barriers)
    g.expect_bytes = static_cast<uint32_t>(v->cg * (g.a_rows + v->tile_n / v->cg) * hk::kRowBytes * v->atoms);
    g.sf_k_blocks = static_cast<int32_t>(lay.k_blocks);
    g.n_pad = int64_t(g.tiles_n) * v->tile_n;
    g.n_tma = static_cast<int32_t>(N & ~int64_t(7));
    g.ldc = ldc;
    g.flags = flags;
    g.timeout_ns = timeout_ns ? timeout_ns : kDefaultTimeoutNs;
    g.tail_start = -1;
    g.total_units = g.num_tiles;
    if (units > g.total_units) units = g.total_units;
    plan.grid_ctas = v->cg * units;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (K > 0) {
        uint8_t* ws = static_cast<uint8_t*>(workspace);
        g.sf_b_row = static_cast<int64_t>(lay.b_offset / 256);
        const int64_t atoms = (lay.tiles_m + lay.tiles_n) * lay.k_blocks;
        const int64_t blocks = std::min<int64_t>(atoms, int64_t(di->sm_count) * 32);
        const bool words = (K % 128) == 0 && (ldsfa % 4) == 0 && (ldsfb % 4) == 0 &&
                           (reinterpret_cast<uintptr_t>(SFA) & 3u) == 0 && (reinterpret_cast<uintptr_t>(SFB) & 3u) == 0;
        hk::mx_scale_blocks_kernel<<<static_cast<unsigned>(blocks), 32 * kMxSfbAtoms, 0, st>>>(
            static_cast<const uint8_t*>(SFA), ldsfa, static_cast<const uint8_t*>(SFB), ldsfb, static_cast<int>(M),
            static_cast<int>(N), static_cast<int>(K / 32), static_cast<int>(lay.tiles_m), static_cast<int>(lay.tiles_n),
            static_cast<int>(lay.k_blocks), lay.tile_n, kMxSfbAtoms, words ? 1 : 0, ws, ws + lay.b_offset);
        e = cudaGetLastError();
        if (e != cudaSuccess) return cuda_fail(HK_ERR_LAUNCH, "launching the MXFP8 scale arrangement", e);
    }
    return launch(&plan, &sw, A, B, C, nullptr, st, nullptr, K > 0 ? workspace : nullptr, lay.total);
}

hk_status hk_gemm_mxfp8(const void* A, const void* B, const void* SFA, const void* SFB, void* C, int64_t M,
                        int64_t N, int64_t K, int64_t lda, int64_t ldb, int64_t ldsfa, int64_t ldsfb, int64_t ldc,
                        void* workspace, size_t workspace_bytes, void* stream) {
    return hk_gemm_mxfp8_ex(A, B, SFA, SFB, C, M, N, K, lda, ldb, ldsfa, ldsfb, ldc, workspace, workspace_bytes, 0u,
                            0u, stream);
}

// ------------------------------------------------- no-allocation variant --
//
// Some callers cannot allocate device memory when they call a GEMM: code
// running inside a memory pool or arena that owns every byte of the device,
// allocator or runtime hooks that must not re-enter cudaMalloc, or services
// that pre-plan all of their memory at start-up. hk_gemm_bf16_noalloc serves
// them: its K-split scratch (fp32 partial products) and its status word live
// in the fixed array below, which is part of the library's device image and
// stays resident on every device that loads the library until the process
// exits. The array is shared by all calls on a device and keeps whatever the
// last call left in it; nothing in it has to start at zero (each call writes
// every partial it reads, and the kernel recognises its own abort flag by a
// launch id that is unique in the process). Calls that overlap on the GPU
// (different streams, or different host threads without ordering) use the
// same array at the same time and race.

constexpr size_t kNoAllocStatusBytes = 256;                   // status word, padded to keep the partials aligned
constexpr size_t kNoAllocScratchBytes = size_t(32) << 20;     // 32 MiB of K-split partials

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocStatusBytes + kNoAllocScratchBytes];

namespace {

// Device address of the fixed array on `device` (the current device). Looked
// up once per device; the host-side symbol itself is not a device address.
// The look-up is set-up work that a stream capture does not allow, so a first
// call on a device made while `stream` captures is refused with a clear error.
hk_status noalloc_scratch(int device, cudaStream_t stream, unsigned char** out) {
    std::lock_guard<std::mutex> lock(g_noalloc_mutex);
    if (!g_noalloc_ptr[device]) {
        cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
        if (cudaStreamIsCapturing(stream, &cs) == cudaSuccess && cs != cudaStreamCaptureStatusNone)
            return fail(HK_ERR_INVALID_ARG,
                        "the first hk_gemm_bf16_noalloc call on device %d looks up its fixed scratch array and must "
                        "come before any stream capture", device);
        void* ptr = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
        if (e != cudaSuccess) return cuda_fail(HK_ERR_CUDA, "looking up the fixed scratch array", e);
        g_noalloc_ptr[device] = static_cast<unsigned char*>(ptr);
    }
    *out = g_noalloc_ptr[device];
    return HK_OK;
}

}  // namespace

hk_status hk_gemm_bf16_noalloc(const void* A, const void* B, void* C, int64_t M, int64_t N, int64_t K,
                               int64_t lda, int64_t ldb, int64_t ldc, int32_t split_k, void* stream) {
    hk_status s = check_shape(M, N, K, lda, ldb, ldc);
    if (s != HK_OK) return s;
    if (split_k < 0) return fail(HK_ERR_INVALID_ARG, "split_k must be >= 0");
    if (M == 0 || N == 0) return HK_OK;
    if ((s = check_pointers(A, B, C, K)) != HK_OK) return s;
    int device = 0;
    cudaError_t e = cudaGetDevice(&device);
    if (e != cudaSuccess) return cuda_fail(HK_ERR_CUDA, "cudaGetDevice", e);
    const DeviceInfo* di = nullptr;
    if ((s = device_info(device, &di)) != HK_OK) return s;
    unsigned char* scratch = nullptr;
    if ((s = noalloc_scratch(device, static_cast<cudaStream_t>(stream), &scratch)) != HK_OK) return s;

    hk_gemm_config cfg;
    std::memset(&cfg, 0, sizeof cfg);
    cfg.split_k = split_k;
    hk_gemm_plan plan;
    if ((s = fill_plan(&plan, M, N, K, lda, ldb, ldc, device, &cfg, di, true)) != HK_OK) return s;
    if (plan.ws_bytes > kNoAllocScratchBytes) {
        if (split_k > 0)
            return fail(HK_ERR_WORKSPACE,
                        "split_k=%d needs %zu bytes of scratch; the fixed scratch array holds %zu bytes",
                        (int)split_k, plan.ws_bytes, kNoAllocScratchBytes);
        cfg.split_k = 1;   // the automatic split does not fit: run without splitting K
        if ((s = fill_plan(&plan, M, N, K, lda, ldb, ldc, device, &cfg, di, true)) != HK_OK) return s;
    }
    plan.owns_status = false;
    StatusWord sw;
    sw.dev = reinterpret_cast<uint32_t*>(scratch);
    return launch(&plan, &sw, A, B, C, scratch + kNoAllocStatusBytes, static_cast<cudaStream_t>(stream));
}

}  // extern "C"
