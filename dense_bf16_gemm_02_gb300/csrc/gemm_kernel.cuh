// Persistent, warp-specialised BF16 GEMM  C = A · Bᵀ  for sm_103a.
//
// One template, two shapes of work unit: a CTA pair (cta_group::2, output
// tile 256 × kTileN) for general shapes, and a single CTA (cta_group::1,
// output tile 128 × kTileN) for problems with at most 128 rows, where a pair
// would leave half of its tensor cores and half of its SMs idle.
//
// The operation and its 256×256 output tile with a 64-wide K step follow the
// HipKittens "L2" detail page (§3 "Target operation" and "Launch config";
// §9.2 GEMM hot loop). Everything else is a Blackwell design rather than the
// pages' AMD one:
//
//  * a cluster of two CTAs (a "pair") owns one 256×256 output tile at a
//    time; each CTA loads 128 rows of A and 128 rows of B per K step with a
//    TMA bulk-tensor copy (128-byte swizzle) into a STAGES-deep shared-memory
//    ring guarded by full/empty mbarriers (the pages' 2-deep LDS double
//    buffer, §4 "Design space": pipeline depth);
//  * one thread of the pair's leader CTA issues tcgen05.mma.cta_group::2
//    (M=256, N=256, K=16) that reads both CTAs' shared memory and
//    accumulates in fp32 in Tensor Memory, two 256-column accumulators per
//    CTA so the epilogue of tile i overlaps the main loop of tile i+1;
//  * roles are warp-specialised (warp 0: TMA producer, warp 1: TMEM
//    allocation and MMA issue, warps 2-5: epilogue, warp 6: block-scaled
//    FP8 only, copies each stage's scales into TMEM) — on Blackwell a
//    producer warp costs the MMA no registers, unlike the static register
//    split that makes the pages reject producer waves (§5 Tab. 2);
//  * the grid is persistent (one pair per two SMs) and walks output tiles in
//    grouped order (GROUP_M tile rows at a time), the counterpart of the
//    pages' cache-aware block remapping (§2 Q2 Pillar 3, §5 Tab. 4);
//  * the epilogue reads TMEM with tcgen05.ld, rounds to bf16 (RNE), stages
//    32×32 sub-tiles in shared memory and writes them with TMA stores.
//
// Every mbarrier wait is bounded: when one runs out the kernel records an
// error code in a device status word, every role drains, TMEM is freed and
// the kernel returns normally.
#pragma once

#include <cuda.h>
#include <cstdint>

#include "ptx.cuh"

namespace hk {

constexpr int kCtaM = 128;           // rows of C (and of A) per CTA
constexpr int kRowBytes = 128;       // bytes of K per stage and row: one 128-byte swizzle row
constexpr int kTileK = 64;           // bf16 elements of K per stage (FP8: 128)
constexpr int kMmaKBytes = 32;       // bytes of K per tcgen05.mma (bf16 K=16, FP8 K=32)
constexpr int kABytes = kCtaM * kRowBytes;         // 16 KiB of A per stage per CTA
constexpr int kEpiCols = 32;                        // columns per epilogue store
constexpr int kEpiWarps = 4;
constexpr int kEpiBufBytes = 32 * kEpiCols * 2;     // 32 rows × 64 B
constexpr int kThreads = 96 + 32 * kEpiWarps;       // 224: producer, MMA, epilogue, MXFP8 scale copier
constexpr int kSmemLimit = 232448;                  // dynamic shared memory per CTA on sm_103

constexpr int pow2_at_least(int x) {
    int r = 32;
    while (r < x) r <<= 1;
    return r;
}

// Operand stages of `stage_bytes` that fit in `avail` bytes beside a ring of
// (stages + ahead) scale slots of `sf_bytes` (no ring when sf_bytes is 0).
constexpr int stages_fit(int avail, int stage_bytes, int sf_bytes, int ahead, int max_stages) {
    const int s = (avail - ahead * sf_bytes) / (stage_bytes + sf_bytes);
    return s > max_stages ? max_stages : s;
}

// Compile-time geometry of one kernel instance. kMx: block-scaled FP8
// (MXFP8, one UE8M0 scale per 32 K elements). kARows < 128 (single CTA,
// M <= kARows): each stage keeps room for kARows rows of A instead of 128, so
// more stages fit and more of B is in flight; the MMA still reads a 128-row A
// tile, whose rows past kARows fall on other (in-bounds) shared memory and
// only feed rows of C that are never stored. kAtoms: 128-byte swizzle atoms
// of K per stage (each operand's stage is kAtoms tiles of rows × 128 bytes,
// one TMA box each). Two atoms halve the mbarrier wait and the commit per
// MMA of the single issuing thread, whose per-stage barrier work otherwise
// outlasts the tensor core's queue of issued MMAs; the ring then holds
// fewer, larger stages (the same bytes in flight).
template <int kCG, int kTileN_, bool kFp8 = false, bool kMx = false, int kARows = kCtaM, int kAtoms = 1>
struct Geometry {
    static_assert(kCG == 1 || kCG == 2, "one CTA or a CTA pair");
    static_assert(!kMx || kFp8, "block scales come with FP8 operands");
    static_assert(kARows == kCtaM || (kCG == 1 && !kMx && kARows % 8 == 0 && kARows >= 8),
                  "short A stages: single-CTA kernels only, whole 8-row swizzle atoms");
    static_assert(kAtoms == 1 || (kAtoms == 2 && kARows == kCtaM), "two K atoms per stage: 128-row A stages");
    static constexpr int kKAtoms = kAtoms;
    static constexpr int kARowsMax = kARows;                          // rows of A a stage holds
    static constexpr int kAAtomBytes = kARowsMax * kRowBytes;         // one K atom of A
    static constexpr int kAStageBytes = kAAtomBytes * kAtoms;
    static_assert(kTileN_ % 16 == 0 && kTileN_ >= 32 && kTileN_ <= 256, "MMA N");
    static constexpr int kTileM = kCtaM * kCG;              // rows of C per tile
    static constexpr int kTileN = kTileN_;                  // columns of C per tile (MMA N)
    static constexpr int kBRows = kTileN / kCG;             // rows of B each CTA loads per stage
    static_assert(kBRows % 8 == 0, "B rows fill whole 8-row swizzle atoms");
    // Half-width units (the tail split) need a valid MMA N of kTileN / 2 and
    // whole swizzle atoms of B in each CTA's half: not so for a 112-wide pair.
    static constexpr bool kHalves = kTileN % (16 * kCG) == 0 && (kTileN / kCG / 2) % 8 == 0;
    // Epilogue: 32-column chunks, the last one narrower when kTileN is not a
    // multiple of 32 (16 columns for a 112-wide tile)
    static constexpr int kEpiChunks = (kTileN + kEpiCols - 1) / kEpiCols;
    static constexpr int kLastChunkCols = kTileN - (kEpiChunks - 1) * kEpiCols;
    static constexpr int kBAtomBytes = kBRows * kRowBytes;            // one K atom of B
    static constexpr int kBBytes = kBAtomBytes * kAtoms;
    static constexpr int kAtomElems = kFp8 ? 128 : 64;     // K elements per atom (one TMA box)
    static constexpr int kKElems = kAtomElems * kAtoms;    // K elements per stage
    // MXFP8: per K atom of a stage (128 elements = 4 scale blocks of 32) one
    // 512-byte scale block for the CTA's 128 A rows and one per 128 B rows of
    // the whole tile (scale blocks of 32 rows × 16 bytes, see tmem_cp_128x16b;
    // in a pair each CTA holds all B scales); in shared memory and in a TMEM
    // slot the blocks go atom by atom: A, B 0, B 1, …
    static constexpr int kSfbAtoms = (kTileN + 127) / 128;
    static constexpr int kSfBlocksPerAtom = 1 + kSfbAtoms;
    static constexpr int kSfBytes = kMx ? 512 * kSfBlocksPerAtom * kAtoms : 0;   // per K block and CTA
    static constexpr int kSfColsPerAtom = kMx ? 4 * kSfBlocksPerAtom : 0;
    static constexpr int kSfCols = kSfColsPerAtom * kAtoms;                  // TMEM columns per K block
    static constexpr int kStageBytes = kAStageBytes + kBBytes;              // operands of one K block
    static constexpr int kFixed = kEpiWarps * 2 * kEpiBufBytes + 256 + 1024;   // epilogue, barriers, alignment
    // Ring depth cap: 8 for the 128-row tiles of the large shapes; the short-A
    // single-CTA kernels and the pairs narrower than 128 columns (streaming
    // kernels, latency-bound: bytes in flight set their rate) take what fits.
    static constexpr int kMaxStages = (kARows < kCtaM || (kCG == 2 && kTileN_ < 128)) ? 12 : 8;
    // MXFP8: the scales of a K block travel in their own ring of
    // kStages + kSfAhead slots (shared memory and TMEM), loaded kSfAhead K
    // blocks ahead of the operands, so that copying them into TMEM is off the
    // MMA's path. The lead is the largest (up to 4) that costs no operand stage.
    static constexpr int kStages = stages_fit(kSmemLimit - kFixed, kStageBytes, kSfBytes, kMx ? 1 : 0, kMaxStages);
    static constexpr int kSfAhead = !kMx ? 0
                                    : stages_fit(kSmemLimit - kFixed, kStageBytes, kSfBytes, 4, kMaxStages) == kStages ? 4
                                    : stages_fit(kSmemLimit - kFixed, kStageBytes, kSfBytes, 3, kMaxStages) == kStages ? 3
                                    : stages_fit(kSmemLimit - kFixed, kStageBytes, kSfBytes, 2, kMaxStages) == kStages ? 2
                                                                                                                : 1;
    static constexpr int kSfSlots = kMx ? kStages + kSfAhead : 0;
    static_assert(kStages >= 3, "pipeline too shallow");
    static constexpr int kOffA = 0;
    static constexpr int kOffB = kOffA + kStages * kAStageBytes;
    // the MMA reads kABytes from the last atom of the last stage's A: it must stay inside the buffer
    static_assert(kOffA + (kStages - 1) * kAStageBytes + (kAtoms - 1) * kAAtomBytes + kABytes <=
                      kOffB + kStages * kBBytes, "A read");
    static constexpr int kOffSf = kOffB + kStages * kBBytes;
    static constexpr int kOffEpi = kOffSf + kSfSlots * kSfBytes;
    static constexpr int kOffBars = kOffEpi + kEpiWarps * 2 * kEpiBufBytes;
    // full[S], empty[S], acc_full[2], acc_empty[2], sf_full[SF] and sf_land[SF] (MXFP8), drain[2] (abort path)
    static constexpr int kBarSfFull = 2 * kStages + 4;
    static constexpr int kBarSfLand = kBarSfFull + kSfSlots;
    static constexpr int kBarDrain = kBarSfLand + kSfSlots;
    static constexpr int kNumBars = kBarDrain + 2;
    static constexpr int kOffTmemHolder = kOffBars + kNumBars * 8;   // [0]: TMEM address, [1..2]: epilogue flags
    static constexpr int kSmemBytes = kOffTmemHolder + 16 + 1024;   // + slack for aligning the base
    static_assert(kSmemBytes <= kSmemLimit, "shared memory");
    // TMEM columns per accumulator: the tile's width in whole 32-column chunks
    // (the epilogue reads 32 columns at a time; a 112-wide tile's last read
    // takes 16 columns past its accumulator, inside the accumulator's stride)
    static constexpr int kAccCols = kEpiChunks * kEpiCols;
    // Two accumulators (the epilogue of one tile overlaps the MMAs of the
    // next) unless they and the scale ring do not fit TMEM's 512 columns: the
    // 256-wide block-scaled tile keeps one, which its epilogue reads whole
    // into registers before it stores anything, so the MMAs wait only for
    // the TMEM reads.
    static constexpr int kAccBufs = 2 * kAccCols + kSfSlots * kSfCols <= 512 ? 2 : 1;
    static constexpr int kColSf = kAccBufs * kAccCols;      // MXFP8: scale ring, kSfCols per slot
    static constexpr int kTmemCols = pow2_at_least(kAccBufs * kAccCols + kSfSlots * kSfCols);
    static_assert(kTmemCols <= 512, "TMEM");
    static constexpr uint32_t kIdesc = kMx    ? idesc_mxf8_f32(kTileM, kTileN)
                                       : kFp8 ? idesc_e4m3_f32(kTileM, kTileN)
                                              : idesc_bf16_f32(kTileM, kTileN);
    static constexpr uint32_t kIdescHalf = !kHalves ? kIdesc
                                           : kFp8   ? idesc_e4m3_f32(kTileM, kTileN / 2)
                                                    : idesc_bf16_f32(kTileM, kTileN / 2);
};

// error bits written to the status word when a bounded wait runs out
constexpr uint32_t kErrProducerEmpty = 1u << 0;
constexpr uint32_t kErrMmaFull = 1u << 1;
constexpr uint32_t kErrMmaAccEmpty = 1u << 2;
constexpr uint32_t kErrEpiAccFull = 1u << 3;

constexpr uint32_t kFlagDropArrive = 0x1u;

struct GemmParams {
    int32_t M, N, K;
    int32_t tiles_m, tiles_n;     // output tiles along M and N
    int32_t k_blocks;             // ceil(K / 64)
    int32_t num_tiles;
    int32_t splits;               // K splits per tile (1: none); work units = num_tiles * splits
    int32_t group_m;
    int32_t a_rows;               // rows of A each CTA loads per stage (128, or M rounded up to 8 if smaller)
    uint32_t expect_bytes;        // bytes that land per stage in the cluster (both CTAs of a pair)
    int64_t n_pad;                // split K: row stride of the partial matrices (tiles_n * tile width)
    float* partials;              // split K: fp32 partial matrices P[split][M][n_pad]
    int32_t sf_k_blocks;          // MXFP8: K blocks of 128 of the arranged scales (k_blocks × atoms per stage)
    float alpha;                  // scale of the accumulator (FP8: scale_a * scale_b; bf16: 1)
    const uint16_t* bias;         // fused epilogue: per-column bf16 bias (N values) or null
    int32_t act;                  // fused epilogue: 0 none, 1 ReLU, 2 GELU (erf), 3 SiLU
    const uint16_t* residual;     // fused epilogue: bf16 M×N matrix added after the activation, or null
    int64_t ldr;                  // its leading dimension (elements; may be C itself with ldr == ldc)
    int32_t tail_start;           // pair kernel: tiles from here on run as two half-width units (-1: none)
    int32_t total_units;          // work units of this launch
    uint32_t expect_bytes_half;   // bytes per stage of a half-width unit
    int32_t n_tma;                // columns [0, n_tma) of C are written by TMA stores (n_tma = N & ~7)
    int64_t ldc;                  // leading dimension of C (elements), for the ragged tail columns
    uint16_t* c_ptr;              // C, for the columns [n_tma, N) a TMA store cannot bound exactly
    uint32_t* status;             // [0]: error bits (sticky), [1]: launch id that aborted
    uint32_t launch_id;
    uint32_t flags;
    uint64_t timeout_ns;
    // MXFP8: scale blocks arranged per (tile, K stage) by mx_scale_blocks_kernel,
    // read through a tensor map over the buffer as rows of 256 bytes (one
    // 512-byte block = 2 rows, so one TMA copy moves it in two row requests);
    // A blocks from row 0, B blocks from row sf_b_row
    int64_t sf_b_row;
};

// Grouped rasterisation: tiles are numbered so that group_m consecutive tile
// rows are swept column by column; the tiles that co-run on the GPU then
// share a few rows of A and a few columns of B in L2.
__device__ __forceinline__ void tile_coords(const GemmParams& p, int t, int& tm, int& tn) {
    const int per_group = p.group_m * p.tiles_n;
    const int g = t / per_group;
    const int first_m = g * p.group_m;
    const int rows = min(p.tiles_m - first_m, p.group_m);
    const int local = t - g * per_group;
    tm = first_m + local % rows;
    tn = local / rows;
}

__device__ __forceinline__ bool aborted(const GemmParams& p) {
    return *reinterpret_cast<volatile uint32_t*>(p.status + 1) == p.launch_id;
}

// Slow path of a bounded wait for phase `parity` of `bar` (kept out of line
// so that the hot loops only carry the first probe). Returns false when the
// wait gave up: either this launch was already aborted by another role, or
// the time limit ran out (then this thread records `code` and aborts the
// launch).
__device__ __noinline__ bool wait_bounded_slow(const GemmParams& p, uint32_t bar, uint32_t parity,
                                               uint32_t code, bool cluster_scope) {
    const uint64_t t0 = global_timer_ns();
    for (uint32_t it = 1;; ++it) {
        if (cluster_scope ? mbar_try_wait_cluster_relaxed(bar, parity) : mbar_try_wait(bar, parity)) return true;
        if ((it & 63u) == 0) {
            if (aborted(p)) return false;
            if (global_timer_ns() - t0 > p.timeout_ns) {
                atomicOr(p.status, code);
                atomicExch(p.status + 1, p.launch_id);
                __threadfence();
                return false;
            }
        }
    }
}

__device__ __forceinline__ bool wait_bounded(const GemmParams& p, uint32_t bar, uint32_t parity,
                                             uint32_t code) {
    if (mbar_try_wait(bar, parity)) return true;
    return wait_bounded_slow(p, bar, parity, code, false);
}

// For barriers that the peer CTA's threads arrive on (relaxed at cluster scope,
// as the arrives; they order tcgen05 operations only).
__device__ __forceinline__ bool wait_bounded_cluster(const GemmParams& p, uint32_t bar, uint32_t parity,
                                                     uint32_t code) {
    if (mbar_try_wait_cluster_relaxed(bar, parity)) return true;
    return wait_bounded_slow(p, bar, parity, code, true);
}

// Bounded wait for a phase expected to take long (a whole main loop): each
// probe lets the hardware suspend the thread for up to 20 µs (it resumes
// when the phase completes), so the waiting thread does not take issue slots
// from the warps that do work. Same failure behaviour as wait_bounded_slow.
__device__ __noinline__ bool wait_bounded_suspend(const GemmParams& p, uint32_t bar, uint32_t parity,
                                                  uint32_t code) {
    const uint64_t t0 = global_timer_ns();
    for (;;) {
        if (mbar_try_wait_suspend(bar, parity, 20000)) return true;
        if (aborted(p)) return false;
        if (global_timer_ns() - t0 > p.timeout_ns) {
            atomicOr(p.status, code);
            atomicExch(p.status + 1, p.launch_id);
            __threadfence();
            return false;
        }
    }
}

// Fused epilogue on one fp32 accumulator value: + bias, then the activation.
__device__ __forceinline__ float epilogue_op(float x, float bias, int act) {
    x += bias;
    switch (act) {
        case 1: return fmaxf(x, 0.0f);
        case 2: return 0.5f * x * (1.0f + erff(x * 0.70710678118654752f));   // x·Φ(x)
        // x·σ(x) through CUDA's fast exponential and division intrinsics: their few
        // fp32 ulps of error are far below the bf16 rounding that follows; for
        // x below about -87 the quotient comes out 0 instead of a value under
        // 1e-36 in magnitude. Measured: 9.6 % -> 5.5 % over the plain GEMM at
        // 8192^3, against expf and an IEEE division
        case 3: return __fdividef(x, 1.0f + __expf(-x));
        default: return x;
    }
}

__device__ __forceinline__ float bf16_bits_to_float(uint16_t h) {
    return __uint_as_float(static_cast<uint32_t>(h) << 16);
}

// + bias, then the activation, on 32 accumulator values of columns col0..col0+31.
__device__ __forceinline__ void apply_bias_act(const GemmParams& p, uint32_t (&v)[32], int col0) {
    float b[32];
    if (p.bias != nullptr && col0 + 32 <= p.N) {
        const uint4* src = reinterpret_cast<const uint4*>(p.bias + col0);   // 64-byte aligned chunk
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const uint4 x = __ldg(src + q);
            const uint32_t w4[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
            for (int h = 0; h < 4; ++h) {
                b[8 * q + 2 * h] = bf16_bits_to_float(static_cast<uint16_t>(w4[h] & 0xFFFFu));
                b[8 * q + 2 * h + 1] = bf16_bits_to_float(static_cast<uint16_t>(w4[h] >> 16));
            }
        }
    } else {
#pragma unroll
        for (int e = 0; e < 32; ++e)
            b[e] = (p.bias != nullptr && col0 + e < p.N) ? bf16_bits_to_float(p.bias[col0 + e]) : 0.0f;
    }
#pragma unroll
    for (int e = 0; e < 32; ++e) v[e] = __float_as_uint(epilogue_op(__uint_as_float(v[e]), b[e], p.act));
}

// The residual of one row, columns col0..col0+31, as 16 packed bf16 pairs
// (zero past N and for rows past M). Issued before the accumulator's TMEM
// load so that the two latencies overlap. Plain (coherent) loads: R may be C
// itself, each element read by the thread that later writes it.
__device__ __forceinline__ void load_residual(const GemmParams& p, int row, int col0, uint32_t (&r)[16]) {
#pragma unroll
    for (int i = 0; i < 16; ++i) r[i] = 0u;
    if (p.residual == nullptr || row >= p.M) return;
    const uint16_t* src = p.residual + static_cast<int64_t>(row) * p.ldr + col0;
    if (col0 + 32 <= p.N) {
        const uint4* q = reinterpret_cast<const uint4*>(src);   // 16-byte aligned: R, ldr % 8, col0 % 32
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const uint4 x = q[j];
            r[4 * j] = x.x; r[4 * j + 1] = x.y; r[4 * j + 2] = x.z; r[4 * j + 3] = x.w;
        }
    } else {
#pragma unroll
        for (int e = 0; e < 32; ++e)
            if (col0 + e < p.N) r[e >> 1] |= static_cast<uint32_t>(src[e]) << (16 * (e & 1));
    }
}

// Apply the fused epilogue to 32 accumulator values of columns col0..col0+31:
// scale, + bias, activation, + residual (r: this row's residual from
// load_residual, ignored when the epilogue has none).
__device__ __forceinline__ void apply_epilogue(const GemmParams& p, uint32_t (&v)[32], int col0,
                                               const uint32_t (&r)[16]) {
    if (p.alpha != 1.0f) {
#pragma unroll
        for (int e = 0; e < 32; ++e) v[e] = __float_as_uint(__uint_as_float(v[e]) * p.alpha);
    }
    if (p.bias != nullptr || p.act != 0) apply_bias_act(p, v, col0);
    if (p.residual != nullptr) {
#pragma unroll
        for (int e = 0; e < 32; ++e) {
            const uint16_t h = static_cast<uint16_t>((e & 1) ? (r[e >> 1] >> 16) : (r[e >> 1] & 0xFFFFu));
            v[e] = __float_as_uint(__uint_as_float(v[e]) + bf16_bits_to_float(h));
        }
    }
}
// K blocks [begin, end) of split `s` of `splits` (as even as possible).
__device__ __forceinline__ void split_range(const GemmParams& p, int s, int& begin, int& end) {
    begin = static_cast<int>((static_cast<int64_t>(s) * p.k_blocks) / p.splits);
    end = static_cast<int>((static_cast<int64_t>(s + 1) * p.k_blocks) / p.splits);
}

// Work unit u -> tile, K split and half. Units before tail_start are whole
// tiles (times the K splits); from tail_start on, each tile of the last,
// partial round of the schedule is run as two units of half its width, so
// that the round keeps twice as many units busy (half = 0 or 1; -1: whole).
__device__ __forceinline__ void unit_info(const GemmParams& p, int u, int& t, int& split, int& half) {
    if (p.tail_start >= 0 && u >= p.tail_start) {
        t = p.tail_start + ((u - p.tail_start) >> 1);
        split = 0;
        half = (u - p.tail_start) & 1;
    } else {
        t = u / p.splits;
        split = u - t * p.splits;
        half = -1;
    }
}

// Abort path: wait for phase `parity` of `bar` for at most `limit_ns`
// (a copy or MMA issued before the abort signals it when it completes).
__device__ __forceinline__ bool wait_drain(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
    const uint64_t t0 = global_timer_ns();
    while (!mbar_try_wait(bar, parity))
        if (global_timer_ns() - t0 > limit_ns) return false;
    return true;
}

constexpr uint64_t kDrainLimitNs = 2000000;   // 2 ms per drain wait (a copy or MMA lands within microseconds)

// Abort path, last step: a short back-off for copies no barrier of this CTA
// can show complete (a peer CTA's loads into a stage this CTA's producer
// never armed, and the loads of a stage whose arrival was withheld on purpose).
__device__ __forceinline__ void drain_unobserved_copies() {
    for (int i = 0; i < 20; ++i) __nanosleep(1000);
}

template <int kCG, int kTileN, bool kFp8, bool kMx = false, int kARows = kCtaM, int kAtoms = 1>
__global__ void __launch_bounds__(kThreads, 1)
gemm_bf16_kernel(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_b,
                 const __grid_constant__ CUtensorMap tmap_c, const __grid_constant__ CUtensorMap tmap_b_half,
                 const GemmParams p) {
    using G = Geometry<kCG, kTileN, kFp8, kMx, kARows, kAtoms>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* const smem = smem_raw + (base - raw);

    const uint32_t warp = threadIdx.x >> 5;
    const uint32_t lane = lane_id();
    const uint32_t rank = kCG == 2 ? cluster_cta_rank() : 0u;   // 0 = leader of the pair
    const int unit = blockIdx.x / kCG;                          // this CTA's pair (or CTA)
    const int num_units = gridDim.x / kCG;

    auto full_bar = [&](int s) { return base + G::kOffBars + 8u * s; };
    auto empty_bar = [&](int s) { return base + G::kOffBars + 8u * (G::kStages + s); };
    auto acc_full_bar = [&](int b) { return base + G::kOffBars + 8u * (2 * G::kStages + b); };
    auto acc_empty_bar = [&](int b) { return base + G::kOffBars + 8u * (2 * G::kStages + 2 + b); };
    // MXFP8 scale slot j: its scales are in TMEM (sf_full) / have landed in shared memory (sf_land)
    auto sf_full_bar = [&](int j) { return base + G::kOffBars + 8u * (G::kBarSfFull + j); };
    auto sf_land_bar = [&](int j) { return base + G::kOffBars + 8u * (G::kBarSfLand + j); };
    // abort path: all tcgen05 operations of the MMA issuer ([0]) and of the scale copier ([1]) complete
    auto drain_bar = [&](int i) { return base + G::kOffBars + 8u * (G::kBarDrain + i); };
    const uint32_t tmem_holder = base + G::kOffTmemHolder;

    if (threadIdx.x == 0) {
        for (int s = 0; s < G::kStages; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(acc_full_bar(b), 1);
            mbar_init(acc_empty_bar(b), kCG * kEpiWarps);
        }
        if constexpr (kMx)
            for (int j = 0; j < G::kSfSlots; ++j) {
                mbar_init(sf_full_bar(j), 1);
                mbar_init(sf_land_bar(j), 1);
            }
        mbar_init(drain_bar(0), 1);
        mbar_init(drain_bar(1), 1);
        fence_mbar_init_cluster();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tensor_map(&tmap_a);
        prefetch_tensor_map(&tmap_b);
        prefetch_tensor_map(&tmap_c);
        // the split-K reduction, launched after this kernel as a programmatic
        // dependent, may be scheduled now; it waits for this grid to complete
        griddep_launch_dependents();
    }
    if (warp == 1) {
        if constexpr (kCG == 2) {
            tmem_alloc_pair(tmem_holder, G::kTmemCols);
            tmem_relinquish_pair();
        } else {
            tmem_alloc_one(tmem_holder, G::kTmemCols);
            tmem_relinquish_one();
        }
    }
    tc_fence_before_sync();
    if constexpr (kCG == 2) cluster_sync(); else __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem_base = *reinterpret_cast<volatile uint32_t*>(smem + G::kOffTmemHolder);

    bool abort_seen = false;

    if (warp == 0) {
        // ------------------------------------------------ TMA producer --
        if (lane == 0) {
            // launched as a programmatic dependent (of the previous kernel on the stream,
            // which may have written A or B; of the scale arrangement for the block-scaled
            // GEMM): nothing from global memory is read before that grid has completed
            griddep_wait();
            int stage = 0;
            uint32_t phase = 0;
            bool dropped = false;
            int64_t fills = 0;            // stages armed and loaded by this producer so far
            int64_t dropped_fill = -1;    // the fill whose arrival the test fault withheld
            const int total = p.total_units;
            // MXFP8 scales: a second cursor over the same (unit, K block) sequence,
            // kSfAhead K blocks ahead of the operand loads, filling the scale ring.
            // Scale slot j is reused for K block g + kSfSlots only once the MMAs of
            // K block g completed; the operand stage wait for K block
            // g + kSfSlots - kSfAhead = g + kStages establishes exactly that.
            int sf_u = unit, sf_kb = 0, sf_kb_end = 0, sf_tm = 0, sf_tn = 0, sf_slot = 0;
            int64_t sf_fills = 0;         // scale slots armed and loaded so far
            auto sf_seek = [&]() {        // the cursor's unit is sf_u: its tile and K range
                if (sf_u >= total) return;
                int t, split, half;
                unit_info(p, sf_u, t, split, half);
                tile_coords(p, t, sf_tm, sf_tn);
                split_range(p, split, sf_kb, sf_kb_end);
            };
            auto sf_load_next = [&]() {   // the next K block's scale blocks into the next slot
                while (sf_u < total && sf_kb >= sf_kb_end) {
                    sf_u += num_units;
                    sf_seek();
                }
                if (sf_u >= total) return;
                const uint32_t land = sf_land_bar(sf_slot);
                if (rank == 0) mbar_arrive_expect_tx(land, static_cast<uint32_t>(kCG * G::kSfBytes));
                const uint32_t land_leader = kCG == 2 ? map_to_cta(land, 0) : land;
                const int64_t a_group = static_cast<int64_t>(sf_tm) * kCG + rank;   // 128-row group
#pragma unroll
                for (int at = 0; at < kAtoms; ++at) {
                    const int64_t kb128 = static_cast<int64_t>(sf_kb) * kAtoms + at;   // K block of 128
                    const uint32_t sf_dst = base + G::kOffSf + sf_slot * G::kSfBytes + at * 512 * G::kSfBlocksPerAtom;
                    const int a_row_sf = static_cast<int>((a_group * p.sf_k_blocks + kb128) * 2);
                    const int b_row_sf = static_cast<int>(
                        p.sf_b_row + (static_cast<int64_t>(sf_tn) * p.sf_k_blocks + kb128) * (2 * G::kSfbAtoms));
                    // (the scale blocks' tensor map rides in the half-B slot)
                    if constexpr (kCG == 2) {
                        tma_load_2d_pair(sf_dst, &tmap_b_half, 0, a_row_sf, land_leader);
                        for (int q = 0; q < G::kSfbAtoms; ++q)
                            tma_load_2d_pair(sf_dst + 512 * (1 + q), &tmap_b_half, 0, b_row_sf + 2 * q, land_leader);
                    } else {
                        tma_load_2d(sf_dst, &tmap_b_half, 0, a_row_sf, land);
                        for (int q = 0; q < G::kSfbAtoms; ++q)
                            tma_load_2d(sf_dst + 512 * (1 + q), &tmap_b_half, 0, b_row_sf + 2 * q, land);
                    }
                }
                ++sf_kb;
                ++sf_fills;
                if (++sf_slot == G::kSfSlots) sf_slot = 0;
            };
            if constexpr (kMx) {
                sf_seek();
                for (int i = 0; i < G::kSfAhead; ++i) sf_load_next();   // slots never used before
            }
            for (int u = unit; u < total && !abort_seen; u += num_units) {
                int t, split, half;
                unit_info(p, u, t, split, half);
                int tm, tn, kb_begin, kb_end;
                tile_coords(p, t, tm, tn);
                split_range(p, split, kb_begin, kb_end);
                const int a_row = tm * G::kTileM + static_cast<int>(rank) * kCtaM;
                const int b_row = half < 0 ? tn * G::kTileN + static_cast<int>(rank) * G::kBRows
                                           : tn * G::kTileN + half * (G::kTileN / 2) +
                                                 static_cast<int>(rank) * (G::kBRows / 2);
                const void* const b_map = half < 0 ? static_cast<const void*>(&tmap_b)
                                                   : static_cast<const void*>(&tmap_b_half);
                const uint32_t stage_bytes = half < 0 ? p.expect_bytes : p.expect_bytes_half;
                for (int kb = kb_begin; kb < kb_end; ++kb) {
                    // a full ring ahead of the MMAs: the wait may suspend the thread (the
                    // probes otherwise cost instructions, not time: measured no change in
                    // kernel cycles either way)
                    if (!(mbar_try_wait(empty_bar(stage), phase ^ 1u) ||
                          wait_bounded_suspend(p, empty_bar(stage), phase ^ 1u, kErrProducerEmpty))) {
                        abort_seen = true;
                        break;
                    }
                    if (rank == 0) {
                        if ((p.flags & kFlagDropArrive) && !dropped) {
                            dropped = true;   // test-only fault: withhold this arrival
                            dropped_fill = fills;
                        } else {
                            mbar_arrive_expect_tx(full_bar(stage), stage_bytes);
                        }
                    }
                    const uint32_t a_dst = base + G::kOffA + stage * G::kAStageBytes;
                    const uint32_t b_dst = base + G::kOffB + stage * G::kBBytes;
#pragma unroll
                    for (int at = 0; at < kAtoms; ++at) {
                        const int kx = kb * G::kKElems + at * G::kAtomElems;
                        if constexpr (kCG == 2) {
                            // both CTAs' copies complete on the leader's barrier
                            const uint32_t leader_full = map_to_cta(full_bar(stage), 0);
                            tma_load_2d_pair(a_dst + at * G::kAAtomBytes, &tmap_a, kx, a_row, leader_full);
                            tma_load_2d_pair(b_dst + at * G::kBAtomBytes, b_map, kx, b_row, leader_full);
                        } else {
                            tma_load_2d(a_dst + at * G::kAAtomBytes, &tmap_a, kx, a_row, full_bar(stage));
                            tma_load_2d(b_dst + at * G::kBAtomBytes, b_map, kx, b_row, full_bar(stage));
                        }
                    }
                    ++fills;
                    if constexpr (kMx) sf_load_next();   // the scales kSfAhead K blocks ahead
                    if (++stage == G::kStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            // Abort: the leader's full and scale barriers count the bytes of both CTAs'
            // loads; wait (bounded) for the fills it armed that may still be in flight.
            if (rank == 0 && (abort_seen || aborted(p))) {
                for (int64_t f = fills - 1; f >= 0 && f >= fills - G::kStages; --f) {
                    if (f == dropped_fill) continue;
                    (void)wait_drain(full_bar(static_cast<int>(f % G::kStages)),
                                     static_cast<uint32_t>((f / G::kStages) & 1), kDrainLimitNs);
                }
                if constexpr (kMx)
                    for (int64_t f = sf_fills - 1; f >= 0 && f >= sf_fills - G::kSfSlots; --f)
                        (void)wait_drain(sf_land_bar(static_cast<int>(f % G::kSfSlots)),
                                         static_cast<uint32_t>((f / G::kSfSlots) & 1), kDrainLimitNs);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------- MMA issuer --
        // The whole warp runs the loop (warp-uniform control flow and
        // descriptor arithmetic) and lane 0 issues the MMAs and commits:
        // measured 3 % faster than a loop run by lane 0 alone.
        if (rank == 0) {
            int stage = 0;
            uint32_t phase = 0;
            int sf_slot = 0;              // MXFP8: scale slot of the current K block
            uint32_t sf_phase = 0;
            int local = 0;
            const int total = p.total_units;
            for (int u = unit; u < total && !abort_seen; u += num_units, ++local) {
                int t, split, half;
                unit_info(p, u, t, split, half);
                int kb_begin, kb_end;
                split_range(p, split, kb_begin, kb_end);
                const uint32_t idesc = half < 0 ? G::kIdesc : G::kIdescHalf;
                const int buf = G::kAccBufs == 2 ? (local & 1) : 0;
                const uint32_t acc_phase = G::kAccBufs == 2 ? ((local >> 1) & 1) : (local & 1);
                const bool acc_free = kCG == 2
                                          ? wait_bounded_cluster(p, acc_empty_bar(buf), acc_phase ^ 1u, kErrMmaAccEmpty)
                                          : wait_bounded(p, acc_empty_bar(buf), acc_phase ^ 1u, kErrMmaAccEmpty);
                if (!acc_free) {
                    abort_seen = true;
                    break;
                }
                tc_fence_after_sync();
                const uint32_t d_tmem = tmem_base + buf * G::kAccCols;
                for (int kb = kb_begin; kb < kb_end; ++kb) {
                    if (!wait_bounded(p, full_bar(stage), phase, kErrMmaFull) ||
                        (kMx && !wait_bounded(p, sf_full_bar(sf_slot), sf_phase, kErrMmaFull))) {
                        abort_seen = true;
                        break;
                    }
                    tc_fence_after_sync();
                    const uint64_t a_desc = smem_desc_kmajor_sw128(base + G::kOffA + stage * G::kAStageBytes);
                    const uint64_t b_desc = smem_desc_kmajor_sw128(base + G::kOffB + stage * G::kBBytes);
                    if constexpr (kMx) {
#pragma unroll
                        for (int at = 0; at < kAtoms; ++at) {
                            // this atom's scales, copied into the stage's TMEM slot by the scale copier
                            const uint32_t sf_tmem = tmem_base + G::kColSf + sf_slot * G::kSfCols + at * G::kSfColsPerAtom;
                            const uint64_t ad = a_desc + static_cast<uint64_t>((at * G::kAAtomBytes) >> 4);
                            const uint64_t bd = b_desc + static_cast<uint64_t>((at * G::kBAtomBytes) >> 4);
#pragma unroll
                            for (int k = 0; k < kRowBytes / kMmaKBytes; ++k) {
                                const uint32_t acc = (kb != kb_begin || at != 0 || k != 0) ? 1u : 0u;
                                // scale block k of the 4 in this atom: byte k of each scale word
                                const uint32_t id = idesc | (static_cast<uint32_t>(k) << 4) |
                                                    (static_cast<uint32_t>(k) << 29);
                                if (lane == 0) {
                                    if constexpr (kCG == 2)
                                        mma_mxf8_pair(d_tmem, ad + 2u * k, bd + 2u * k, id, sf_tmem, sf_tmem + 4, acc);
                                    else
                                        mma_mxf8_one(d_tmem, ad + 2u * k, bd + 2u * k, id, sf_tmem, sf_tmem + 4, acc);
                                }
                            }
                        }
                    } else {
#pragma unroll
                        for (int at = 0; at < kAtoms; ++at) {
                            // descriptors of atom `at` (start address field in 16-byte units)
                            const uint64_t ad = a_desc + static_cast<uint64_t>((at * G::kAAtomBytes) >> 4);
                            const uint64_t bd = b_desc + static_cast<uint64_t>((at * G::kBAtomBytes) >> 4);
#pragma unroll
                            for (int k = 0; k < kRowBytes / kMmaKBytes; ++k) {
                                // advance 32 bytes along K inside the swizzle atom (16 bf16 or 32 FP8)
                                const uint32_t acc = (kb != kb_begin || at != 0 || k != 0) ? 1u : 0u;
                                if (lane == 0) {
                                    if constexpr (kCG == 2 && kFp8)
                                        mma_f8_pair(d_tmem, ad + 2u * k, bd + 2u * k, idesc, acc);
                                    else if constexpr (kCG == 2)
                                        mma_bf16_pair(d_tmem, ad + 2u * k, bd + 2u * k, idesc, acc);
                                    else if constexpr (kFp8)
                                        mma_f8_one(d_tmem, ad + 2u * k, bd + 2u * k, idesc, acc);
                                    else
                                        mma_bf16_one(d_tmem, ad + 2u * k, bd + 2u * k, idesc, acc);
                                }
                            }
                        }
                    }
                    // free this stage (in both CTAs of a pair) once the MMAs above have read it
                    if (lane == 0) {
                        if constexpr (kCG == 2) mma_commit_pair_mask(empty_bar(stage), 0x3);
                        else mma_commit_one(empty_bar(stage));
                    }
                    if (++stage == G::kStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                    if (kMx && ++sf_slot == G::kSfSlots) {
                        sf_slot = 0;
                        sf_phase ^= 1u;
                    }
                }
                if (abort_seen) break;
                // accumulator complete: hand it to the epilogue(s)
                if (lane == 0) {
                    if constexpr (kCG == 2) mma_commit_pair_mask(acc_full_bar(buf), 0x3);
                    else mma_commit_one(acc_full_bar(buf));
                }
            }
            // Abort: every MMA this thread issued completes before TMEM is freed
            if (abort_seen || aborted(p)) {
                if (lane == 0) {
                    if constexpr (kCG == 2) mma_commit_pair_mask(drain_bar(0), 0x1);
                    else mma_commit_one(drain_bar(0));
                }
                (void)wait_drain(drain_bar(0), 0, kDrainLimitNs);
            }
        }
    } else if (warp == 2 + kEpiWarps) {
        // ---------------------------------------- MXFP8 scale copier --
        // Once a K block's scale blocks have landed in their slot (sf_land), copy
        // them into the slot's TMEM columns and signal sf_full, on which the MMA
        // thread waits besides the operands' full barrier. Issued here rather
        // than by the MMA thread, the copies never stand between two MMAs in
        // that thread's stream (measured: 397 -> 354 us at 8192^3); loaded
        // kSfAhead K blocks ahead of the operands, they are done before the MMA
        // needs them (measured at 8192^3: 576K -> 509K kernel cycles against
        // copying a stage's scales once its operands had landed, when the MMA
        // waited for the copy after the operands).
        if constexpr (kMx) {
            if (rank == 0 && lane == 0) {
                int sf_slot = 0;
                uint32_t sf_phase = 0;
                for (int u = unit; u < p.total_units && !abort_seen; u += num_units) {
                    int t, split, half;
                    unit_info(p, u, t, split, half);
                    int kb_begin, kb_end;
                    split_range(p, split, kb_begin, kb_end);
                    for (int kb = kb_begin; kb < kb_end; ++kb) {
                        if (!wait_bounded(p, sf_land_bar(sf_slot), sf_phase, kErrMmaFull)) {
                            abort_seen = true;
                            break;
                        }
                        tc_fence_after_sync();
                        const uint32_t sf_src = base + G::kOffSf + sf_slot * G::kSfBytes;
                        const uint32_t sf_tmem = tmem_base + G::kColSf + sf_slot * G::kSfCols;
#pragma unroll
                        for (int q = 0; q < G::kSfBlocksPerAtom * kAtoms; ++q) {   // atom by atom: A, B 0, B 1, …
                            if constexpr (kCG == 2)
                                tmem_cp_128x16b_pair(sf_tmem + 4 * q, smem_desc_plain(sf_src + 512 * q, 16, 128));
                            else
                                tmem_cp_128x16b(sf_tmem + 4 * q, smem_desc_plain(sf_src + 512 * q, 16, 128));
                        }
                        if constexpr (kCG == 2) mma_commit_pair_mask(sf_full_bar(sf_slot), 0x1);
                        else mma_commit_one(sf_full_bar(sf_slot));
                        if (++sf_slot == G::kSfSlots) {
                            sf_slot = 0;
                            sf_phase ^= 1u;
                        }
                    }
                }
                // Abort: every scale copy this thread issued completes before TMEM is freed
                if (abort_seen || aborted(p)) {
                    if constexpr (kCG == 2) mma_commit_pair_mask(drain_bar(1), 0x1);
                    else mma_commit_one(drain_bar(1));
                    (void)wait_drain(drain_bar(1), 0, kDrainLimitNs);
                }
            }
        }
    } else {
        // --------------------------------------------------- epilogue --
        // no global read or write (C, bias, residual, split partials) before the
        // grid this one depends on has completed
        griddep_wait();
        const uint32_t q = warp & 3u;                  // TMEM lane quarter this warp may read
        const uint32_t epi = base + G::kOffEpi + (warp - 2) * 2 * kEpiBufBytes;
        const uint32_t swz = (lane >> 1) & 3u;         // 64-byte swizzle of this lane's row
        uint32_t chunk_count = 0;

        // Round 32 fp32 values of this lane's row to bf16 and write them to C
        // at (row0 + lane, col0): staged through 64-byte-swizzled shared
        // memory and written by a TMA store; when N is not a multiple of 8
        // the last (< 8) columns are written with plain stores, since a TMA
        // store bounds the innermost dimension only to 16-byte granules.
        auto store_packed = [&](const uint32_t (&w)[16], int row0, int col0) {
            const uint32_t sbuf = epi + (chunk_count & 1u) * kEpiBufBytes;
            if (lane == 0) bulk_wait_group_read<1>();   // the store that last used sbuf has read it
            __syncwarp();
            const uint32_t row_addr = sbuf + lane * 64u;
#pragma unroll
            for (int j = 0; j < 4; ++j)
                st_shared_v4(row_addr + ((static_cast<uint32_t>(j) ^ swz) << 4), w[4 * j], w[4 * j + 1],
                             w[4 * j + 2], w[4 * j + 3]);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0 && row0 < p.M && col0 < p.n_tma) tma_store_2d(&tmap_c, sbuf, col0, row0);
            if (lane == 0) bulk_commit_group();
            if (p.N > p.n_tma && col0 + kEpiCols > p.n_tma && col0 < p.N) {
                const int row = row0 + static_cast<int>(lane);
                if (row < p.M) {
                    uint16_t* const crow = p.c_ptr + static_cast<int64_t>(row) * p.ldc;
#pragma unroll
                    for (int e = 0; e < kEpiCols; ++e) {   // static indices keep w[] in registers
                        const int j = col0 + e;
                        if (j >= p.n_tma && j < p.N)
                            crow[j] = static_cast<uint16_t>((e & 1) ? (w[e >> 1] >> 16) : (w[e >> 1] & 0xFFFFu));
                    }
                }
            }
            ++chunk_count;
        };
        auto store_chunk = [&](uint32_t (&v)[32], int row0, int col0, const uint32_t (&r)[16]) {
            if (p.bias != nullptr || p.act != 0 || p.alpha != 1.0f || p.residual != nullptr) apply_epilogue(p, v, col0, r);
            uint32_t w[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) w[i] = pack_bf16x2_rn(v[2 * i], v[2 * i + 1]);
            store_packed(w, row0, col0);
        };
        // The last, narrower chunk of a tile whose width is not a multiple of 32
        // (16 columns of a 112-wide tile): the 32 values are computed as for a
        // full chunk (the upper 16 come from TMEM columns past the accumulator
        // and are dropped), and this lane's row gets the first kLastChunkCols
        // by plain stores, 16-byte ones where they fit inside N (C's rows are
        // 16-byte aligned, as its tensor map requires, and col0 is a multiple of 16).
        auto store_chunk_narrow = [&](uint32_t (&v)[32], int row, int col0, const uint32_t (&r)[16]) {
            if (p.bias != nullptr || p.act != 0 || p.alpha != 1.0f || p.residual != nullptr) apply_epilogue(p, v, col0, r);
            constexpr int kCols = G::kLastChunkCols;
            uint32_t w[kCols / 2];
#pragma unroll
            for (int i = 0; i < kCols / 2; ++i) w[i] = pack_bf16x2_rn(v[2 * i], v[2 * i + 1]);
            if (row >= p.M) return;
            uint16_t* const crow = p.c_ptr + static_cast<int64_t>(row) * p.ldc;
            if (col0 + kCols <= p.N) {
                uint4* const dst = reinterpret_cast<uint4*>(crow + col0);
#pragma unroll
                for (int q = 0; q < kCols / 8; ++q) dst[q] = make_uint4(w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]);
            } else {
#pragma unroll
                for (int e = 0; e < kCols; ++e)   // static indices keep w[] in registers
                    if (col0 + e < p.N)
                        crow[col0 + e] = static_cast<uint16_t>((e & 1) ? (w[e >> 1] >> 16) : (w[e >> 1] & 0xFFFFu));
            }
        };

        int local = 0;
        const int total = p.total_units;
        for (int u = unit; u < total; u += num_units, ++local) {
            int t, split, half;
            unit_info(p, u, t, split, half);
            int tm, tn;
            tile_coords(p, t, tm, tn);
            const int chunks = half < 0 ? G::kEpiChunks : (G::kTileN / 2) / kEpiCols;
            const int col_base = tn * G::kTileN + (half < 0 ? 0 : half * (G::kTileN / 2));
            const int buf = G::kAccBufs == 2 ? (local & 1) : 0;
            const uint32_t acc_phase = G::kAccBufs == 2 ? ((local >> 1) & 1) : (local & 1);
            {
                // One thread waits for the accumulator, suspended rather than polling (the
                // issuing threads of the producer and the MMA share the SM's issue slots;
                // measured 2-3 % fewer kernel cycles with two accumulators, 7 % with the
                // block-scaled pair's one, where four polling warps took the MMA thread's
                // issue slots for the whole main loop); the four epilogue warps then meet
                // at a named barrier, where the other three wait without issuing. The
                // result goes through a flag per tile parity: the writer of tile t+2's flag
                // has passed tile t+1's barrier, so every warp has read tile t's.
                volatile uint32_t* const acc_ok =
                    reinterpret_cast<volatile uint32_t*>(smem + G::kOffTmemHolder + 4) + (local & 1);
                if (warp == 2 && lane == 0)
                    *acc_ok = wait_bounded_suspend(p, acc_full_bar(buf), acc_phase, kErrEpiAccFull) ? 1u : 0u;
                __syncwarp();
                named_barrier_sync(1, 32 * kEpiWarps);
                if (*acc_ok == 0u) {
                    abort_seen = true;
                    break;
                }
            }
            tc_fence_after_sync();
            const int tile_row = static_cast<int>(rank) * kCtaM + static_cast<int>(q) * 32;   // in the tile
            const int row0 = tm * G::kTileM + tile_row;
            const int row = row0 + static_cast<int>(lane);
            const uint32_t t_row = tmem_base + ((q * 32u) << 16) + buf * G::kAccCols;
            // split K: this lane's row of this split's fp32 partial matrix
            float* const part_row =
                p.partials + (static_cast<int64_t>(split) * p.M + row) * p.n_pad + tn * G::kTileN;
            if constexpr (G::kAccBufs == 1) {
                // one accumulator: read all of it (as bf16 pairs), release it, then store.
                // Such tiles never split K, never come in halves and have no fused epilogue.
                static_assert(G::kLastChunkCols == kEpiCols, "one accumulator: whole 32-column chunks");
                constexpr int kChunks = G::kTileN / kEpiCols;
                uint32_t w[kChunks][16];
#pragma unroll
                for (int c = 0; c < kChunks; c += 2) {
                    uint32_t v0[32], v1[32];
                    if (p.k_blocks > 0) {
                        tmem_load_32cols(t_row + c * kEpiCols, v0);
                        tmem_load_32cols(t_row + (c + 1) * kEpiCols, v1);
                        tmem_wait_ld();
                    } else {
#pragma unroll
                        for (int i = 0; i < 32; ++i) v0[i] = v1[i] = 0u;
                    }
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        w[c][i] = pack_bf16x2_rn(v0[2 * i], v0[2 * i + 1]);
                        w[c + 1][i] = pack_bf16x2_rn(v1[2 * i], v1[2 * i + 1]);
                    }
                }
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0) {
                    if constexpr (kCG == 2) mbar_arrive_cluster_relaxed(map_to_cta(acc_empty_bar(buf), 0));
                    else mbar_arrive(acc_empty_bar(buf));
                }
#pragma unroll
                for (int c = 0; c < kChunks; ++c) store_packed(w[c], row0, col_base + c * kEpiCols);
            } else {
#pragma unroll 1
                for (int c = 0; c < chunks; ++c) {
                    uint32_t v[32];
                    uint32_t r[16];
                    if (p.splits == 1) load_residual(p, row, col_base + c * kEpiCols, r);
                    if (p.k_blocks > 0) {
                        tmem_load_32cols(t_row + c * kEpiCols, v);
                        tmem_wait_ld();
                    } else {
#pragma unroll
                        for (int i = 0; i < 32; ++i) v[i] = 0u;
                    }
                    if (c == chunks - 1) {
                        // every TMEM read of this accumulator is done: release it to the MMA
                        tc_fence_before_sync();
                        __syncwarp();
                        if (lane == 0) {
                            if constexpr (kCG == 2) mbar_arrive_cluster_relaxed(map_to_cta(acc_empty_bar(buf), 0));
                            else mbar_arrive(acc_empty_bar(buf));
                        }
                    }
                    // (only whole-width units have a narrow last chunk: no half units then)
                    const bool narrow = G::kLastChunkCols < kEpiCols && c == chunks - 1;
                    if (p.splits == 1) {
                        if constexpr (G::kLastChunkCols < kEpiCols) {
                            if (narrow) store_chunk_narrow(v, row, col_base + c * kEpiCols, r);
                            else store_chunk(v, row0, col_base + c * kEpiCols, r);
                        } else {
                            store_chunk(v, row0, col_base + c * kEpiCols, r);
                        }
                    } else if (row < p.M) {
                        // this split's partial (rows of n_pad = tiles_n × kTileN columns)
                        float4* dst = reinterpret_cast<float4*>(part_row + c * kEpiCols);
                        const int n4 = narrow ? G::kLastChunkCols / 4 : kEpiCols / 4;
#pragma unroll
                        for (int j = 0; j < 8; ++j)
                            if (j < n4)
                                dst[j] = make_float4(__uint_as_float(v[4 * j]), __uint_as_float(v[4 * j + 1]),
                                                     __uint_as_float(v[4 * j + 2]), __uint_as_float(v[4 * j + 3]));
                    }
                }
            }
        }
        if (lane == 0) bulk_wait_group<0>();
        __syncwarp();
    }

    if (abort_seen || aborted(p)) drain_unobserved_copies();
    __syncwarp();
    tc_fence_before_sync();
    if constexpr (kCG == 2) cluster_sync(); else __syncthreads();
    if (warp == 1) {
        tc_fence_after_sync();
        if constexpr (kCG == 2) tmem_dealloc_pair(tmem_base, G::kTmemCols);
        else tmem_dealloc_one(tmem_base, G::kTmemCols);
    }
}

// Split K, second pass: C = bf16_rne(act(P[0] + P[1] + ... + P[splits-1] +
// bias) + R), summed in this fixed order (so the result does not depend on
// which split finished first). Each thread handles 8 consecutive columns of
// one row. Launched as a programmatic dependent of the GEMM, so that its launch
// overlaps the GEMM; it waits for the GEMM grid to complete before reading.
__global__ void __launch_bounds__(256)
splitk_reduce_kernel(const float* __restrict__ partials, int32_t splits, int32_t M, int32_t N, int64_t n_pad,
                     uint16_t* C, int64_t ldc, const uint16_t* __restrict__ bias, int32_t act,
                     float alpha, const uint16_t* residual, int64_t ldr) {
    griddep_wait();
    const int64_t groups_per_row = (N + 7) / 8;
    const int64_t total = static_cast<int64_t>(M) * groups_per_row;
    const int64_t split_stride = static_cast<int64_t>(M) * n_pad;
    for (int64_t g = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; g < total;
         g += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t row = g / groups_per_row;
        const int col = static_cast<int>(g - row * groups_per_row) * 8;
        const float4* src = reinterpret_cast<const float4*>(partials + row * n_pad + col);
        float4 a = __ldcs(src), b = __ldcs(src + 1);
#pragma unroll 4
        for (int sp = 1; sp < splits; ++sp) {
            const float4* q = reinterpret_cast<const float4*>(partials + sp * split_stride + row * n_pad + col);
            const float4 x = __ldcs(q), y = __ldcs(q + 1);
            a.x += x.x; a.y += x.y; a.z += x.z; a.w += x.w;
            b.x += y.x; b.y += y.y; b.z += y.z; b.w += y.w;
        }
        if (alpha != 1.0f) {
            a.x *= alpha; a.y *= alpha; a.z *= alpha; a.w *= alpha;
            b.x *= alpha; b.y *= alpha; b.z *= alpha; b.w *= alpha;
        }
        if (bias != nullptr || act != 0) {
            float bb[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) bb[e] = (bias != nullptr && col + e < N) ? bf16_bits_to_float(bias[col + e]) : 0.0f;
            a.x = epilogue_op(a.x, bb[0], act); a.y = epilogue_op(a.y, bb[1], act);
            a.z = epilogue_op(a.z, bb[2], act); a.w = epilogue_op(a.w, bb[3], act);
            b.x = epilogue_op(b.x, bb[4], act); b.y = epilogue_op(b.y, bb[5], act);
            b.z = epilogue_op(b.z, bb[6], act); b.w = epilogue_op(b.w, bb[7], act);
        }
        if (residual != nullptr) {   // plain loads: R may be C, read here before this thread writes it
            float rr[8];
            const uint16_t* rsrc = residual + row * ldr + col;
            if (col + 8 <= N) {
                const uint4 x = *reinterpret_cast<const uint4*>(rsrc);
                const uint32_t w4[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
                for (int h = 0; h < 4; ++h) {
                    rr[2 * h] = bf16_bits_to_float(static_cast<uint16_t>(w4[h] & 0xFFFFu));
                    rr[2 * h + 1] = bf16_bits_to_float(static_cast<uint16_t>(w4[h] >> 16));
                }
            } else {
#pragma unroll
                for (int e = 0; e < 8; ++e) rr[e] = col + e < N ? bf16_bits_to_float(rsrc[e]) : 0.0f;
            }
            a.x += rr[0]; a.y += rr[1]; a.z += rr[2]; a.w += rr[3];
            b.x += rr[4]; b.y += rr[5]; b.z += rr[6]; b.w += rr[7];
        }
        const uint32_t w0 = pack_bf16x2_rn(__float_as_uint(a.x), __float_as_uint(a.y));
        const uint32_t w1 = pack_bf16x2_rn(__float_as_uint(a.z), __float_as_uint(a.w));
        const uint32_t w2 = pack_bf16x2_rn(__float_as_uint(b.x), __float_as_uint(b.y));
        const uint32_t w3 = pack_bf16x2_rn(__float_as_uint(b.z), __float_as_uint(b.w));
        uint16_t* dst = C + row * ldc + col;
        if (col + 8 <= N) {
            *reinterpret_cast<uint4*>(dst) = make_uint4(w0, w1, w2, w3);   // 16-byte aligned: ldc, col % 8 == 0
        } else {
            const uint32_t w[4] = {w0, w1, w2, w3};
            for (int e = 0; col + e < N; ++e)
                dst[e] = static_cast<uint16_t>((e & 1) ? (w[e >> 1] >> 16) : (w[e >> 1] & 0xFFFFu));
        }
    }
}

// MXFP8 scale blocks. The caller's scales are row-major, one byte per 32 K
// elements (sa: M × kb_total, row stride ldsa; sb: N × kb_total, ldsb). The
// kernel needs, per (tile, 128-element K stage), 512-byte blocks whose byte
// r·16 + q·4 + j holds the scale of row 32·q + r (of a 128-row group) and K
// block 4·stage + j: one block per 128-row group of A and `b_groups` blocks
// for the B rows of an N tile of `tile_n` rows. Rows or K blocks outside the
// matrix get 0 (2^-127; the operands there are zero). A CTA of 32·b_groups
// threads builds one (tile, stage) atom per step: A atoms first, then B
// atoms; thread `line` writes the 16-byte line r = line % 32 of block
// line / 32 (4 rows × the 4 scales of the stage), so a warp's stores are one
// contiguous 512-byte block. `words`: every row's 4 scales of a stage are one
// aligned 32-bit word (scale pointers and strides multiples of 4, kb_total a
// multiple of 4), read with one load instead of four.
__global__ void mx_scale_blocks_kernel(const uint8_t* __restrict__ sa, int64_t ldsa, const uint8_t* __restrict__ sb,
                                       int64_t ldsb, int M, int N, int kb_total, int tiles_m, int tiles_n,
                                       int k_blocks, int tile_n, int b_groups, int words, uint8_t* __restrict__ out_a,
                                       uint8_t* __restrict__ out_b) {
    griddep_launch_dependents();   // the GEMM (a programmatic dependent) may be scheduled now
    const int64_t atoms_a = static_cast<int64_t>(tiles_m) * k_blocks;
    const int64_t atoms = atoms_a + static_cast<int64_t>(tiles_n) * k_blocks;
    const int line = static_cast<int>(threadIdx.x);
    const int group = line >> 5, r = line & 31;
    for (int64_t atom = blockIdx.x; atom < atoms; atom += gridDim.x) {
        const bool is_a = atom < atoms_a;
        if (is_a && group > 0) continue;   // an A atom is one block (32 lines)
        const int64_t a_local = is_a ? atom : atom - atoms_a;
        const int tile = static_cast<int>(a_local / k_blocks);
        const int stage = static_cast<int>(a_local - static_cast<int64_t>(tile) * k_blocks);
        const uint8_t* src = is_a ? sa : sb;
        const int64_t ld = is_a ? ldsa : ldsb;
        const int rows = is_a ? M : N;
        const int blk0 = 4 * stage;
        uint32_t w[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int local = 128 * group + 32 * q + r;
            const int row = is_a ? 128 * tile + local : tile_n * tile + local;
            uint32_t v = 0;
            if ((is_a || local < tile_n) && row < rows) {
                const uint8_t* p = src + static_cast<int64_t>(row) * ld;
                if (words) {
                    // kb_total is a multiple of 4 here: a word is either in the row or past it
                    // (a K block added to make the count of 128-element blocks even)
                    if (blk0 < kb_total) v = __ldg(reinterpret_cast<const uint32_t*>(p + blk0));
                } else {
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        if (blk0 + j < kb_total) v |= static_cast<uint32_t>(__ldg(p + blk0 + j)) << (8 * j);
                }
            }
            w[q] = v;
        }
        const int64_t out_line = is_a ? atom * 32 + line : a_local * (32 * b_groups) + line;
        uint8_t* dst = (is_a ? out_a : out_b) + out_line * 16;
        *reinterpret_cast<uint4*>(dst) = make_uint4(w[0], w[1], w[2], w[3]);
    }
}

}  // namespace hk
