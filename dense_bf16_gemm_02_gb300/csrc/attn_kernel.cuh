// Attention forward (MHA / GQA)  O = softmax(Q·Kᵀ/√D)·V  for sm_103a.
//
// The operation is the pages' second workload (HipKittens "L2" detail page,
// §3 "Target operation" table, rows "MHA fwd" / "GQA fwd": Q [B, Hq, S, D],
// K and V [B, Hkv, S, D], bf16 in, FP32 accumulation, bf16 out; §5
// "Numerical considerations": online softmax in base 2 with temperature
// sqrt(1/D)·log2(e); §9.3: QKᵀ, row max, exp2, row sum, rescale of the
// running output, P·V, then a final 1/l and the log-sum-exp per row).
// The pages' kernel is an 8-wave ping-pong on AMD matrix cores. This one is
// a Blackwell design:
//
//  * a work item is two 128-row query tiles of one (batch, query head); both
//    tiles share every K/V block that a TMA producer warp streams through a
//    shared-memory ring (128 keys per block, 128-byte swizzle);
//  * the grid is persistent (one CTA per SM) and each CTA walks its work
//    items back to back, so the next item's Q and first K/V blocks load while
//    the current item ends, and launch and set-up are paid once per CTA;
//  * one thread issues tcgen05.mma: S_t = Q_t·K_jᵀ (M=128, N=128, K=D) into
//    Tensor Memory, and O_t += P_t·V_j (M=128, N=D, K=128) with P_t and V_j
//    (MN-major, so V is never transposed) read from shared memory;
//  * two softmax warpgroups, one per query tile, each thread owning one row
//    (optionally at D = 64 two warpgroups per tile, each thread owning half a
//    row: the halves swap partial row maxima and, at the end, row sums through
//    shared memory with a bounded tagged exchange):
//    tcgen05.ld of the row of S, then at once a "S read" signal, so that the
//    MMA thread computes S_t for the next block while this one is still in
//    masking, row max, exp2 on the special function unit and row sum; the
//    bf16 P goes to shared memory (128-byte swizzled, the layout the MMA
//    reads). The softmax of a tile therefore never waits for its own P·V,
//    and the tensor core alternates between the two tiles (the Blackwell
//    counterpart of the pages' ping-pong);
//  * K/V blocks are streamed in the order the MMAs consume them (K of the
//    next block ahead of V of the current one);
//  * the running output is rescaled only when a row's maximum grows by more
//    than 2^8 (the result is the same softmax: P and l share the stale
//    maximum), and the rescale is done in Tensor Memory by the row's thread;
//  * the epilogue multiplies by 1/l, rounds to bf16 (RNE) and stores each
//    row directly; the log-sum-exp goes to an optional fp32 array.
//
// Each KV head's K and V are read by Hq/Hkv query heads; work items are
// numbered head-fastest so the heads of a group run together and share K/V
// in L2.
// Every mbarrier wait is bounded like the GEMM's: a wait that runs out
// records an error in the device status word, the CTA drains and returns.
#pragma once

#include <cuda.h>
#include <cstdint>

#include "ptx.cuh"

#ifndef HK_ATTN_D64_ROW_SPLIT
#define HK_ATTN_D64_ROW_SPLIT 1
#endif

namespace hk {
namespace attn {

constexpr int kTileQ = 128;         // query rows per tile (MMA M)
constexpr int kTiles = 2;           // query tiles per CTA
constexpr int kBlockKV = 128;       // keys per K/V block
constexpr int kSmemLimit = 232448;
constexpr float kRescaleThreshold = 8.0f;   // log2 units: rescale O when the max grows by > 2^8

constexpr uint32_t kErrTmaEmpty = 1u << 8;
constexpr uint32_t kErrMmaKv = 1u << 9;
constexpr uint32_t kErrMmaP = 1u << 10;
constexpr uint32_t kErrMmaO = 1u << 11;
constexpr uint32_t kErrSoftmaxS = 1u << 12;
constexpr uint32_t kErrEpilogueO = 1u << 13;
constexpr uint32_t kErrSoftmaxPair = 1u << 14;

constexpr uint32_t kFlagDropArrive = 0x1u;

template <int kD>
struct AttnGeometry {
    static_assert(kD == 64 || kD == 128, "head dimension 64 or 128");
    // Softmax threads per query row. At D = 64 a block's MMAs take half the
    // time of D = 128's while its softmax work per score is the same; a row can
    // be split over two threads (64 scores each; warps w and w + 8 read the
    // same TMEM lanes) that exchange partial maxima through shared memory
    // (HK_ATTN_D64_ROW_SPLIT = 2). Measured at B16 H64/8 S4096 D64: 848 TFLOP/s
    // split against 943 whole (608 threads leave ~100 registers per thread,
    // and each row then waits for its partner), so rows stay whole.
    static constexpr int kRowSplit = kD == 64 ? HK_ATTN_D64_ROW_SPLIT : 1;
    static constexpr int kCols = kBlockKV / kRowSplit;         // scores of a block per softmax thread
    static constexpr int kSoftmaxWarps = 4 * kTiles * kRowSplit;
    static constexpr int kSoftmaxThreads = 32 * kSoftmaxWarps;
    static constexpr int kWarpTma = kSoftmaxWarps;             // then one MMA-issuing warp per tile
    static constexpr int kWarpMma = kSoftmaxWarps + 1;
    static constexpr int kThreads = 32 * (kSoftmaxWarps + 1 + kTiles);
    static constexpr int kChunks = kD / 64;                   // 128-byte column chunks per row
    static constexpr int kChunkBytes = 128 * 128;             // 128 rows × 128 B (one TMA box)
    static constexpr int kTileBytes = kChunks * kChunkBytes;  // one Q tile, one K block or one V block
    static constexpr int kQBytes = kTiles * kTileBytes;
    // bf16 P of a tile: in its own TMEM columns when they fit (D = 64), else in
    // shared memory as two 64-key chunks (D = 128: O and S fill the TMEM)
    static constexpr bool kPInTmem = kD == 64;
    static constexpr int kPBytes = kPInTmem ? 0 : kTileQ * kBlockKV * 2;
    static constexpr int kSlotsFit = (kSmemLimit - kQBytes - kTiles * kPBytes - 2048) / kTileBytes;
    static constexpr int kSlots = kSlotsFit > 8 ? 8 : kSlotsFit;   // K/V ring
    static_assert(kSlots >= 3, "K/V ring too shallow");
    static constexpr int kOffQ = 0;
    static constexpr int kOffP = kQBytes;
    static constexpr int kOffKV = kOffP + kTiles * kPBytes;
    static constexpr int kOffBars = kOffKV + kSlots * kTileBytes;
    // q_full, kv_full[kSlots], kv_empty[kSlots], s_full[2], s_free[2], p_full[2], o_done[2], q_empty
    static constexpr int kNumBars = 1 + 2 * kSlots + 9;
    static constexpr int kOffTmemHolder = kOffBars + kNumBars * 8;
    // split rows: the halves' exchange slots, [parity][tile][row][half] of
    // (value, tag) pairs (a partial maximum or row sum and its exchange number)
    static constexpr int kOffXchg = (kOffTmemHolder + 16 + 15) & ~15;
    static constexpr int kXchgBytes = kRowSplit > 1 ? 2 * kTiles * kTileQ * kRowSplit * 8 : 0;
    static constexpr int kSmemBytes = kOffXchg + kXchgBytes + 1024;
    static_assert(kSmemBytes <= kSmemLimit, "shared memory");
    // TMEM columns: O_0, O_1 (kD each), then S_0, S_1 (128 each), then (D = 64)
    // P_0, P_1 (64 each: two bf16 per column)
    static constexpr int kColO = 0;
    static constexpr int kColS = 2 * kD;
    static constexpr int kColP = 2 * kD + 2 * kBlockKV;
    static_assert(!kPInTmem || kColP + 2 * (kBlockKV / 2) <= 512, "TMEM");
    static constexpr int kTmemCols = 512;
    static constexpr uint32_t kIdescS = idesc_bf16_f32(kTileQ, kBlockKV);
    static constexpr uint32_t kIdescPV = idesc_bf16_f32(kTileQ, kD) | (1u << 16);   // B (V) MN-major
};

// Ring position of each K/V block in the order the MMAs use them:
// K_0, then (K_{j+1}, V_j) for j = 0 .. n-2, then V_{n-1}.
__device__ __forceinline__ int pos_k(int j) { return j == 0 ? 0 : 2 * j - 1; }
__device__ __forceinline__ int pos_v(int j, int n) { return j + 1 < n ? 2 * j + 2 : 2 * n - 1; }

struct AttnParams {
    int32_t B, Hq, Hkv, S;
    int32_t causal;
    int32_t q_pairs;          // ceil(S / 256): work items per (batch, query head)
    int32_t n_items;          // B * Hq * q_pairs
    int32_t kv_blocks;        // ceil(S / 128)
    float scale_log2;         // log2(e) / sqrt(D)
    uint16_t* O;              // [B, Hq, S, D] bf16
    float* lse;               // [B, Hq, S] natural-log sum of exp of the scaled scores, or null
    uint32_t* status;         // [0]: error bits (sticky), [1]: launch id that aborted
    uint32_t launch_id;
    uint32_t flags;
    uint64_t timeout_ns;
};

__device__ __forceinline__ bool attn_aborted(const AttnParams& p) {
    return *reinterpret_cast<volatile uint32_t*>(p.status + 1) == p.launch_id;
}

// Bounded waits. On the S -> softmax -> P·V chain a wait polls with
// non-suspending probes: a suspended mbarrier wait was measured to resume
// several hundred cycles after its phase completed. The TMA producer, whose
// waits are off that chain, lets the hardware suspend it instead, so that it
// takes no issue slots from the softmax warps. The polling loop is inline (an
// out-of-line call would save and restore the caller's live registers through
// local memory on every wait); the clock is read every 4096 probes (or after
// each suspension), and only a wait that has lasted 20 µs calls out to check
// the launch's abort flag (a global load) and the time limit.
enum class Wait { kPoll, kSuspend };

// Returns true when the wait must give up (this launch was aborted, or the
// time limit ran out; then it records `code` and aborts the launch).
__device__ __noinline__ bool attn_wait_expired(const AttnParams& p, uint64_t waited_ns, uint32_t code) {
    if (attn_aborted(p)) return true;
    if (waited_ns <= p.timeout_ns) return false;
    atomicOr(p.status, code);
    atomicExch(p.status + 1, p.launch_id);
    __threadfence();
    return true;
}

__device__ __forceinline__ bool attn_wait(const AttnParams& p, uint32_t bar, uint32_t parity, uint32_t code,
                                          Wait mode = Wait::kPoll) {
    uint64_t t0 = 0;
    for (uint32_t it = 1;; ++it) {
        bool done;
        if (mode == Wait::kSuspend) done = mbar_try_wait_suspend(bar, parity, 20000);
        else done = mbar_test_wait(bar, parity);
        if (done) return true;
        if (mode == Wait::kSuspend || (it & 4095u) == 0) {
            const uint64_t now = global_timer_ns();
            if (t0 == 0) t0 = now;
            else if (now - t0 >= 20000 && attn_wait_expired(p, now - t0, code)) return false;
        }
    }
}

// Lane 0 waits; the result is broadcast and every lane then observes the
// completed phase itself.
__device__ __forceinline__ bool attn_wait_warp(const AttnParams& p, uint32_t bar, uint32_t parity, uint32_t code) {
    uint32_t ok = 0;
    if (lane_id() == 0) ok = attn_wait(p, bar, parity, code) ? 1u : 0u;
    ok = __shfl_sync(0xffffffffu, ok, 0);
    if (ok) (void)mbar_test_wait(bar, parity);
    __syncwarp();
    return ok != 0;
}

// K/V blocks query tile `row0` needs: all of them, or (causal) those up to
// the block holding the tile's last row. 0 for a tile entirely past S.
__device__ __forceinline__ int tile_blocks(const AttnParams& p, int row0) {
    if (row0 >= p.S) return 0;
    if (!p.causal) return p.kv_blocks;
    const int last = row0 / kBlockKV + 1;
    return last < p.kv_blocks ? last : p.kv_blocks;
}

// One work item: two query tiles (256 rows) of one (batch, query head).
// Items are numbered head-fastest, so the query heads of one KV group run
// side by side; causal: the longest rows first.
struct AttnItem {
    int bh, kvh, q0, n_t0, n_t1, n_all;
};

__device__ __forceinline__ AttnItem attn_item(const AttnParams& p, int w) {
    AttnItem it;
    const int bh_count = p.B * p.Hq;
    const int slot_q = w / bh_count;
    it.bh = w - slot_q * bh_count;
    const int qp = p.causal ? p.q_pairs - 1 - slot_q : slot_q;
    const int b = it.bh / p.Hq;
    const int h = it.bh - b * p.Hq;
    it.kvh = b * p.Hkv + h / (p.Hq / p.Hkv);
    it.q0 = qp * (kTiles * kTileQ);
    it.n_t0 = tile_blocks(p, it.q0);
    it.n_t1 = tile_blocks(p, it.q0 + kTileQ);
    it.n_all = it.n_t0 > it.n_t1 ? it.n_t0 : it.n_t1;
    return it;
}

template <int kD>
__global__ void __launch_bounds__(AttnGeometry<kD>::kThreads, 1)
attn_fwd_kernel(const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_k,
                const __grid_constant__ CUtensorMap tmap_v, const AttnParams p) {
    using G = AttnGeometry<kD>;
    constexpr int kWarpTma = G::kWarpTma;
    constexpr int kWarpMma = G::kWarpMma;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* const smem = smem_raw + (base - raw);

    const uint32_t warp = threadIdx.x >> 5;
    const uint32_t lane = lane_id();

    // Persistent: CTA c takes work items c, c + G, c + 2G, ... (G = gridDim.x).
    // Barrier phases run on across items: the K/V ring's as a slot index and a
    // phase bit, S/P/O's of each tile as the parity of its blocks so far (state
    // that stays bounded however many items a CTA takes).
    const uint32_t q_full = base + G::kOffBars;
    auto kv_full = [&](int s) { return base + G::kOffBars + 8u * (1 + s); };
    auto kv_empty = [&](int s) { return base + G::kOffBars + 8u * (1 + G::kSlots + s); };
    auto s_full = [&](int t) { return base + G::kOffBars + 8u * (1 + 2 * G::kSlots + t); };
    auto s_free = [&](int t) { return base + G::kOffBars + 8u * (3 + 2 * G::kSlots + t); };
    auto p_full = [&](int t) { return base + G::kOffBars + 8u * (5 + 2 * G::kSlots + t); };
    auto o_done = [&](int t) { return base + G::kOffBars + 8u * (7 + 2 * G::kSlots + t); };
    const uint32_t q_empty = base + G::kOffBars + 8u * (9 + 2 * G::kSlots);
    auto p_smem = [&](int t) { return base + G::kOffP + static_cast<uint32_t>(t) * G::kPBytes; };
    auto slot_addr = [&](int s) { return base + G::kOffKV + static_cast<uint32_t>(s) * G::kTileBytes; };
    const uint32_t tmem_holder = base + G::kOffTmemHolder;
    const int first_item = static_cast<int>(blockIdx.x);
    const int item_step = static_cast<int>(gridDim.x);

    if (threadIdx.x == 0) {
        mbar_init(q_full, 1);
        mbar_init(q_empty, kTiles);   // each tile's MMA issuer, once its last S of the item is done
        for (int s = 0; s < G::kSlots; ++s) {
            mbar_init(kv_full(s), 1);
            mbar_init(kv_empty(s), kTiles);   // each tile's issuer arrives once per K/V position
        }
        for (int t = 0; t < kTiles; ++t) {
            mbar_init(s_full(t), 1);
            mbar_init(s_free(t), 4 * 32 * G::kRowSplit);   // every softmax thread of the tile
            mbar_init(p_full(t), 4 * 32 * G::kRowSplit);
            mbar_init(o_done(t), 1);
        }
        fence_mbar_init_cluster();
    }
    if (warp == kWarpTma && lane == 0) {
        prefetch_tensor_map(&tmap_q);
        prefetch_tensor_map(&tmap_k);
        prefetch_tensor_map(&tmap_v);
    }
    if (warp == kWarpMma) {
        tmem_alloc_one(tmem_holder, G::kTmemCols);
        tmem_relinquish_one();
    }
    if constexpr (G::kXchgBytes > 0) {   // exchange tags start at 0 (the first exchange is number 1)
        for (int i = static_cast<int>(threadIdx.x); i < G::kXchgBytes / 4; i += static_cast<int>(blockDim.x))
            reinterpret_cast<volatile uint32_t*>(smem + G::kOffXchg)[i] = 0u;
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem_base = *reinterpret_cast<volatile uint32_t*>(smem + G::kOffTmemHolder);
    bool abort_seen = false;

    if (warp == kWarpTma) {
        // ------------------------------------------------ TMA producer --
        if (lane == 0) {
            int slot = 0;          // K/V ring slot of the next position
            uint32_t ring_ph = 0;  // its phase: flips each time the ring wraps
            int li = 0;      // items done by this CTA
            for (int w = first_item; w < p.n_items && !abort_seen; w += item_step, ++li) {
                const AttnItem it = attn_item(p, w);
                // Q of this item once both issuers have finished the previous item's S
                if (li > 0 && !attn_wait(p, q_empty, (li - 1) & 1, kErrTmaEmpty, Wait::kSuspend)) {
                    abort_seen = true;
                    break;
                }
                const int tiles = it.n_t1 > 0 ? 2 : 1;
                mbar_arrive_expect_tx(q_full, static_cast<uint32_t>(tiles * G::kTileBytes));
                for (int t = 0; t < tiles; ++t)
                    for (int c = 0; c < G::kChunks; ++c)
                        tma_load_3d(base + G::kOffQ + t * G::kTileBytes + c * G::kChunkBytes, &tmap_q, c * 64,
                                    it.q0 + t * kTileQ, it.bh, q_full);
                for (int u = 0; u < 2 * it.n_all && !abort_seen; ++u) {
                    const int s = slot;
                    const uint32_t parity = ring_ph ^ 1u;
                    if (++slot == G::kSlots) {
                        slot = 0;
                        ring_ph ^= 1u;
                    }
                    if (!attn_wait(p, kv_empty(s), parity, kErrTmaEmpty, Wait::kSuspend)) {
                        abort_seen = true;
                        break;
                    }
                    if ((p.flags & kFlagDropArrive) && li == 0 && u == 0) continue;   // test hook: never fill the first slot
                    // position u of the item's consumption order: K_0, (K_{j+1}, V_j)..., V_{n-1}
                    bool is_k;
                    int blk;
                    if (u == 0) {
                        is_k = true;
                        blk = 0;
                    } else if (u - 1 < 2 * (it.n_all - 1)) {
                        is_k = ((u - 1) & 1) == 0;
                        blk = is_k ? (u - 1) / 2 + 1 : (u - 1) / 2;
                    } else {
                        is_k = false;
                        blk = it.n_all - 1;
                    }
                    mbar_arrive_expect_tx(kv_full(s), G::kTileBytes);
                    for (int c = 0; c < G::kChunks; ++c)
                        tma_load_3d(slot_addr(s) + c * G::kChunkBytes, is_k ? &tmap_k : &tmap_v, c * 64,
                                    blk * kBlockKV, it.kvh, kv_full(s));
                }
            }
        }
    } else if (warp == kWarpMma || warp == kWarpMma + 1) {
        // ------------------------------------------- MMA issue, one warp per tile --
        // A tcgen05.mma holds its issuing thread for about the time it
        // computes; with one issuer per tile, each issuer's barrier waits and
        // commits overlap the other tile's MMAs. Both issuers arrive once on
        // every K/V position and on q_empty for every item (a plain arrive,
        // after the data landed, for what their tile does not use), so the
        // barrier counts stay fixed across items.
        const int t = static_cast<int>(warp) - kWarpMma;
        if (lane == 0) {
            auto wait = [&](uint32_t bar, uint32_t parity, uint32_t code) {
                if (abort_seen) return false;
                if (!attn_wait(p, bar, parity, code)) abort_seen = true;
                return !abort_seen;
            };
            int s0 = 0;          // ring slot of the item's first K/V position
            uint32_t ph0 = 0;    // and its phase
            auto kv_slot = [&](int u) { return (s0 + u) % G::kSlots; };
            auto kv_parity = [&](int u) { return ph0 ^ static_cast<uint32_t>(((s0 + u) / G::kSlots) & 1); };
            const uint32_t qa = base + G::kOffQ + t * G::kTileBytes;
            const uint32_t s_tmem = tmem_base + G::kColS + t * kBlockKV;
            const uint32_t o_tmem = tmem_base + G::kColO + t * kD;
            const uint32_t pa = p_smem(t);
            const uint32_t p_tmem = tmem_base + G::kColP + t * (kBlockKV / 2);
            uint32_t jp = 0;       // parity of this tile's blocks in earlier items
            bool any_block = false;  // has this tile had a block before (then S waits for s_free)
            int li = 0;
            for (int w = first_item; w < p.n_items && !abort_seen; w += item_step, ++li) {
                const AttnItem it = attn_item(p, w);
                const int n = t ? it.n_t1 : it.n_t0;
                const int n_all = it.n_all;
                if (!wait(q_full, li & 1, kErrMmaKv)) break;
                // S_t = Q_t · K_jᵀ of block j (item position u), once the softmax has
                // read this tile's previous S; the last S of the item releases Q
                auto issue_s = [&](int j, int u) {
                    if ((j > 0 || any_block) && !wait(s_free(t), jp ^ static_cast<uint32_t>((j - 1) & 1), kErrMmaP))
                        return false;
                    if (!wait(kv_full(kv_slot(u)), kv_parity(u), kErrMmaKv)) return false;
                    tc_fence_after_sync();
                    const uint32_t ka = slot_addr(kv_slot(u));
#pragma unroll
                    for (int kk = 0; kk < kD / 16; ++kk) {
                        const uint32_t off = (kk >> 2) * G::kChunkBytes + (kk & 3) * 32;
                        mma_bf16_one(s_tmem, smem_desc_kmajor_sw128(qa + off), smem_desc_kmajor_sw128(ka + off),
                                     G::kIdescS, kk > 0 ? 1u : 0u);
                    }
                    mma_commit_one(s_full(t));
                    mma_commit_one(kv_empty(kv_slot(u)));
                    if (j == n - 1) mma_commit_one(q_empty);
                    return true;
                };
                if (n == 0) {
                    mbar_arrive(q_empty);   // this tile has no rows in the item
                } else if (issue_s(0, 0)) {
                    for (int j = 0; j < n && !abort_seen; ++j) {
                        if (j + 1 < n && !issue_s(j + 1, pos_k(j + 1))) break;
                        // O_t += P_t · V_j once P_t is ready
                        const int uv = pos_v(j, n_all);
                        if (!wait(kv_full(kv_slot(uv)), kv_parity(uv), kErrMmaKv)) break;
                        if (!wait(p_full(t), jp ^ static_cast<uint32_t>(j & 1), kErrMmaP)) break;
                        tc_fence_after_sync();
                        const uint32_t va = slot_addr(kv_slot(uv));
#pragma unroll
                        for (int kk = 0; kk < kBlockKV / 16; ++kk) {
                            const uint64_t vdesc = smem_desc_mnmajor(va + kk * 2048, 128, G::kChunkBytes);
                            const uint32_t acc = (j == 0 && kk == 0) ? 0u : 1u;
                            if constexpr (G::kPInTmem)
                                mma_bf16_ts_one(o_tmem, p_tmem + kk * 8, vdesc, G::kIdescPV, acc);
                            else
                                mma_bf16_one(o_tmem,
                                             smem_desc_kmajor_sw128(pa + (kk >> 2) * G::kChunkBytes + (kk & 3) * 32),
                                             vdesc, G::kIdescPV, acc);
                        }
                        mma_commit_one(o_done(t));
                        mma_commit_one(kv_empty(kv_slot(uv)));
                    }
                }
                // K/V positions of blocks this tile does not use: arrive once each has landed
                auto release = [&](int u) {
                    if (!wait(kv_full(kv_slot(u)), kv_parity(u), kErrMmaKv)) return false;
                    mbar_arrive(kv_empty(kv_slot(u)));
                    return true;
                };
                for (int j = n; j < n_all && !abort_seen; ++j)
                    if (!release(pos_k(j)) || !release(pos_v(j, n_all))) break;
                ph0 ^= static_cast<uint32_t>(((s0 + 2 * n_all) / G::kSlots) & 1);
                s0 = (s0 + 2 * n_all) % G::kSlots;
                jp ^= static_cast<uint32_t>(n & 1);
                any_block = any_block || n > 0;
            }
        }
    } else {
        // ------------------------------------------ softmax warpgroups --
        // Warp w: tile (w / 4) % 2, TMEM lane quarter w % 4 (the quarter a warp
        // may access), and with split rows half w / 8 of each row's scores.
        constexpr int kSplit = G::kRowSplit;
        constexpr int kCols = G::kCols;
        const int t = static_cast<int>(warp >> 2) & 1;
        const uint32_t quarter = warp & 3u;
        const int half = kSplit > 1 ? static_cast<int>(warp >> 3) : 0;
        const int r = static_cast<int>(quarter * 32 + lane);
        const uint32_t lane_off = (quarter * 32u) << 16;
        const uint32_t s_addr = tmem_base + lane_off + G::kColS + t * kBlockKV + half * kCols;
        const uint32_t o_addr = tmem_base + lane_off + G::kColO + t * kD;
        const float c = p.scale_log2;
        // Split rows: the two threads of a row swap a value (partial maximum, row
        // sum) through shared memory. Each writes its value, then the exchange's
        // number as a tag, and polls (bounded) for its partner's tag: no hardware
        // barrier, so a half that gives up on a wait cannot leave the other
        // stuck. Slots alternate by exchange parity: a half writes a slot again
        // only after reading its partner's next tag, written after the partner
        // read this slot.
        uint32_t xn = 0;   // exchanges so far (the same sequence in both halves)
        auto exchange = [&](float mine, float& theirs) -> bool {
            volatile uint32_t* const x = reinterpret_cast<volatile uint32_t*>(smem + G::kOffXchg) +
                                         2 * ((((xn & 1) * kTiles + t) * kTileQ + r) * kSplit);
            const uint32_t tag = ++xn;
            x[2 * half] = __float_as_uint(mine);
            __threadfence_block();
            x[2 * half + 1] = tag;
            uint64_t t0 = 0;
            for (uint32_t it = 1; x[2 * (half ^ 1) + 1] != tag; ++it) {
                if ((it & 1023u) == 0) {
                    const uint64_t now = global_timer_ns();
                    if (t0 == 0) t0 = now;
                    else if (now - t0 >= 20000 && attn_wait_expired(p, now - t0, kErrSoftmaxPair)) return false;
                }
            }
            __threadfence_block();
            theirs = __uint_as_float(x[2 * (half ^ 1)]);
            return true;
        };
        uint32_t jp = 0;   // parity of this tile's blocks in earlier items
        for (int w = first_item; w < p.n_items && !abort_seen; w += item_step) {
            int n, key_end;
            {
                const AttnItem it = attn_item(p, w);
                n = t ? it.n_t1 : it.n_t0;
                const int q = it.q0 + t * kTileQ + r;       // this thread's query row
                key_end = p.causal ? (q + 1 < p.S ? q + 1 : p.S) : p.S;   // keys [0, key_end) are visible
            }
            float m = 0.0f;   // running max of the scaled scores (log2 units) used for P
            float l = 0.0f;   // running sum of P (of this thread's columns)
            for (int j = 0; j < n; ++j) {
                const uint32_t par = jp ^ static_cast<uint32_t>(j & 1);   // phase of this block's barriers
                if (!attn_wait_warp(p, s_full(t), par, kErrSoftmaxS)) {
                    abort_seen = true;
                    break;
                }
                tc_fence_after_sync();
                uint32_t v[kCols];
                tmem_load_32cols_at<0>(s_addr + 0, v);
                tmem_load_32cols_at<32>(s_addr + 32, v);
                if constexpr (kCols == 128) {
                    tmem_load_32cols_at<64 % kCols>(s_addr + 64, v);
                    tmem_load_32cols_at<96 % kCols>(s_addr + 96, v);
                }
                tmem_wait_ld();
                // S is in registers: the MMA thread may compute the next block's S here
                tc_fence_before_sync();
                mbar_arrive(s_free(t));
                const int lim = key_end - j * kBlockKV - half * kCols;     // visible columns of this thread's share
                if (lim < kCols) {
#pragma unroll
                    for (int e = 0; e < kCols; ++e)
                        if (e >= lim) v[e] = __float_as_uint(-INFINITY);
                }
                // row max: independent chains of three-input maxima, then a tree
                constexpr int kChains = kCols / 16;
                float acc[kChains];
#pragma unroll
                for (int k = 0; k < kChains; ++k) {
                    const int e0 = 16 * k;
                    float a = fmax3(__uint_as_float(v[e0]), __uint_as_float(v[e0 + 1]), __uint_as_float(v[e0 + 2]));
#pragma unroll
                    for (int e = 3; e < 15; e += 2)
                        a = fmax3(a, __uint_as_float(v[e0 + e]), __uint_as_float(v[e0 + e + 1]));
                    acc[k] = fmaxf(a, __uint_as_float(v[e0 + 15]));
                }
                float mx;
                if constexpr (kChains == 8)
                    mx = fmax3(fmax3(acc[0], acc[1], acc[2]), fmax3(acc[3], acc[4], acc[5]), fmaxf(acc[6], acc[7]));
                else
                    mx = fmaxf(fmax3(acc[0], acc[1], acc[2]), acc[3]);
                if constexpr (kSplit > 1) {   // the row's maximum over both halves
                    float other;
                    if (!exchange(mx, other)) {
                        abort_seen = true;
                        break;
                    }
                    mx = fmaxf(mx, other);
                }
                const float m_blk = mx * c;
                float alpha = 1.0f;
                if (j == 0) {
                    m = m_blk;
                } else if (m_blk > m + kRescaleThreshold) {
                    alpha = ex2_approx(m - m_blk);
                    m = m_blk;
                    l *= alpha;
                }
                // P = 2^(s·c - m) in bf16; the scale-and-shift and the row sum run on packed pairs
                const uint64_t c2 = f32x2(c, c);
                const uint64_t nm2 = f32x2(-m, -m);
                uint64_t sum2[4] = {0, 0, 0, 0};
                uint32_t pk[kCols / 2];
                // D = 64, whole rows (P in TMEM): the first half of the row's P is stored,
                // asynchronously, while the second half is computed, and the wait for the
                // previous P·V (single P buffer) and the rescale of O come before that
                // store (measured: 910 -> 930 TFLOP/s at B16 H64/8 S4096 D64, causal equal)
                constexpr bool kEarlyP = G::kPInTmem && kCols == 128;
                constexpr int kFirstPairs = kEarlyP ? kCols / 4 : kCols / 2;
                // rescale the running output (warp-wide when any row of the warp needs it; with
                // split rows each half rescales its half of O's columns); the stores complete
                // at the caller's tcgen05.wait::st
                auto rescale_o = [&]() {
                    if (__any_sync(0xffffffffu, alpha != 1.0f)) {
#pragma unroll
                        for (int cc = 0; cc < kD / 32 / kSplit; ++cc) {
                            const uint32_t oc = o_addr + 32 * (cc + half * (kD / 32 / kSplit));
                            uint32_t o[32];
                            tmem_load_32cols(oc, o);
                            tmem_wait_ld();
#pragma unroll
                            for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
                            tmem_store_32cols(oc, o);
                        }
                    }
                };
                // P of the score pair e (keys 2e, 2e + 1) and its share of the row sum
                auto exp_pair = [&](int e) {
                    const uint64_t x =
                        ffma2(f32x2(__uint_as_float(v[2 * e]), __uint_as_float(v[2 * e + 1])), c2, nm2);
                    float x0, x1;
                    f32x2_split(x, x0, x1);
                    const float p0 = ex2_approx(x0);
                    const float p1 = ex2_approx(x1);
                    sum2[e & 3] = fadd2(sum2[e & 3], f32x2(p0, p1));
                    pk[e] = pack_bf16x2_rn(__float_as_uint(p0), __float_as_uint(p1));
                };
#pragma unroll
                for (int e = 0; e < kFirstPairs; ++e) exp_pair(e);
                const uint32_t p_addr_e = tmem_base + lane_off + G::kColP + t * (kBlockKV / 2) + half * (kCols / 2);
                if constexpr (kEarlyP) {
                    if (j > 0 && !attn_wait_warp(p, o_done(t), par ^ 1u, kErrEpilogueO)) {
                        abort_seen = true;
                        break;
                    }
                    tc_fence_after_sync();
                    rescale_o();
                    tmem_store_32cols(p_addr_e, *reinterpret_cast<const uint32_t(*)[32]>(&pk[0]));
                }
#pragma unroll
                for (int e = kFirstPairs; e < kCols / 2; ++e) exp_pair(e);
                {
                    const uint64_t s01 = fadd2(fadd2(sum2[0], sum2[1]), fadd2(sum2[2], sum2[3]));
                    float lo, hi;
                    f32x2_split(s01, lo, hi);
                    l += lo + hi;
                }
                if constexpr (kEarlyP) {
                    tmem_store_32cols(p_addr_e + 32, *reinterpret_cast<const uint32_t(*)[32]>(&pk[32]));
                    tmem_wait_st();
                } else {
                    // P·V of the previous block must be done before its P is overwritten and O rescaled
                    if (j > 0 && !attn_wait_warp(p, o_done(t), par ^ 1u, kErrEpilogueO)) {
                        abort_seen = true;
                        break;
                    }
                    tc_fence_after_sync();
                    rescale_o();
                    tmem_wait_st();
                    if constexpr (G::kPInTmem) {
                        // this thread's keys of P into the tile's own TMEM columns (two bf16 per column)
                        const uint32_t p_addr = tmem_base + lane_off + G::kColP + t * (kBlockKV / 2) + half * (kCols / 2);
#pragma unroll
                        for (int cc = 0; cc < kCols / 64; ++cc)
                            tmem_store_32cols(p_addr + 32 * cc, *reinterpret_cast<const uint32_t(*)[32]>(&pk[32 * cc]));
                        tmem_wait_st();
                    } else {
                        // this row of P into the 128-byte-swizzled K-major tile the MMA reads:
                        // keys [64 h, 64 h + 64) in chunk h, 16-byte unit x of row r at unit x ^ (r % 8)
                        static_assert(kSplit == 1 || G::kPInTmem, "P in shared memory with whole rows per thread");
#pragma unroll
                        for (int hh = 0; hh < 2; ++hh) {
                            const uint32_t row = p_smem(t) + hh * G::kChunkBytes + static_cast<uint32_t>(r) * 128u;
#pragma unroll
                            for (int x = 0; x < 8; ++x)
                                st_shared_v4(row + ((static_cast<uint32_t>(x) ^ (static_cast<uint32_t>(r) & 7u)) << 4),
                                             pk[32 * hh + 4 * x], pk[32 * hh + 4 * x + 1], pk[32 * hh + 4 * x + 2],
                                             pk[32 * hh + 4 * x + 3]);
                        }
                        fence_proxy_async_smem();
                    }
                }
                tc_fence_before_sync();
                mbar_arrive(p_full(t));
            }
            // -------------------------------------------------- epilogue --
            // (reading O here, before this warp publishes the next item's first P,
            // orders these reads before the P·V that overwrites O)
            if (!abort_seen && n > 0) {
                if (!attn_wait_warp(p, o_done(t), jp ^ static_cast<uint32_t>((n - 1) & 1), kErrEpilogueO)) {
                    abort_seen = true;
                } else {
                    tc_fence_after_sync();
                    float l_other = 0.0f;
                    if constexpr (kSplit > 1) abort_seen = !exchange(l, l_other);   // the row sum over both halves
                    l += l_other;
                    const AttnItem it = attn_item(p, w);
                    const int q = abort_seen ? p.S : it.q0 + t * kTileQ + r;   // no stores after a failed exchange
                    const float inv_l = 1.0f / l;
                    uint16_t* out = p.O + (static_cast<int64_t>(it.bh) * p.S + q) * kD;
#pragma unroll
                    for (int cc = 0; cc < kD / 32 / kSplit; ++cc) {
                        const int col = 32 * (cc + half * (kD / 32 / kSplit));
                        uint32_t o[32];
                        tmem_load_32cols(o_addr + col, o);
                        tmem_wait_ld();
                        uint32_t pk[16];
#pragma unroll
                        for (int e = 0; e < 16; ++e)
                            pk[e] = pack_bf16x2_rn(__float_as_uint(__uint_as_float(o[2 * e]) * inv_l),
                                                   __float_as_uint(__uint_as_float(o[2 * e + 1]) * inv_l));
                        if (q < p.S) {
#pragma unroll
                            for (int w4 = 0; w4 < 4; ++w4)
                                st_global_v4(out + col + 8 * w4, pk[4 * w4], pk[4 * w4 + 1], pk[4 * w4 + 2],
                                             pk[4 * w4 + 3]);
                        }
                    }
                    if (p.lse != nullptr && q < p.S && half == 0)
                        p.lse[static_cast<int64_t>(it.bh) * p.S + q] = (m + log2f(l)) * 0.69314718055994531f;
                    tc_fence_before_sync();
                }
            }
            jp ^= static_cast<uint32_t>(n & 1);
        }
    }

    if (abort_seen || attn_aborted(p)) {
        // let copies and MMAs that were already issued land before teardown
        for (int i = 0; i < 200; ++i) __nanosleep(1000);
    }
    tc_fence_before_sync();
    __syncthreads();
    if (warp == kWarpMma) {
        tc_fence_after_sync();
        tmem_dealloc_one(tmem_base, G::kTmemCols);
    }
}

}  // namespace attn
}  // namespace hk
