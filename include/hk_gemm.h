/*
 * hk_gemm — dense BF16 GEMM  C = A · Bᵀ  for NVIDIA GB300 (sm_103a).
 *
 * The operation is the one the HipKittens pages measure most ("L2" detail
 * page, §3 "Target operation" table, row "BF16 GEMM": bf16 inputs, FP32
 * accumulation, bf16 output; §7 and §9.2 describe its hot loop as the
 * "ABt" product, so the second operand is stored N×K and used transposed;
 * §3 "Launch config" fixes the 256×256 output tile and 64-wide K step).
 *
 * Semantics of every entry point that computes:
 *
 *     C[i*ldc + j] = bf16_rne( Σ_{k<K}  A[i*lda + k] · B[j*ldb + k] )
 *
 * for 0 ≤ i < M, 0 ≤ j < N, with products and sums in FP32 on the tensor
 * cores (the order of the FP32 additions is unspecified), rounded once to
 * bf16 with round-to-nearest-even. There is no alpha/beta and no
 * accumulation into C; entries of C outside the M×N window (the padding
 * between N and ldc) are never written.
 *
 * Layout: A is M×K row-major, B is N×K row-major ("TN"), C is M×N row-major,
 * all bf16 (2 bytes per element, passed as raw device pointers). Leading
 * dimensions are in ELEMENTS.
 *
 * Ownership: A, B, C and any workspace are caller-owned DEVICE memory on the
 * device the call runs on. The library never frees them. C must not overlap
 * A or B.
 *
 * Alignment (a requirement of the Tensor Memory Accelerator): A, B and C
 * must be 16-byte aligned and lda, ldb, ldc multiples of 8, else
 * HK_ERR_MISALIGNED.
 *
 * Edge values: M == 0 or N == 0 -> HK_OK, nothing launched (pointers may be
 * NULL). K == 0 -> C (M×N) is filled with +0. Negative sizes, lda < K,
 * ldb < K, ldc < N or sizes ≥ 2^31 -> HK_ERR_INVALID_ARG.
 *
 * Device: the library runs on compute capability 10.3 (GB300) only; any
 * other device -> HK_ERR_UNSUPPORTED_DEVICE. There is no CPU fallback.
 *
 * Asynchrony: computing calls enqueue work on `stream` (a cudaStream_t; NULL
 * is the legacy default stream) and return without synchronising. Launch
 * failures are returned as HK_ERR_LAUNCH. Every wait inside the kernel is
 * bounded; a wait that runs out sets a device status word, the kernel drains
 * and returns, and the status is read with hk_gemm_plan_device_status or
 * hk_gemm_last_device_status after the stream has been synchronised.
 *
 * Thread safety: plans are immutable after creation and may be run from
 * several host threads at once; hk_gemm_bf16 is thread safe.
 */
#ifndef HK_GEMM_H
#define HK_GEMM_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum hk_status {
    HK_OK = 0,
    HK_ERR_INVALID_ARG = 1,        /* a size, leading dimension or pointer is invalid */
    HK_ERR_MISALIGNED = 2,         /* pointer not 16-byte aligned or ld not a multiple of 8 */
    HK_ERR_UNSUPPORTED_DEVICE = 3, /* not a compute capability 10.3 device */
    HK_ERR_LAUNCH = 4,             /* the CUDA launch (or a CUDA runtime call) failed */
    HK_ERR_TIMEOUT = 5,            /* a bounded wait inside the kernel ran out */
    HK_ERR_WORKSPACE = 6,          /* workspace missing, too small or misaligned */
    HK_ERR_CUDA = 7                /* another CUDA runtime error (see hk_gemm_last_error_string) */
} hk_status;

/* Plan flags (hk_gemm_config.flags). */
#define HK_FLAG_NONE 0u
/* Test only: the producer withholds its arrival on the first shared-memory
 * stage, so a bounded wait on that stage runs out (the MMA issuer's) and
 * the call reports HK_ERR_TIMEOUT through the device status word. No GPU
 * fault is caused. */
#define HK_FLAG_FAULT_DROP_ARRIVE 0x1u
/* Keep the tiles of the last partial round whole (by default, when they fill
 * at most half of the CTA pairs, each runs as two halves of half the tile's
 * width: 256x128 for the 256x256 pair, 256x64 for the 256x128 pair). */
#define HK_FLAG_NO_TAIL_SPLIT 0x2u

/* Fused epilogue activations: C = bf16(act(A·Bᵀ + bias) [+ R]). */
#define HK_ACT_NONE 0
#define HK_ACT_RELU 1               /* max(x, 0) */
#define HK_ACT_GELU 2               /* x·Φ(x) = 0.5·x·(1 + erf(x/√2)) */
#define HK_ACT_SILU 3               /* x·σ(x) = x / (1 + e^(−x)) */

/* Kernel variants (hk_gemm_config.kernel). A "pair" kernel runs on clusters
 * of two CTAs (tcgen05 cta_group::2) with 256-row output tiles; a "single"
 * kernel runs one CTA per output tile of 128 rows and suits M <= 128. The
 * 256x128 and 256x112 pairs (bf16 only) stream a narrower slice of B per
 * pair: for 128 < M <= 256 with few output tiles they fill the GPU without a
 * K split (N = 8192 makes 74 tiles of 112 for the 76 pairs of a GB300, 64 of
 * 128), and its 23 KB stages leave room for a ninth in the ring (the
 * streaming rate of these shapes grows with the bytes in flight). The 256x112
 * pair never runs the last round's tiles as half-width units
 * (HK_FLAG_NO_TAIL_SPLIT is implied). */
#define HK_KERNEL_AUTO 0            /* chosen by the plan's time model: single-CTA kernels for M <= 128, pairs above 384 (E4M3: 128), either between */
#define HK_KERNEL_PAIR_256x256 1
#define HK_KERNEL_SINGLE_128x256 2
#define HK_KERNEL_SINGLE_128x192 3
#define HK_KERNEL_SINGLE_128x128 4
#define HK_KERNEL_SINGLE_128x64 5
#define HK_KERNEL_PAIR_256x128 6
#define HK_KERNEL_PAIR_256x112 7

/* Tuning knobs of a plan. Zero in any field selects the default. */
typedef struct hk_gemm_config {
    int32_t group_m;        /* grouped rasterisation: height of a group in output-tile rows (default 8) */
    int32_t max_clusters;   /* cap on the persistent grid, in work units (CTA pairs or CTAs; default: all that fit) */
    int32_t split_k;        /* K splits per output tile (0: chosen by the plan, which splits only when
                               the tiles do not fill one wave; 1: never; > 1: forced) */
    int32_t kernel;         /* HK_KERNEL_* (default HK_KERNEL_AUTO) */
    uint64_t timeout_ns;    /* limit of each bounded wait in the kernel (default 1 s) */
    uint32_t flags;         /* HK_FLAG_* */
    uint32_t activation;    /* fused epilogue activation, HK_ACT_* (used by hk_gemm_plan_run_epilogue) */
    int32_t input_type;     /* HK_INPUT_BF16 (default) or HK_INPUT_E4M3 (1-byte operands, ld multiples of 16) */
    float alpha;            /* scale applied to the fp32 accumulator before rounding (0: 1.0) */
} hk_gemm_config;

#define HK_INPUT_BF16 0
#define HK_INPUT_E4M3 1

/* What a plan chose (for logging and benchmarks). */
typedef struct hk_gemm_plan_info {
    int64_t M, N, K;
    int32_t kernel;                   /* HK_KERNEL_* actually used */
    int32_t ctas_per_unit;            /* 2 for a pair kernel, 1 for a single-CTA kernel */
    int32_t tile_m, tile_n, tile_k;   /* output tile of one work unit and K step */
    int32_t stages;                   /* depth of the shared-memory ring */
    int32_t num_tiles;                /* output tiles */
    int32_t grid_ctas;                /* CTAs launched */
    int32_t group_m;
    int32_t split_k;
    int32_t kernels_per_run;          /* kernel launches one run enqueues */
    int32_t smem_bytes;               /* dynamic shared memory per CTA */
    size_t workspace_bytes;
    int32_t tail_split_tiles;         /* tiles of the last round run as two half-width units */
    int32_t reserved;
} hk_gemm_plan_info;

typedef struct hk_gemm_plan hk_gemm_plan;

/* One-shot GEMM on the current device: C = bf16(A · Bᵀ).
 * Equivalent to a plan with the default config run with no workspace (the
 * default plan never needs one). The first call on a device creates a small
 * per-device context (a 16-byte device status word) and is therefore not
 * capturable in a CUDA graph; later calls allocate nothing. The plans of
 * recent shapes are kept (a small per-process cache, also used by
 * hk_gemm_bf16_epilogue, hk_gemm_bf16_fused and hk_gemm_fp8_e4m3), and each
 * keeps the tensor maps of its last A, B and C, so a repeated call does no
 * planning and, with the same pointers, no tensor-map encoding. */
hk_status hk_gemm_bf16(const void* A, const void* B, void* C,
                       int64_t M, int64_t N, int64_t K,
                       int64_t lda, int64_t ldb, int64_t ldc, void* stream);

/* Create a plan for one problem shape on `device`. `config` may be NULL.
 * Does all host-side work once: argument checks, device check, tile and
 * schedule choice, and allocates the plan's 16-byte device status word.
 * On success *out owns the plan; free it with hk_gemm_plan_destroy. */
hk_status hk_gemm_plan_create(hk_gemm_plan** out, int64_t M, int64_t N, int64_t K,
                              int64_t lda, int64_t ldb, int64_t ldc, int device,
                              const hk_gemm_config* config);

/* Bytes of device workspace a run needs (0 when no K split is used). With
 * S > 1 splits it holds S fp32 partial matrices (S × M × N', N' = N rounded
 * up to the tile width); a second kernel sums them in split order
 * (deterministic) and writes C. */
size_t hk_gemm_plan_workspace_size(const hk_gemm_plan* plan);

/* Fill *info with what the plan chose. */
hk_status hk_gemm_plan_get_info(const hk_gemm_plan* plan, hk_gemm_plan_info* info);

/* Enqueue one GEMM with the plan's shape on `stream`. `workspace` must hold
 * hk_gemm_plan_workspace_size(plan) bytes, 256-byte aligned (may be NULL when
 * that size is 0); it is scratch, owned by the caller, and must not be used by
 * another run that can overlap this one. The call allocates nothing. */
hk_status hk_gemm_plan_run(const hk_gemm_plan* plan, const void* A, const void* B, void* C,
                           void* workspace, size_t workspace_bytes, void* stream);

/* GEMM with a fused epilogue (the HipKittens pages fuse nothing into their
 * GEMM; this is the cheapest extension once the epilogue stage exists):
 *     C[i,j] = bf16_rne( act( Σ_k A[i,k]·B[j,k] + bias[j] ) )
 * computed in fp32 (accumulator + bias, then the activation) before the one
 * rounding. `bias` is a device vector of N bf16 values, 16-byte aligned, or
 * NULL (no bias); `activation` is an HK_ACT_* code (HK_ERR_INVALID_ARG
 * otherwise). Everything else as hk_gemm_bf16. */
hk_status hk_gemm_bf16_epilogue(const void* A, const void* B, void* C, const void* bias,
                                int64_t M, int64_t N, int64_t K,
                                int64_t lda, int64_t ldb, int64_t ldc,
                                int32_t activation, void* stream);

/* Plan form: the activation is hk_gemm_config.activation of the plan; the
 * bias (or NULL) is given per run. Otherwise as hk_gemm_plan_run. */
hk_status hk_gemm_plan_run_epilogue(const hk_gemm_plan* plan, const void* A, const void* B, void* C,
                                    const void* bias, void* workspace, size_t workspace_bytes,
                                    void* stream);

/* GEMM with a fused epilogue that also adds a residual:
 *     C[i,j] = bf16_rne( act( Σ_k A[i,k]·B[j,k] + bias[j] ) + R[i,j] )
 * in fp32 before the one rounding. The HipKittens "L2" detail page (§8
 * "Deployment context", Fusion scope) keeps the residual add in a separate
 * memory-bound kernel; here it rides in the GEMM's epilogue, which reads R
 * once while the tensor cores work on the next tile. `R` is a device matrix
 * of M×N bf16 values, row-major with leading dimension `ldr` (elements, a
 * multiple of 8 and ≥ N), 16-byte aligned (else HK_ERR_MISALIGNED), or NULL
 * (no residual). R may be C itself (same pointer, ldr == ldc): an in-place
 * update C ← act(A·Bᵀ + bias) + C; any other overlap of R and C is rejected
 * with HK_ERR_INVALID_ARG. `bias` and `activation` as hk_gemm_bf16_epilogue;
 * everything else as hk_gemm_bf16. */
hk_status hk_gemm_bf16_fused(const void* A, const void* B, void* C, const void* bias, const void* R,
                             int64_t M, int64_t N, int64_t K,
                             int64_t lda, int64_t ldb, int64_t ldc, int64_t ldr,
                             int32_t activation, void* stream);

/* Plan form of hk_gemm_bf16_fused: the activation is the plan's
 * hk_gemm_config.activation; bias, R and ldr are given per run (a K split
 * adds bias, activation and R in its reduction kernel). Also for E4M3 plans:
 * alpha, then bias, activation and R. Otherwise as hk_gemm_plan_run. */
hk_status hk_gemm_plan_run_fused(const hk_gemm_plan* plan, const void* A, const void* B, void* C,
                                 const void* bias, const void* R, int64_t ldr,
                                 void* workspace, size_t workspace_bytes, void* stream);

/* FP8 GEMM (the pages' second GEMM: 8-bit floating-point inputs, FP32
 * accumulation, bf16 output), with one scale per operand tensor:
 *     C[i,j] = bf16_rne( (scale_a·scale_b) · Σ_k e4m3(A[i,k])·e4m3(B[j,k]) )
 * A (M×K) and B (N×K) hold E4M3 codes (1 sign, 4 exponent bits with bias 7,
 * 3 fraction bits; no infinities; largest magnitude 448), row-major,
 * K-contiguous; C is bf16 as in hk_gemm_bf16. lda and ldb are in elements
 * (= bytes) and must be multiples of 16, ldc a multiple of 8 (else
 * HK_ERR_MISALIGNED); scale_a·scale_b is formed in double and rounded once
 * to float. The products accumulate in fp32 on the tensor cores
 * (tcgen05.mma kind::f8f6f4). Block-scaled MXFP8 is not provided. */
hk_status hk_gemm_fp8_e4m3(const void* A, const void* B, void* C,
                           int64_t M, int64_t N, int64_t K,
                           int64_t lda, int64_t ldb, int64_t ldc,
                           float scale_a, float scale_b, void* stream);

/* MXFP8 GEMM (the pages' FP8 GEMM row: MXFP8 inputs, FP32 accumulation; a
 * bf16 output here): E4M3 operands whose K dimension is cut into blocks of 32
 * elements, each block of each row scaled by one UE8M0 byte E (value
 * 2^(E-127); 255 is NaN, as in the OCP MX format):
 *     C[i,j] = bf16_rne( Σ_b 2^(SFA[i,b]-127)·2^(SFB[j,b]-127)·Σ_{k in block b} A[i,k]·B[j,k] )
 * A (M×K) and B (N×K) hold E4M3 codes as in hk_gemm_fp8_e4m3 (lda, ldb
 * multiples of 16); SFA (M × K/32) and SFB (N × K/32) hold the scale bytes,
 * row-major with row strides ldsfa, ldsfb ≥ K/32 (bytes, any alignment); C is
 * bf16 as in hk_gemm_bf16. K must be a multiple of 32 (else
 * HK_ERR_INVALID_ARG). The products accumulate in fp32 on the tensor cores
 * (tcgen05.mma kind::mxf8f6f4 with block scales: 256×256 tiles on CTA pairs
 * when M > 128, else 128×192 tiles on one CTA).
 * `workspace` (device memory, 256-byte aligned, caller-owned, at least
 * hk_gemm_mxfp8_workspace_size(M, N, K) bytes, else HK_ERR_WORKSPACE)
 * receives the scales rearranged per tile and K stage by a small kernel
 * that runs first on `stream`; calls that overlap on the GPU must not share
 * it. Errors and asynchrony as hk_gemm_bf16. */
hk_status hk_gemm_mxfp8(const void* A, const void* B, const void* SFA, const void* SFB, void* C,
                        int64_t M, int64_t N, int64_t K,
                        int64_t lda, int64_t ldb, int64_t ldsfa, int64_t ldsfb, int64_t ldc,
                        void* workspace, size_t workspace_bytes, void* stream);

/* The same with test and tuning controls: `flags` takes
 * HK_FLAG_FAULT_DROP_ARRIVE (the producer withholds one arrival on the
 * first stage, so a bounded wait runs out and the status word reports
 * HK_ERR_TIMEOUT; other bits are rejected with HK_ERR_INVALID_ARG),
 * `timeout_ns` bounds each wait (0: 1 s). */
hk_status hk_gemm_mxfp8_ex(const void* A, const void* B, const void* SFA, const void* SFB, void* C,
                           int64_t M, int64_t N, int64_t K,
                           int64_t lda, int64_t ldb, int64_t ldsfa, int64_t ldsfb, int64_t ldc,
                           void* workspace, size_t workspace_bytes, uint32_t flags, uint64_t timeout_ns,
                           void* stream);

/* Bytes of workspace hk_gemm_mxfp8 needs for this shape (0 when M, N or K is 0). */
size_t hk_gemm_mxfp8_workspace_size(int64_t M, int64_t N, int64_t K);

/* Synchronise the plan's device and read-and-clear its status word:
 * HK_OK, or HK_ERR_TIMEOUT if a bounded wait ran out in any run since the
 * last read. */
hk_status hk_gemm_plan_device_status(hk_gemm_plan* plan);

/* The same for the calls of the one-shot entry points (hk_gemm_bf16,
 * hk_gemm_bf16_epilogue, hk_gemm_bf16_fused, hk_gemm_fp8_e4m3, hk_gemm_mxfp8(_ex),
 * hk_attention_fwd(_ex), hk_gemm_bf16_noalloc) on `device`. */
hk_status hk_gemm_last_device_status(int device);

void hk_gemm_plan_destroy(hk_gemm_plan* plan);

/* GEMM that allocates nothing, for callers that cannot call cudaMalloc when
 * they run a GEMM (code inside a memory pool or arena that owns all device
 * memory, allocator or runtime hooks that must not re-enter the allocator,
 * services that fix their memory at start-up). This entry point has no
 * counterpart on the HipKittens pages; it exists for those callers.
 *
 * Same operation, arguments and errors as hk_gemm_bf16, plus `split_k`
 * (0: chosen automatically, 1: never split K, > 1: forced). Its K-split
 * scratch and its status word live in one fixed array inside the library's
 * device image: 32 MiB of scratch, resident on every device that loads the
 * library until the process exits. A forced split_k whose fp32 partials
 * (split_k × M × N rounded up to the tile width × 4 bytes) exceed 32 MiB is
 * rejected with HK_ERR_WORKSPACE; an automatic split that would not fit is
 * not taken. The caller provides A, B and C; nothing is allocated, freed or
 * set up through an allocating library routine.
 *
 * The first call on a device looks up the array's device address (once, with
 * that device current); make that first call before any stream capture (a
 * first call whose stream is capturing is refused with HK_ERR_INVALID_ARG).
 * All calls on a device share the array and it keeps the last call's
 * contents (nothing in it needs to start at zero). Calls that overlap on the
 * GPU race on it: order them on one stream or serialise them. A bounded wait
 * that runs out in this variant is reported by hk_gemm_last_device_status(),
 * which reads and clears the status word in the array without allocating. */
hk_status hk_gemm_bf16_noalloc(const void* A, const void* B, void* C,
                               int64_t M, int64_t N, int64_t K,
                               int64_t lda, int64_t ldb, int64_t ldc,
                               int32_t split_k, void* stream);

/* Attention forward, MHA or GQA (the pages' second workload: HipKittens "L2"
 * detail page, §3 "Target operation" table, rows "MHA fwd" / "GQA fwd";
 * §5 "Numerical considerations" and §9.3 for the online softmax with
 * temperature sqrt(1/D)):
 *
 *     O[b,h,i,:] = bf16_rne( Σ_j P[i,j] · V[b,g,j,:] ),
 *     P[i,:]     = softmax_j( Q[b,h,i,:]·K[b,g,j,:] / sqrt(D) ),
 *     g = h / (Hq / Hkv)  (consecutive query heads share a KV head),
 *
 * over the keys j < S, or j ≤ i when `causal` is non-zero. Q·Kᵀ and P·V run
 * on the tensor cores (bf16 operands, fp32 accumulation); P is rounded to
 * bf16 before P·V and the row sums use the unrounded fp32 P; exp is the
 * hardware base-2 exponential. `lse`, when not NULL, receives per row the
 * natural-log sum ln Σ_j exp(Q·K/sqrt(D)) in fp32, [B, Hq, S].
 *
 * Layout: Q and O are [B, Hq, S, D], K and V are [B, Hkv, S, D], contiguous
 * row-major bf16 device arrays (16-byte aligned, else HK_ERR_MISALIGNED);
 * lse is a 4-byte-aligned fp32 device array or NULL. O must not overlap the
 * inputs. D must be 64 or 128, Hkv ≥ 1 must divide Hq, and B·Hq·S must stay
 * below 2^31 (else HK_ERR_INVALID_ARG). B, Hq or S equal to 0: HK_OK,
 * nothing launched. Asynchronous on `stream`; a bounded wait that runs out
 * is reported by hk_gemm_last_device_status(device). */
hk_status hk_attention_fwd(const void* Q, const void* K, const void* V, void* O, float* lse,
                           int64_t B, int64_t Hq, int64_t Hkv, int64_t S, int64_t D,
                           int32_t causal, void* stream);

/* The same with test and tuning controls: `flags` takes
 * HK_FLAG_FAULT_DROP_ARRIVE (the producer never fills the first K/V slot,
 * so a bounded wait runs out and the status word reports HK_ERR_TIMEOUT),
 * `timeout_ns` bounds each wait (0: 1 s). */
hk_status hk_attention_fwd_ex(const void* Q, const void* K, const void* V, void* O, float* lse,
                              int64_t B, int64_t Hq, int64_t Hkv, int64_t S, int64_t D,
                              int32_t causal, uint32_t flags, uint64_t timeout_ns, void* stream);

/* Static description of a status code. */
const char* hk_status_string(hk_status status);

/* Detail of the last error on the calling host thread (never NULL). */
const char* hk_gemm_last_error_string(void);

#ifdef __cplusplus
}
#endif

#endif /* HK_GEMM_H */
