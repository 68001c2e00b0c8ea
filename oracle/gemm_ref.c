/*
 * CPU oracle for the dense BF16 GEMM  C = A * B^T  (TEST INFRASTRUCTURE ONLY).
 *
 * Only the tests, the smoke check and the CPU-baseline leg of the benchmark
 * link this file; the CUDA library never does, and the two share no code.
 *
 * What it computes (HipKittens, "L2" detail page, §3 "Target operation" table:
 * BF16 GEMM, bf16 inputs, FP32 accumulation, bf16 output; §7 code listing
 * descriptions and §9.2: the GEMM hot loop is the "ABt" product, i.e. the
 * second operand is stored N x K and used transposed):
 *
 *     C[i][j] = round_bf16_rne( sum_{k=0}^{K-1} double(A[i][k]) * double(B[j][k]) )
 *
 * A is M x K row-major with leading dimension lda (elements), B is N x K
 * row-major with leading dimension ldb, C is M x N row-major with leading
 * dimension ldc. All three hold IEEE binary16-brain-float (bf16) bit patterns.
 *
 * Precision: the pages fix only bf16 in / fp32 accumulate / bf16 out. The
 * oracle is the exact definition instead: every bf16 x bf16 product is exact
 * in binary64 (8 + 8 significant bits), the sum runs in binary64 in increasing
 * k starting from +0.0, and the result is rounded ONCE, binary64 -> bf16, with
 * round-to-nearest-even written out from the IEEE 754 definition (no detour
 * through binary32, so there is no double rounding).
 *
 * The file also holds the fused-epilogue and FP8 variants of the GEMM and the
 * attention forward (GQA) of the same page; each section states its source.
 *
 * Build: plain C99, no -ffast-math, -ffp-contract=off (a fused multiply-add
 * would not change these exact products, but the flag keeps the arithmetic
 * literally what is written here).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

/* bf16 bit pattern -> binary64 value: the bf16 bits are the upper half of a
 * binary32; widening binary32 -> binary64 is exact. */
static double bf16_bits_to_double(uint16_t h) {
    uint32_t u = ((uint32_t)h) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* binary64 -> bf16 with IEEE round-to-nearest, ties-to-even.
 * bf16: 1 sign bit, 8 exponent bits (bias 127), 7 fraction bits.
 * Normal numbers: |x| in [2^E, 2^(E+1)), E >= -126, quantum 2^(E-7).
 * Subnormals (|x| < 2^-126): quantum 2^-133.
 * Values that round to >= 2^128 overflow to infinity. */
uint16_t oracle_round_bf16(double x) {
    uint16_t sign = signbit(x) ? 0x8000u : 0u;
    if (isnan(x)) return (uint16_t)(sign | 0x7FC0u);
    double a = fabs(x);
    if (a == 0.0) return sign;
    if (isinf(a)) return (uint16_t)(sign | 0x7F80u);

    int e2;
    (void)frexp(a, &e2);          /* a = f * 2^e2, f in [0.5, 1) */
    int E = e2 - 1;               /* a in [2^E, 2^(E+1)) */
    int qexp = (E < -126 ? -126 : E) - 7;

    double r = ldexp(a, -qexp);   /* exact: scaling by a power of two */
    double fl = floor(r);
    double frac = r - fl;         /* exact: r < 2^9 */
    double n = fl;
    if (frac > 0.5) {
        n = fl + 1.0;
    } else if (frac == 0.5) {
        if (fmod(fl, 2.0) != 0.0) n = fl + 1.0;   /* tie: go to the even neighbour */
    }
    double v = ldexp(n, qexp);    /* exact */
    if (v >= 0x1p128) return (uint16_t)(sign | 0x7F80u);

    /* v is a bf16 value, hence exactly representable in binary32; its
     * binary32 encoding has 16 zero low bits and the upper half is the bf16. */
    float vf = (float)v;
    uint32_t u;
    memcpy(&u, &vf, sizeof u);
    return (uint16_t)(sign | (uint16_t)(u >> 16));
}

/* The unrounded binary64 dot product of row i of A with row j of B. */
double oracle_dot_f64(const uint16_t* A, const uint16_t* B, int64_t K,
                      int64_t lda, int64_t ldb, int64_t i, int64_t j) {
    const uint16_t* a = A + i * lda;
    const uint16_t* b = B + j * ldb;
    double s = 0.0;
    for (int64_t k = 0; k < K; ++k) s += bf16_bits_to_double(a[k]) * bf16_bits_to_double(b[k]);
    return s;
}

/* ---- fused epilogue (bias + activation) ----------------------------------
 * C[i][j] = round_bf16_rne( act( sum_k A[i][k] * B[j][k] + bias[j] ) ), the
 * bias a bf16 vector of N entries (or none), act one of
 *   0 none:  x
 *   1 ReLU:  max(x, 0)
 *   2 GELU:  x * Phi(x) = 0.5 * x * (1 + erf(x / sqrt(2)))   (the exact, erf form)
 *   3 SiLU:  x * sigmoid(x) = x / (1 + exp(-x))
 * all evaluated in binary64 before the single rounding to bf16.
 *
 * Residual add (the fused epilogue's third step; the HipKittens "L2" detail
 * page, §8 "Deployment context", Fusion scope, names the residual add among
 * the memory-bound operations the pages keep in a kernel of their own):
 *   C[i][j] = round_bf16_rne( act( sum_k A[i][k] * B[j][k] + bias[j] ) + R[i][j] )
 * R an M x N bf16 matrix with leading dimension ldr, added after the
 * activation (the residual stream of a transformer block takes the block's
 * output unchanged), still in binary64 and still before the one rounding. */
double oracle_activation(double x, int act) {
    switch (act) {
        case 1: return x > 0.0 ? x : 0.0;
        case 2: return 0.5 * x * (1.0 + erf(x / sqrt(2.0)));
        case 3: return x / (1.0 + exp(-x));
        default: return x;
    }
}

/* ---- threading: a plain static split of a list of work items ---------- */

typedef struct {
    const uint16_t* A;
    const uint16_t* B;
    uint16_t* out;
    const uint16_t* bias;  /* epilogue: per-column bias (bf16) or NULL */
    int act;               /* epilogue: activation code */
    int64_t N, K, lda, ldb, ldo;
    const int64_t* rows;   /* entry mode: row index per entry; row mode: row list */
    const int64_t* cols;   /* entry mode only */
    int64_t begin, end;    /* range of work items for this thread */
    int mode;              /* 0: full rows, 1: single entries */
    const uint16_t* res;   /* epilogue: residual R (bf16, M x N, leading dimension ldr) or NULL */
    int64_t ldr;
} work_t;

/* One output entry: the dot product, then (if requested) bias and
 * activation, then (if requested) the residual. */
static uint16_t entry(const work_t* w, int64_t i, int64_t j) {
    double x = oracle_dot_f64(w->A, w->B, w->K, w->lda, w->ldb, i, j);
    if (w->bias || w->act) {
        if (w->bias) x += bf16_bits_to_double(w->bias[j]);
        x = oracle_activation(x, w->act);
    }
    if (w->res) x += bf16_bits_to_double(w->res[i * w->ldr + j]);
    return oracle_round_bf16(x);
}

static void* worker(void* p) {
    work_t* w = (work_t*)p;
    for (int64_t t = w->begin; t < w->end; ++t) {
        if (w->mode == 0) {
            int64_t i = w->rows ? w->rows[t] : t;
            uint16_t* o = w->out + t * w->ldo;
            for (int64_t j = 0; j < w->N; ++j) o[j] = entry(w, i, j);
        } else {
            w->out[t] = entry(w, w->rows[t], w->cols[t]);
        }
    }
    return NULL;
}

static int resolve_threads(int threads, int64_t items) {
    if (threads <= 0) {
        long n = sysconf(_SC_NPROCESSORS_ONLN);
        threads = n > 0 ? (int)n : 1;
    }
    if (threads > 256) threads = 256;
    if (items < threads) threads = items > 0 ? (int)items : 1;
    return threads;
}

static int run_parallel(work_t base, int64_t items, int threads) {
    threads = resolve_threads(threads, items);
    pthread_t tid[256];
    int joined[256];
    work_t w[256];
    for (int t = 0; t < threads; ++t) {
        w[t] = base;
        w[t].begin = items * t / threads;
        w[t].end = items * (t + 1) / threads;
        joined[t] = 0;
        if (t == threads - 1) {
            worker(&w[t]);
        } else if (pthread_create(&tid[t], NULL, worker, &w[t]) == 0) {
            joined[t] = 1;
        } else {
            worker(&w[t]);   /* could not start a thread: do the share inline */
        }
    }
    for (int t = 0; t < threads - 1; ++t)
        if (joined[t]) pthread_join(tid[t], NULL);
    return threads;
}

/* Full GEMM: C (M x N, leading dimension ldc) = round(A * B^T).
 * Returns the number of threads used. */
int oracle_gemm_bf16(const uint16_t* A, const uint16_t* B, uint16_t* C,
                     int64_t M, int64_t N, int64_t K,
                     int64_t lda, int64_t ldb, int64_t ldc, int threads) {
    work_t w = {A, B, C, NULL, 0, N, K, lda, ldb, ldc, NULL, NULL, 0, 0, 0, NULL, 0};
    return run_parallel(w, M, threads);
}

/* Selected full rows: out[t][j] = C[rows[t]][j] for t < nrows (out has
 * leading dimension N). Returns the number of threads used. */
int oracle_gemm_bf16_rows(const uint16_t* A, const uint16_t* B, uint16_t* out,
                          int64_t N, int64_t K, int64_t lda, int64_t ldb,
                          const int64_t* rows, int64_t nrows, int threads) {
    work_t w = {A, B, out, NULL, 0, N, K, lda, ldb, N, rows, NULL, 0, 0, 0, NULL, 0};
    return run_parallel(w, nrows, threads);
}

/* Selected entries: out[t] = C[rows[t]][cols[t]]. Returns threads used. */
int oracle_gemm_bf16_entries(const uint16_t* A, const uint16_t* B, uint16_t* out,
                             int64_t K, int64_t lda, int64_t ldb,
                             const int64_t* rows, const int64_t* cols, int64_t count,
                             int threads) {
    work_t w = {A, B, out, NULL, 0, 0, K, lda, ldb, 0, rows, cols, 0, 0, 1, NULL, 0};
    return run_parallel(w, count, threads);
}

/* Full GEMM with the fused epilogue: C = round(act(A * B^T + bias)). */
int oracle_gemm_bf16_epilogue(const uint16_t* A, const uint16_t* B, const uint16_t* bias, uint16_t* C,
                              int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb, int64_t ldc,
                              int act, int threads) {
    work_t w = {A, B, C, bias, act, N, K, lda, ldb, ldc, NULL, NULL, 0, 0, 0, NULL, 0};
    return run_parallel(w, M, threads);
}

/* Selected entries with the fused epilogue. */
int oracle_gemm_bf16_epilogue_entries(const uint16_t* A, const uint16_t* B, const uint16_t* bias,
                                      uint16_t* out, int64_t K, int64_t lda, int64_t ldb, int act,
                                      const int64_t* rows, const int64_t* cols, int64_t count, int threads) {
    work_t w = {A, B, out, bias, act, 0, K, lda, ldb, 0, rows, cols, 0, 0, 1, NULL, 0};
    return run_parallel(w, count, threads);
}

/* Full GEMM with bias, activation and residual:
 * C = round(act(A * B^T + bias) + R); bias and R may each be NULL. */
int oracle_gemm_bf16_fused(const uint16_t* A, const uint16_t* B, const uint16_t* bias, const uint16_t* R,
                           int64_t ldr, uint16_t* C, int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb,
                           int64_t ldc, int act, int threads) {
    work_t w = {A, B, C, bias, act, N, K, lda, ldb, ldc, NULL, NULL, 0, 0, 0, R, ldr};
    return run_parallel(w, M, threads);
}

/* Selected entries of the same. */
int oracle_gemm_bf16_fused_entries(const uint16_t* A, const uint16_t* B, const uint16_t* bias, const uint16_t* R,
                                   int64_t ldr, uint16_t* out, int64_t K, int64_t lda, int64_t ldb, int act,
                                   const int64_t* rows, const int64_t* cols, int64_t count, int threads) {
    work_t w = {A, B, out, bias, act, 0, K, lda, ldb, 0, rows, cols, 0, 0, 1, R, ldr};
    return run_parallel(w, count, threads);
}

/* ---- FP8 (E4M3) GEMM with per-tensor scales ------------------------------
 * C[i][j] = round_bf16_rne( sa * sb * sum_k e4m3(A[i][k]) * e4m3(B[j][k]) )
 * (the FP8 GEMM row of the HipKittens "L2" detail page's §3 "Target
 * operation" table: 8-bit inputs, FP32 accumulation, bf16 output; here with
 * one scale per operand tensor). E4M3 (the OCP 8-bit format): 1 sign bit, 4
 * exponent bits with bias 7, 3 fraction bits; exponent field 0 encodes
 * subnormals m/8 * 2^-6; S.1111.111 is NaN; there is no infinity; the largest
 * finite magnitude is 1.75 * 2^8 = 448. Every E4M3 value and every product
 * of two is exact in binary64. */
double oracle_e4m3_to_double(uint8_t b) {
    int s = (b >> 7) & 1, e = (b >> 3) & 0xF, m = b & 7;
    double v;
    if (e == 0xF && m == 7) return NAN;
    if (e == 0) v = ldexp((double)m / 8.0, -6);
    else v = ldexp(1.0 + (double)m / 8.0, e - 7);
    return s ? -v : v;
}

typedef struct {
    const uint8_t* A;
    const uint8_t* B;
    uint16_t* out;
    int64_t N, K, lda, ldb, ldo;
    const int64_t* rows;
    const int64_t* cols;
    int64_t begin, end;
    int mode;
    double scale;
} work8_t;

static uint16_t entry8(const work8_t* w, int64_t i, int64_t j) {
    const uint8_t* a = w->A + i * w->lda;
    const uint8_t* b = w->B + j * w->ldb;
    double s = 0.0;
    for (int64_t k = 0; k < w->K; ++k) s += oracle_e4m3_to_double(a[k]) * oracle_e4m3_to_double(b[k]);
    return oracle_round_bf16(w->scale * s);
}

static void* worker8(void* p) {
    work8_t* w = (work8_t*)p;
    for (int64_t t = w->begin; t < w->end; ++t) {
        if (w->mode == 0) {
            int64_t i = w->rows ? w->rows[t] : t;
            uint16_t* o = w->out + t * w->ldo;
            for (int64_t j = 0; j < w->N; ++j) o[j] = entry8(w, i, j);
        } else {
            w->out[t] = entry8(w, w->rows[t], w->cols[t]);
        }
    }
    return NULL;
}

static int run_parallel8(work8_t base, int64_t items, int threads) {
    threads = resolve_threads(threads, items);
    pthread_t tid[256];
    int joined[256];
    work8_t w[256];
    for (int t = 0; t < threads; ++t) {
        w[t] = base;
        w[t].begin = items * t / threads;
        w[t].end = items * (t + 1) / threads;
        joined[t] = 0;
        if (t == threads - 1) worker8(&w[t]);
        else if (pthread_create(&tid[t], NULL, worker8, &w[t]) == 0) joined[t] = 1;
        else worker8(&w[t]);
    }
    for (int t = 0; t < threads - 1; ++t)
        if (joined[t]) pthread_join(tid[t], NULL);
    return threads;
}

/* Full FP8 GEMM; `scale` = sa * sb (taken in binary64). */
int oracle_gemm_fp8e4m3(const uint8_t* A, const uint8_t* B, uint16_t* C, int64_t M, int64_t N, int64_t K,
                        int64_t lda, int64_t ldb, int64_t ldc, double scale, int threads) {
    work8_t w = {A, B, C, N, K, lda, ldb, ldc, NULL, NULL, 0, 0, 0, scale};
    return run_parallel8(w, M, threads);
}

/* Selected entries of the FP8 GEMM. */
int oracle_gemm_fp8e4m3_entries(const uint8_t* A, const uint8_t* B, uint16_t* out, int64_t K, int64_t lda,
                                int64_t ldb, double scale, const int64_t* rows, const int64_t* cols,
                                int64_t count, int threads) {
    work8_t w = {A, B, out, 0, K, lda, ldb, 0, rows, cols, 0, 0, 1, scale};
    return run_parallel8(w, count, threads);
}

/* ---- MXFP8 GEMM (E4M3 blocks of 32 with UE8M0 scales) --------------------
 * The FP8 GEMM row of the HipKittens "L2" detail page's §3 "Target
 * operation" table is an MXFP8 product: FP8 (E4M3) operands whose K dimension
 * is cut into blocks of 32 consecutive elements, each block of each row
 * carrying one shared scale, FP32 accumulation, here a bf16 output. The scale
 * byte is UE8M0 (the OCP MX format's 8-bit unsigned exponent): value
 * 2^(E - 127), E = 255 is NaN. With KB = K / 32 blocks:
 *   C[i][j] = round_bf16_rne( sum_b SA[i][b] * SB[j][b] * sum_{k in block b} A[i][k] * B[j][k] ).
 * Each block sum of 32 exact products is exact in binary64 (the products span
 * fewer than 53 bits of exponent and mantissa); the scales are powers of two;
 * the sum over blocks runs in binary64 in increasing b; one rounding. */
double oracle_ue8m0_to_double(uint8_t e) {
    if (e == 255) return NAN;
    return ldexp(1.0, (int)e - 127);
}

typedef struct {
    const uint8_t *A, *B, *SA, *SB;
    uint16_t* out;
    int64_t N, K, lda, ldb, ldsa, ldsb, ldo;
    const int64_t* rows;
    const int64_t* cols;
    int64_t begin, end;
    int mode;
} workmx_t;

static uint16_t entry_mx(const workmx_t* w, int64_t i, int64_t j) {
    const uint8_t* a = w->A + i * w->lda;
    const uint8_t* b = w->B + j * w->ldb;
    const uint8_t* sa = w->SA + i * w->ldsa;
    const uint8_t* sb = w->SB + j * w->ldsb;
    double s = 0.0;
    for (int64_t blk = 0; blk < w->K / 32; ++blk) {
        double d = 0.0;
        for (int64_t k = 32 * blk; k < 32 * blk + 32; ++k)
            d += oracle_e4m3_to_double(a[k]) * oracle_e4m3_to_double(b[k]);
        s += oracle_ue8m0_to_double(sa[blk]) * oracle_ue8m0_to_double(sb[blk]) * d;
    }
    return oracle_round_bf16(s);
}

static void* worker_mx(void* p) {
    workmx_t* w = (workmx_t*)p;
    for (int64_t t = w->begin; t < w->end; ++t) {
        if (w->mode == 0) {
            uint16_t* o = w->out + t * w->ldo;
            for (int64_t j = 0; j < w->N; ++j) o[j] = entry_mx(w, t, j);
        } else {
            w->out[t] = entry_mx(w, w->rows[t], w->cols[t]);
        }
    }
    return NULL;
}

static int run_parallel_mx(workmx_t base, int64_t items, int threads) {
    threads = resolve_threads(threads, items);
    pthread_t tid[256];
    int joined[256];
    workmx_t w[256];
    for (int t = 0; t < threads; ++t) {
        w[t] = base;
        w[t].begin = items * t / threads;
        w[t].end = items * (t + 1) / threads;
        joined[t] = 0;
        if (t == threads - 1) worker_mx(&w[t]);
        else if (pthread_create(&tid[t], NULL, worker_mx, &w[t]) == 0) joined[t] = 1;
        else worker_mx(&w[t]);
    }
    for (int t = 0; t < threads - 1; ++t)
        if (joined[t]) pthread_join(tid[t], NULL);
    return threads;
}

/* Full MXFP8 GEMM; K must be a multiple of 32; SA is M x K/32 (row stride
 * ldsa bytes), SB is N x K/32 (ldsb). */
int oracle_gemm_mxfp8(const uint8_t* A, const uint8_t* B, const uint8_t* SA, const uint8_t* SB, uint16_t* C,
                      int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb, int64_t ldsa, int64_t ldsb,
                      int64_t ldc, int threads) {
    workmx_t w = {A, B, SA, SB, C, N, K, lda, ldb, ldsa, ldsb, ldc, NULL, NULL, 0, 0, 0};
    return run_parallel_mx(w, M, threads);
}

/* Selected entries of the MXFP8 GEMM. */
int oracle_gemm_mxfp8_entries(const uint8_t* A, const uint8_t* B, const uint8_t* SA, const uint8_t* SB,
                              uint16_t* out, int64_t K, int64_t lda, int64_t ldb, int64_t ldsa, int64_t ldsb,
                              const int64_t* rows, const int64_t* cols, int64_t count, int threads) {
    workmx_t w = {A, B, SA, SB, out, 0, K, lda, ldb, ldsa, ldsb, 0, rows, cols, 0, 0, 1};
    return run_parallel_mx(w, count, threads);
}

/* ---- attention forward (GQA) ----------------------------------------------
 * The pages' second workload (HipKittens "L2" detail page, §3 "Target
 * operation" table, rows MHA / GQA fwd: Q [B, Hq, S, D], K and V
 * [B, Hkv, S, D], O [B, Hq, S, D], bf16 in, FP32 accumulate, bf16 out; §5
 * "Numerical considerations": softmax with temperature sqrt(1/D)):
 *     O[b,h,i,:] = round_bf16( sum_j P[i,j] V[b,g,j,:] ),
 *     P[i,:] = softmax_j( (Q[b,h,i,:] . K[b,g,j,:]) / sqrt(D) ),  g = h / (Hq/Hkv),
 * with j <= i when causal. Written as the definition: the scores in binary64,
 * the softmax as exp(s_j - max_j s) / sum (the shift by the maximum changes
 * nothing mathematically and keeps exp finite), one rounding at the end.
 * The log-sum-exp of each row's scaled scores, ln sum_j exp(s_j), which the
 * pages' forward kernel also stores for the backward pass (§9.3 "Attention
 * forward", epilogue), is written to lse when it is not NULL. */
typedef struct {
    const uint16_t *Q, *K, *V;
    uint16_t* O;
    double* lse;
    int64_t B, Hq, Hkv, S, D;
    int causal;
    int64_t begin, end;   /* range of (b, h, i) rows */
} attn_t;

static void* attn_worker(void* p) {
    attn_t* w = (attn_t*)p;
    double* s = (double*)malloc(sizeof(double) * (size_t)w->S);
    double* o = (double*)malloc(sizeof(double) * (size_t)w->D);
    const double scale = 1.0 / sqrt((double)w->D);
    const int64_t group = w->Hq / w->Hkv;
    for (int64_t r = w->begin; r < w->end; ++r) {
        const int64_t i = r % w->S, h = (r / w->S) % w->Hq, b = r / (w->S * w->Hq), g = h / group;
        const uint16_t* q = w->Q + ((b * w->Hq + h) * w->S + i) * w->D;
        const uint16_t* kb = w->K + (b * w->Hkv + g) * w->S * w->D;
        const uint16_t* vb = w->V + (b * w->Hkv + g) * w->S * w->D;
        const int64_t n = w->causal ? i + 1 : w->S;
        double mx = -INFINITY;
        for (int64_t j = 0; j < n; ++j) {
            double d = 0.0;
            for (int64_t t = 0; t < w->D; ++t) d += bf16_bits_to_double(q[t]) * bf16_bits_to_double(kb[j * w->D + t]);
            s[j] = d * scale;
            if (s[j] > mx) mx = s[j];
        }
        double sum = 0.0;
        for (int64_t j = 0; j < n; ++j) { s[j] = exp(s[j] - mx); sum += s[j]; }
        for (int64_t t = 0; t < w->D; ++t) o[t] = 0.0;
        for (int64_t j = 0; j < n; ++j)
            for (int64_t t = 0; t < w->D; ++t) o[t] += s[j] * bf16_bits_to_double(vb[j * w->D + t]);
        uint16_t* out = w->O + ((b * w->Hq + h) * w->S + i) * w->D;
        for (int64_t t = 0; t < w->D; ++t) out[t] = oracle_round_bf16(o[t] / sum);
        if (w->lse) w->lse[r] = mx + log(sum);
    }
    free(s);
    free(o);
    return NULL;
}

/* O = attention(Q, K, V) for the rows [row_begin, row_end) of the flattened
 * (b, h, i) index (all rows: 0, B*Hq*S). Returns the number of threads used. */
int oracle_attention_fwd(const uint16_t* Q, const uint16_t* K, const uint16_t* V, uint16_t* O, double* lse,
                         int64_t B, int64_t Hq, int64_t Hkv, int64_t S, int64_t D, int causal,
                         int64_t row_begin, int64_t row_end, int threads) {
    const int64_t items = row_end - row_begin;
    threads = resolve_threads(threads, items);
    pthread_t tid[256];
    int joined[256];
    attn_t w[256];
    for (int t = 0; t < threads; ++t) {
        attn_t a = {Q, K, V, O, lse, B, Hq, Hkv, S, D, causal, row_begin + items * t / threads,
                    row_begin + items * (t + 1) / threads};
        w[t] = a;
        joined[t] = 0;
        if (t == threads - 1) attn_worker(&w[t]);
        else if (pthread_create(&tid[t], NULL, attn_worker, &w[t]) == 0) joined[t] = 1;
        else attn_worker(&w[t]);
    }
    for (int t = 0; t < threads - 1; ++t)
        if (joined[t]) pthread_join(tid[t], NULL);
    return threads;
}
