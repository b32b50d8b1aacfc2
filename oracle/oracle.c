/*
 * CPU oracle for the low-M dense bf16 GEMM  C[M,N] = A[M,K] . W[N,K]^T.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path links, loads or
 * calls this file; only the tests, the smoke check and the benchmark's CPU
 * baseline do.  It shares no code, header, table or helper with the CUDA
 * library.
 *
 * What it computes, and from where:
 *   - "Fix two synchronization gaps in the MiniMax M3 low-M split-K GEMM"
 *     (TensorRT-LLM PR), Hardware verification: the kernel's bf16 output is
 *     checked per launch against a higher-precision product of the same bf16
 *     inputs.  The plain definition of that product is written out here: the
 *     bf16 inputs are decoded exactly, every product and the k-ordered sum are
 *     taken in fp64, and the sum is rounded ONCE, directly from fp64 to bf16
 *     with round-to-nearest-even (the pages name no rounding mode; RNE is the
 *     reading taken).  No blocking, no splitting of K, no reordering.
 *   - "warpgroup_mma_wait does not properly synchronize across warpgroups"
 *     (Triton issue), reproducer: with one operand all ones and the other
 *     integer valued, every partial sum is an exact integer, so the expected
 *     output is a plain column sum.  oracle_exact_gemm_bf16 below evaluates
 *     the dot products with no rounding at all (a fixed-point accumulator
 *     wide enough for every bf16 product), then rounds once; the tests use it
 *     to pin the fp64 path.
 *
 * Layouts: A is row-major [M,K], W is row-major [N,K] (K contiguous), C is
 * row-major [M,N]; all bf16 values are passed as their 16-bit patterns.
 */
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* bf16 is the top half of an IEEE binary32 pattern, so the decode is exact. */
double oracle_bf16_to_f64(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/*
 * Round an fp64 value to bf16 with round-to-nearest, ties-to-even, working on
 * the fp64 bit pattern so there is no intermediate rounding to fp32.
 * bf16: 1 sign bit, 8 exponent bits (bias 127), 7 stored mantissa bits;
 * normal numbers 2^-126 .. (2 - 2^-7) * 2^127, subnormals m * 2^-133.
 */
uint16_t oracle_f64_to_bf16_rne(double x)
{
    uint64_t bits;
    memcpy(&bits, &x, sizeof bits);
    uint16_t sign = (uint16_t)((bits >> 63) << 15);
    int exp_field = (int)((bits >> 52) & 0x7ff);
    uint64_t frac = bits & ((1ull << 52) - 1);

    if (exp_field == 0x7ff)                      /* Inf or NaN */
        return frac ? (uint16_t)(sign | 0x7fc0) : (uint16_t)(sign | 0x7f80);
    if (exp_field == 0)                          /* zero or fp64 subnormal: far below bf16's range */
        return sign;

    int e = exp_field - 1023;                    /* |x| = mant * 2^(e-52), mant in [2^52, 2^53) */
    uint64_t mant = frac | (1ull << 52);
    if (e > 127)
        return (uint16_t)(sign | 0x7f80);        /* beyond the largest finite bf16 */

    /* The bf16 quantum at |x|: 2^(e-7) for normals, 2^-133 below 2^-126. */
    int qe = (e >= -126 ? e : -126) - 7;
    int sh = 52 + qe - e;                        /* |x| / 2^qe = mant >> sh (plus a remainder) */
    uint64_t n;
    if (sh >= 54) {
        n = 0;                                   /* |x| < half a quantum */
    } else {
        n = mant >> sh;
        uint64_t rem = mant & ((1ull << sh) - 1);
        uint64_t half = 1ull << (sh - 1);
        if (rem > half || (rem == half && (n & 1)))
            n += 1;
    }
    if (e < -126)                                /* subnormal quantum: the pattern is n itself */
        return (uint16_t)(sign | (uint16_t)n);   /* n == 128 carries into the smallest normal */
    /* normal: n in [128, 256]; n == 256 carries into the exponent (and 0x7f80 = Inf) */
    return (uint16_t)(sign | (uint16_t)(((uint32_t)(e + 127) << 7) + (uint32_t)(n - 128)));
}

/* ---------------------------------------------------------------- fp64 path */

typedef struct {
    const uint16_t *A, *W;
    uint16_t *C;
    double *S;
    int M, N, K;
    int c_begin, c_end;
} oracle_slice_t;

static void *oracle_gemm_slice(void *arg)
{
    const oracle_slice_t *t = (const oracle_slice_t *)arg;
    for (int r = 0; r < t->M; ++r) {
        for (int c = t->c_begin; c < t->c_end; ++c) {
            const uint16_t *a = t->A + (size_t)r * t->K;
            const uint16_t *w = t->W + (size_t)c * t->K;
            double s = 0.0;
            for (int k = 0; k < t->K; ++k)      /* k order; each product is exact in fp64 */
                s += oracle_bf16_to_f64(a[k]) * oracle_bf16_to_f64(w[k]);
            if (t->S)
                t->S[(size_t)r * t->N + c] = s;
            if (t->C)
                t->C[(size_t)r * t->N + c] = oracle_f64_to_bf16_rne(s);
        }
    }
    return NULL;
}

/*
 * C[r,c] = bf16_rne( sum_k f64(A[r,k]) * f64(W[c,k]) ), S[r,c] = the fp64 sum.
 * Either output may be NULL.  Columns are split across nthreads host threads;
 * every element is computed by exactly one thread in the same k order, so the
 * result does not depend on nthreads.  Returns 0, or -1 on bad arguments.
 */
int oracle_gemm_bf16_f64(const uint16_t *A, const uint16_t *W, uint16_t *C, double *S,
                         int M, int N, int K, int nthreads)
{
    if (M < 0 || N < 0 || K < 0 || (M * (long)N > 0 && (!A || !W)))
        return -1;
    if (nthreads < 1)
        nthreads = 1;
    if (nthreads > N)
        nthreads = N > 0 ? N : 1;
    oracle_slice_t *sl = (oracle_slice_t *)calloc((size_t)nthreads, sizeof *sl);
    pthread_t *th = (pthread_t *)calloc((size_t)nthreads, sizeof *th);
    char *running = (char *)calloc((size_t)nthreads, 1);
    if (!sl || !th || !running) {
        free(sl);
        free(th);
        free(running);
        return -1;
    }
    for (int i = 0; i < nthreads; ++i) {
        sl[i] = (oracle_slice_t){A, W, C, S, M, N, K,
                                 (int)((long)N * i / nthreads), (int)((long)N * (i + 1) / nthreads)};
        if (i > 0)
            running[i] = pthread_create(&th[i], NULL, oracle_gemm_slice, &sl[i]) == 0;
    }
    oracle_gemm_slice(&sl[0]);
    for (int i = 1; i < nthreads; ++i) {
        if (running[i])
            pthread_join(th[i], NULL);
        else
            oracle_gemm_slice(&sl[i]);           /* a thread that failed to start: run its slice here */
    }
    free(running);
    free(sl);
    free(th);
    return 0;
}

/* --------------------------------------------------------------- exact path */

/*
 * Every finite bf16 value is i * 2^x with an integer |i| < 256 and x >= -133,
 * so every product of two is p * 2^y with |p| < 2^16 and y >= -266.  A sum of
 * up to 2^16 such products, with y <= 240, fits in a fixed-point number whose
 * least significant bit is 2^-266 and which spans fewer than 560 bits.  The
 * accumulator holds it as signed 32-bit limbs kept in int64 with deferred
 * carries; nothing is rounded until the final single rounding to bf16.
 */
#define EXACT_LSB_EXP (-266)
#define EXACT_LIMBS 20                            /* 640 bits */

static int bf16_to_int_pow2(uint16_t b, int32_t *i, int *x)
{
    int ef = (b >> 7) & 0xff;
    int m = b & 0x7f;
    int s = (b >> 15) ? -1 : 1;
    if (ef == 0xff)
        return -1;                               /* Inf/NaN: not representable exactly */
    if (ef == 0) {
        *i = s * m;
        *x = -133;
    } else {
        *i = s * (128 + m);
        *x = ef - 127 - 7;
    }
    return 0;
}

/* Round the exact fixed-point value (limbs normalized, LSB 2^-266) once to bf16 RNE. */
static uint16_t exact_round_to_bf16(int64_t *limb)
{
    /* normalize: every limb in [0, 2^32), the top limb carries the sign */
    for (int i = 0; i < EXACT_LIMBS - 1; ++i) {
        int64_t carry = limb[i] >> 32;           /* arithmetic shift: floor division */
        limb[i] -= carry * ((int64_t)1 << 32);
        limb[i + 1] += carry;
    }
    uint16_t sign = 0;
    if (limb[EXACT_LIMBS - 1] < 0) {             /* two's complement negate */
        sign = 0x8000;
        int64_t borrow = 0;
        for (int i = 0; i < EXACT_LIMBS; ++i) {
            int64_t v = -limb[i] - borrow;
            borrow = 0;
            if (i < EXACT_LIMBS - 1 && v < 0) {
                v += (int64_t)1 << 32;
                borrow = 1;
            }
            limb[i] = v;
        }
    }
    /* magnitude = sum limb[i] * 2^(32 i) * 2^-266; find the top set bit */
    int top = -1;
    for (int i = EXACT_LIMBS - 1; i >= 0 && top < 0; --i)
        if (limb[i])
            for (int b = 31; b >= 0; --b)
                if ((limb[i] >> b) & 1) {
                    top = 32 * i + b;
                    break;
                }
    if (top < 0)
        return sign;                             /* exact zero rounds to +0 (or -0 never arises) */
    int e = top + EXACT_LSB_EXP;                 /* value in [2^e, 2^(e+1)) */
    if (e > 127)
        return (uint16_t)(sign | 0x7f80);
    int qe = (e >= -126 ? e : -126) - 7;
    int qbit = qe - EXACT_LSB_EXP;               /* bit index of the quantum; >= 0 */
#define BIT(k) ((k) < 0 ? 0 : (int)((limb[(k) / 32] >> ((k) % 32)) & 1))
    uint64_t n = 0;                              /* at most 8 bits: magnitude >> qbit */
    for (int k = top; k >= qbit; --k)
        n = (n << 1) | (uint64_t)BIT(k);
    int guard = BIT(qbit - 1);
    int sticky = 0;
    for (int k = qbit - 2; k >= 0 && !sticky; --k)
        sticky = BIT(k);
#undef BIT
    if (guard && (sticky || (n & 1)))
        n += 1;
    if (e < -126)
        return (uint16_t)(sign | (uint16_t)n);
    return (uint16_t)(sign | (uint16_t)(((uint32_t)(e + 127) << 7) + (uint32_t)(n - 128)));
}

/*
 * C[r,c] = bf16_rne( exact sum_k A[r,k] * W[c,k] ), single-threaded.
 * Returns 0, -1 on bad arguments or K > 65536, -2 on a non-finite input.
 */
int oracle_exact_gemm_bf16(const uint16_t *A, const uint16_t *W, uint16_t *C, int M, int N, int K)
{
    if (M < 0 || N < 0 || K < 0 || K > 65536 || (M * (long)N > 0 && (!A || !W || !C)))
        return -1;
    for (int r = 0; r < M; ++r) {
        for (int c = 0; c < N; ++c) {
            int64_t limb[EXACT_LIMBS];
            memset(limb, 0, sizeof limb);
            for (int k = 0; k < K; ++k) {
                int32_t ia, iw;
                int xa, xw;
                if (bf16_to_int_pow2(A[(size_t)r * K + k], &ia, &xa) ||
                    bf16_to_int_pow2(W[(size_t)c * K + k], &iw, &xw))
                    return -2;
                int64_t p = (int64_t)ia * iw;    /* |p| < 2^16 */
                int pos = xa + xw - EXACT_LSB_EXP; /* >= 0 */
                limb[pos / 32] += p * ((int64_t)1 << (pos % 32)); /* |term| < 2^47 */
            }
            C[(size_t)r * N + c] = exact_round_to_bf16(limb);
        }
    }
    return 0;
}
