/*
 * oracle_gemm.c -- plain CPU reference for C = A * B.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing in the product path may link, load or
 * call this file: only the tests, the smoke check and the bench's CPU
 * baseline use it. It shares no code, header, table or helper with the
 * CUDA library.
 *
 * What it computes. "Hiding Memory Latency in CUDA: Asynchronous Loads and
 * Software Pipelines" (section "A tiled GEMM is the canonical example" and
 * section 15, "The main idea") and "Pipeline GPU Kernel" (Step 5, item 4)
 * agree that software pipelining only reorders the loads of a tiled
 * matrix multiply and leaves its arithmetic alone.  The reference result is
 * therefore the plain definition of the product:
 *
 *     C[i][j] = sum over k < K of A[i][k] * B[k][j]
 *
 * Layouts (the library's boundary): A is row-major M x K, so A[i][k] sits at
 * A[i*K + k]; B is column-major K x N, so B[k][j] sits at Bcm[j*K + k]; C is
 * row-major M x N.
 *
 * Precision. Floating-point inputs (IEEE binary16 or bfloat16, passed as raw
 * 16-bit patterns) are decoded exactly to double and the sum is taken in
 * double, in increasing k, one product at a time. Every binary16/bfloat16
 * product is exact in double (at most 22 significant bits), so the only
 * rounding is in the running sum. Integer inputs (int8) are summed in int64,
 * which is exact. For the tolerance the float routine also returns
 * S[i][j] = sum over k of |A[i][k] * B[k][j]|.
 *
 * The loop over output rows is split across OpenMP threads; each output
 * element is still one sequential sum, so the thread count never changes a
 * result bit.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/* Input element encodings accepted by oracle_gemm_float. */
#define ORACLE_IN_F16 0
#define ORACLE_IN_BF16 1

/* IEEE 754 binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits.
 * Written out from the format's definition. */
double oracle_decode_f16(uint16_t h) {
    int sign = (h >> 15) & 1;
    int expo = (h >> 10) & 0x1f;
    int frac = h & 0x3ff;
    double v;
    if (expo == 0) {
        v = ldexp((double)frac, -24); /* subnormal: frac * 2^(1-15-10) */
    } else if (expo == 31) {
        v = frac ? NAN : INFINITY;
    } else {
        v = ldexp((double)(1024 + frac), expo - 25); /* (1.frac) * 2^(e-15) */
    }
    return sign ? -v : v;
}

/* bfloat16: the upper 16 bits of an IEEE binary32 (1 sign, 8 exponent bits
 * with bias 127, 7 fraction bits). */
double oracle_decode_bf16(uint16_t h) {
    int sign = (h >> 15) & 1;
    int expo = (h >> 7) & 0xff;
    int frac = h & 0x7f;
    double v;
    if (expo == 0) {
        v = ldexp((double)frac, -133); /* subnormal: frac * 2^(1-127-7) */
    } else if (expo == 255) {
        v = frac ? NAN : INFINITY;
    } else {
        v = ldexp((double)(128 + frac), expo - 134); /* (1.frac) * 2^(e-127) */
    }
    return sign ? -v : v;
}

static double decode(int in_type, uint16_t h) {
    return in_type == ORACLE_IN_BF16 ? oracle_decode_bf16(h) : oracle_decode_f16(h);
}

/* Decodes an array of 16-bit patterns to double (one pass, no arithmetic). */
static double* decode_all(int in_type, const uint16_t* src, int64_t n) {
    double* dst = (double*)malloc((size_t)(n > 0 ? n : 1) * sizeof(double));
    if (!dst) return NULL;
    for (int64_t t = 0; t < n; ++t) dst[t] = decode(in_type, src[t]);
    return dst;
}

int oracle_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void oracle_set_threads(int n) {
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

/*
 * Full float product. C and S are row-major M x N (S may be NULL).
 * Returns 0, or -1 when memory for the decoded inputs cannot be had.
 */
int oracle_gemm_float(int64_t M, int64_t N, int64_t K, int in_type,
                      const uint16_t* A, const uint16_t* Bcm,
                      double* C, double* S) {
    double* a = decode_all(in_type, A, M * K);
    double* b = decode_all(in_type, Bcm, N * K);
    if (!a || !b) {
        free(a);
        free(b);
        return -1;
    }
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t i = 0; i < M; ++i) {
        const double* ai = a + i * K;
        for (int64_t j = 0; j < N; ++j) {
            const double* bj = b + j * K;
            double sum = 0.0, sabs = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                double p = ai[k] * bj[k];
                sum += p;
                sabs += fabs(p);
            }
            C[i * N + j] = sum;
            if (S) S[i * N + j] = sabs;
        }
    }
    free(a);
    free(b);
    return 0;
}

/*
 * The same definition at a list of (row, col) positions only, for shapes
 * whose full product is too large for the CPU. out and sabs have n entries.
 */
int oracle_gemm_float_at(int64_t M, int64_t N, int64_t K, int in_type,
                         const uint16_t* A, const uint16_t* Bcm,
                         int64_t n, const int64_t* rows, const int64_t* cols,
                         double* out, double* sabs) {
    (void)M;
    (void)N;
#pragma omp parallel for schedule(dynamic, 16)
    for (int64_t t = 0; t < n; ++t) {
        const uint16_t* ai = A + rows[t] * K;
        const uint16_t* bj = Bcm + cols[t] * K;
        double sum = 0.0, s = 0.0;
        for (int64_t k = 0; k < K; ++k) {
            double p = decode(in_type, ai[k]) * decode(in_type, bj[k]);
            sum += p;
            s += fabs(p);
        }
        out[t] = sum;
        if (sabs) sabs[t] = s;
    }
    return 0;
}

/* Full int8 product, exact: C is row-major M x N in int64. */
int oracle_gemm_s8(int64_t M, int64_t N, int64_t K,
                   const int8_t* A, const int8_t* Bcm, int64_t* C) {
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t i = 0; i < M; ++i) {
        const int8_t* ai = A + i * K;
        for (int64_t j = 0; j < N; ++j) {
            const int8_t* bj = Bcm + j * K;
            int64_t sum = 0;
            for (int64_t k = 0; k < K; ++k) sum += (int64_t)ai[k] * (int64_t)bj[k];
            C[i * N + j] = sum;
        }
    }
    return 0;
}

/* int8 product at a list of (row, col) positions. */
int oracle_gemm_s8_at(int64_t M, int64_t N, int64_t K,
                      const int8_t* A, const int8_t* Bcm,
                      int64_t n, const int64_t* rows, const int64_t* cols,
                      int64_t* out) {
    (void)M;
    (void)N;
#pragma omp parallel for schedule(dynamic, 16)
    for (int64_t t = 0; t < n; ++t) {
        const int8_t* ai = A + rows[t] * K;
        const int8_t* bj = Bcm + cols[t] * K;
        int64_t sum = 0;
        for (int64_t k = 0; k < K; ++k) sum += (int64_t)ai[k] * (int64_t)bj[k];
        out[t] = sum;
    }
    return 0;
}
