/*
 * oracle.c -- fp64 CPU oracle for the dense product C = A*B.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may include, link,
 * load or call this file: only tests/, __graft_entry__.smoke() and bench.py's
 * cpu_baseline / reference arm use it.  It shares no code, header, helper or
 * constant with the CUDA library (accelerator_gb300/csrc), and it imports none.
 *
 * What it computes, and where that is defined:
 *   - The product itself: "Shared Memory Tiling for Matrix Multiplication"
 *     (anylearn.cc), opening formula: with A of size M x K and B of size K x N,
 *     C_ij = sum over k = 0 .. K-1 of A_ik * B_kj.
 *   - Row-major storage: "Matrix Multiplication -- Naive to Tiled", section 02
 *     (Naive Implementation): A_ik is A[i*K + k], B_kj is B[k*N + j] and C_ij
 *     is C[i*N + j]; there are no leading-dimension arguments.
 *   - The sum-of-all-elements check in double precision: "From 306 ms to
 *     86 ms" (kpapadogiannis.dev), the "How each kernel was timed" box.
 *   - The generalised product C := alpha*A*B + beta*C: "Matrix
 *     Multiplication -- Naive to Tiled", section 07, the cuBLAS comparison
 *     call (oracle_update, oracle_update_f32).
 *
 * Readings taken where the pages are silent (each is also listed in the
 * design notes):
 *   - Accumulation is in double, k ascending.  The pages' own CPU reference
 *     accumulates in float; a checker must be more accurate than what it
 *     checks, so this one widens every input exactly to double first.
 *   - K == 0 gives the empty sum, 0.  M == 0 or N == 0 gives an empty C.
 *   - Alongside C the oracle returns S_ij = sum_k |A_ik * B_kj|, the scale
 *     against which a result is judged: |C - Cref| <= tol * S_ij.
 *   - Input formats.  FP32 values widen exactly.  BF16 values arrive as their
 *     16-bit patterns (sign, 8 exponent bits, 7 fraction bits: the top half of
 *     an IEEE binary32) and widen exactly.  The TF32 diagnostic format keeps
 *     the sign, the 8 exponent bits and the top 10 fraction bits of a binary32
 *     and clears the other 13 (truncation), then widens exactly.  FP16 values
 *     arrive as IEEE binary16 patterns (sign, 5 exponent bits with bias 15,
 *     10 fraction bits; exponent 0 holds the subnormals) and widen exactly.
 *     The TF32-nearest format rounds a binary32 to the nearest value with 10
 *     fraction bits, ties away from zero (the rounding of the GEMM_TF32_RN
 *     mode), and widens that exactly.
 *
 * Each product of two widened binary32 values has at most 48 significant
 * bits and is therefore exact in double; only the running sums round.  The
 * library is built with -ffp-contract=off so that x86 and Arm agree bit for
 * bit.
 *
 * oracle_gemm_f32_chain is a second, narrower reference: the product as a
 * binary32 machine computes it with one fused multiply-add per term, k
 * ascending (fmaf is correctly rounded in C99).  The pages leave the order
 * and rounding of the sum open; this is the reading the library's FP32 mode
 * documents, and tests compare it bit for bit where the library does not split
 * the K range.
 *
 * The update's pins: hand-worked cases (tests/golden/update_hand.txt),
 * alpha = 1 / beta = 0 giving the product, beta = 0 ignoring a NaN C, alpha
 * = 0 ignoring a NaN product, a tie that shows alpha*P is rounded once, and a
 * case whose fused and unfused results differ.
 *
 * Parity pins (tests/test_oracle.py): identity and permutation matrices,
 * hand-worked integer products (tests/golden/), rank-1 closed forms, all-ones
 * inputs, the sum identity, S against C on non-negative inputs, the exact
 * widening of known BF16/TF32 bit patterns, and agreement with numpy's float64
 * matmul on small random inputs.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum {
    ORACLE_F32 = 0,       /* binary32 values                          */
    ORACLE_BF16 = 1,      /* bfloat16 bit patterns (uint16)           */
    ORACLE_TF32_TRUNC = 2,/* binary32, low 13 fraction bits cleared   */
    ORACLE_F64 = 3,       /* binary64 values, used as given           */
    ORACLE_F16 = 4,       /* IEEE binary16 bit patterns (uint16)      */
    ORACLE_TF32_RNA = 5   /* binary32 rounded to TF32, nearest, ties away */
};

static double from_bits32(uint32_t u) {
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* The value of an IEEE binary16 pattern (finite inputs only). */
static double from_half(uint16_t h) {
    const int sign = h >> 15, e = (h >> 10) & 0x1F, f = h & 0x3FF;
    double v = e == 0 ? ldexp((double)f, -24)                 /* subnormal: f * 2^-24 */
                      : ldexp((double)(1024 + f), e - 25);    /* (1 + f/1024) * 2^(e-15) */
    return sign ? -v : v;
}

/* A binary32 value rounded to the nearest TF32 value, ties away from zero.
 * TF32 keeps binary32's sign and 8-bit exponent and 10 fraction bits, so a
 * value of magnitude in [2^e, 2^(e+1)) lies on a grid of spacing 2^(e-10)
 * (for e >= -126; below, the subnormals, the spacing stays 2^-136).  The
 * magnitude is split into the grid point below it and the remainder; a
 * remainder of half the spacing or more rounds up (a tie goes away from
 * zero).  Rounding up past the largest TF32 value, (2 - 2^-10) * 2^127, gives
 * infinity.  Zero, infinity and NaN are kept.  Every step is exact in double. */
static double tf32_nearest_away(float f) {
    if (f == 0.0f || isinf(f) || isnan(f)) return (double)f;
    const double a = fabs((double)f);
    int e2 = 0;
    (void)frexp(a, &e2);                /* a = m * 2^e2, m in [0.5, 1): a in [2^(e2-1), 2^e2) */
    const int e = e2 - 1 < -126 ? -126 : e2 - 1;
    const double spacing = ldexp(1.0, e - 10);
    const double below = floor(a / spacing) * spacing;
    double v = (a - below >= 0.5 * spacing) ? below + spacing : below;
    if (v >= ldexp(1.0, 128)) v = INFINITY;
    return f < 0.0f ? -v : v;
}

/* Element idx of an input matrix in format fmt, widened exactly to double. */
static double widen(int fmt, const void* p, int64_t idx) {
    switch (fmt) {
    case ORACLE_F32:
        return (double)((const float*)p)[idx];
    case ORACLE_BF16:
        return from_bits32((uint32_t)((const uint16_t*)p)[idx] << 16);
    case ORACLE_TF32_TRUNC: {
        uint32_t u;
        memcpy(&u, (const float*)p + idx, sizeof u);
        return from_bits32(u & 0xFFFFE000u);
    }
    case ORACLE_F16:
        return from_half(((const uint16_t*)p)[idx]);
    case ORACLE_TF32_RNA:
        return tf32_nearest_away(((const float*)p)[idx]);
    default:
        return ((const double*)p)[idx];
    }
}

static int valid(int fmt, const void* A, const void* B, int64_t M, int64_t K,
                 int64_t N) {
    if (fmt < ORACLE_F32 || fmt > ORACLE_TF32_RNA) return 0;
    if (M < 0 || K < 0 || N < 0) return 0;
    if ((M > 0 && K > 0 && !A) || (K > 0 && N > 0 && !B)) return 0;
    return 1;
}

static void set_threads(int nthreads) {
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
}

/* Number of threads the parallel loops will use (1 without OpenMP). */
int oracle_threads(int nthreads) {
#ifdef _OPENMP
    set_threads(nthreads);
    return omp_get_max_threads();
#else
    (void)nthreads;
    return 1;
#endif
}

/* Widen a rows x cols input matrix into a freshly allocated double array. */
static double* widen_matrix(int fmt, const void* p, int64_t rows, int64_t cols) {
    int64_t n = rows * cols;
    double* w = (double*)malloc((size_t)(n > 0 ? n : 1) * sizeof(double));
    if (!w) return NULL;
    for (int64_t t = 0; t < n; ++t) w[t] = widen(fmt, p, t);
    return w;
}

/*
 * Full product.  C[i*N+j] = sum_k A_ik B_kj and, when S is not NULL,
 * S[i*N+j] = sum_k |A_ik B_kj|, every sum in double with k ascending.  Rows of
 * C are independent, so they are shared among threads; the order of each sum
 * does not depend on the thread count.  Returns 0, or -1 on a bad argument or
 * an allocation failure.
 */
int oracle_gemm(int fmt, const void* A, const void* B, int64_t M, int64_t K,
                int64_t N, double* C, double* S, int nthreads) {
    if (!valid(fmt, A, B, M, K, N) || (M > 0 && N > 0 && !C)) return -1;
    if (M == 0 || N == 0) return 0;
    double* a = widen_matrix(fmt, A, M, K);
    double* b = widen_matrix(fmt, B, K, N);
    if (!a || !b) {
        free(a);
        free(b);
        return -1;
    }
    set_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t i = 0; i < M; ++i) {
        for (int64_t j = 0; j < N; ++j) {
            double acc = 0.0, scale = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                double prod = a[i * K + k] * b[k * N + j];
                acc += prod;
                scale += fabs(prod);
            }
            C[i * N + j] = acc;
            if (S) S[i * N + j] = scale;
        }
    }
    free(a);
    free(b);
    return 0;
}

/*
 * The same sums for n chosen entries only: C[t] = C_{rows[t], cols[t]} and
 * S[t] likewise.  Widens on the fly, so it works on inputs of any size.
 */
int oracle_dot(int fmt, const void* A, const void* B, int64_t M, int64_t K,
               int64_t N, const int64_t* rows, const int64_t* cols, int64_t n,
               double* C, double* S, int nthreads) {
    if (!valid(fmt, A, B, M, K, N) || n < 0 || (n > 0 && (!rows || !cols || !C)))
        return -1;
    for (int64_t t = 0; t < n; ++t)
        if (rows[t] < 0 || rows[t] >= M || cols[t] < 0 || cols[t] >= N) return -1;
    set_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 16)
    for (int64_t t = 0; t < n; ++t) {
        int64_t i = rows[t], j = cols[t];
        double acc = 0.0, scale = 0.0;
        for (int64_t k = 0; k < K; ++k) {
            double prod = widen(fmt, A, i * K + k) * widen(fmt, B, k * N + j);
            acc += prod;
            scale += fabs(prod);
        }
        C[t] = acc;
        if (S) S[t] = scale;
    }
    return 0;
}

/*
 * Sum of all elements of C without forming C: exchanging the order of the
 * sums, sum_ij C_ij = sum_k (sum_i A_ik) (sum_j B_kj).  The matching scale
 * sum_ij S_ij = sum_k (sum_i |A_ik|) (sum_j |B_kj|) is returned in *abs_total.
 * Costs O(MK + KN).
 */
int oracle_sum(int fmt, const void* A, const void* B, int64_t M, int64_t K,
               int64_t N, double* total, double* abs_total) {
    if (!valid(fmt, A, B, M, K, N) || !total) return -1;
    double t = 0.0, ta = 0.0;
    for (int64_t k = 0; k < K; ++k) {
        double colA = 0.0, colA_abs = 0.0, rowB = 0.0, rowB_abs = 0.0;
        for (int64_t i = 0; i < M; ++i) {
            double v = widen(fmt, A, i * K + k);
            colA += v;
            colA_abs += fabs(v);
        }
        for (int64_t j = 0; j < N; ++j) {
            double v = widen(fmt, B, k * N + j);
            rowB += v;
            rowB_abs += fabs(v);
        }
        t += colA * rowB;
        ta += colA_abs * rowB_abs;
    }
    *total = t;
    if (abs_total) *abs_total = ta;
    return 0;
}

/*
 * C[i*N+j] = the binary32 chain acc = fmaf(A_ik, B_kj, acc), k = 0 .. K-1,
 * from acc = 0.  Returns 0, or -1 on a bad argument.
 */
int oracle_gemm_f32_chain(const float* A, const float* B, int64_t M, int64_t K, int64_t N,
                          float* C, int nthreads) {
    if (M < 0 || K < 0 || N < 0 || (M > 0 && K > 0 && !A) || (K > 0 && N > 0 && !B) ||
        (M > 0 && N > 0 && !C))
        return -1;
    set_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t i = 0; i < M; ++i) {
        for (int64_t j = 0; j < N; ++j) {
            float acc = 0.0f;
            for (int64_t k = 0; k < K; ++k) acc = fmaf(A[i * K + k], B[k * N + j], acc);
            C[i * N + j] = acc;
        }
    }
    return 0;
}

/*
 * The update C := alpha * P + beta * C_in of the generalised product, with P
 * the product A*B ("Matrix Multiplication -- Naive to Tiled", section 07, the
 * cuBLAS comparison call, whose comment states C = alpha*A*B + beta*C), in
 * double, element by element over n entries.  BLAS conventions where the
 * page is silent: beta == 0 reads no C_in (it may be NULL, and a NaN there
 * does not propagate); alpha == 0 reads no P (the product is not needed).
 * Returns 0, or -1 on a bad argument.
 */
int oracle_update(const double* P, const float* C_in, int64_t n, double alpha, double beta,
                  double* out) {
    if (n < 0 || (n > 0 && (!out || (alpha != 0.0 && !P) || (beta != 0.0 && !C_in))))
        return -1;
    for (int64_t t = 0; t < n; ++t) {
        double v = alpha != 0.0 ? alpha * P[t] : 0.0;
        if (beta != 0.0) v += beta * (double)C_in[t];
        out[t] = v;
    }
    return 0;
}

/*
 * The same update as a binary32 machine computes it from the binary32 sum P:
 * t = alpha * P rounded once, then out = fmaf(beta, C_in, t) (one fused
 * multiply-add, rounded once).  beta == 0 gives t without reading C_in;
 * alpha == 0 gives beta * C_in rounded once (0 when beta == 0 as well),
 * without reading P.  This is the reading the library's binary32 epilogue
 * documents; the page leaves the rounding open.
 */
int oracle_update_f32(const float* P, const float* C_in, int64_t n, float alpha, float beta,
                      float* out) {
    if (n < 0 || (n > 0 && (!out || (alpha != 0.0f && !P) || (beta != 0.0f && !C_in))))
        return -1;
    for (int64_t t = 0; t < n; ++t) {
        if (alpha == 0.0f) {
            out[t] = beta != 0.0f ? beta * C_in[t] : 0.0f;
        } else {
            const float s = alpha * P[t];
            out[t] = beta != 0.0f ? fmaf(beta, C_in[t], s) : s;
        }
    }
    return 0;
}

/* Element-wise widening of n inputs of format fmt (to test the formats). */
int oracle_widen(int fmt, const void* p, int64_t n, double* out) {
    if (fmt < ORACLE_F32 || fmt > ORACLE_TF32_RNA || n < 0 || (n > 0 && (!p || !out)))
        return -1;
    for (int64_t t = 0; t < n; ++t) out[t] = widen(fmt, p, t);
    return 0;
}
