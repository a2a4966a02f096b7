/*
 * CPU oracle for dense C = A·B.  TEST INFRASTRUCTURE ONLY.
 *
 * Only the test suite, the smoke check and the benchmark's CPU-baseline leg may
 * load this library.  The product (the CUDA library) never links, loads or calls
 * it, and the two share no source, header, table or helper.
 *
 * What it computes is the plain definition the pages give:
 *
 *     C[i,j] = sum_{k=0}^{K-1} A[i,k] * B[k,j]
 *
 * ("Chapter 5 Operators and Runtime", section 5.2.1, the element loop and the
 * 2MKN FLOP count; "SGEMM measured and the three ledgers", section 2, the
 * FLOP convention; "MTT S4000 FP16 GEMM", section 1, FP32-or-better
 * accumulation.)  Here every product and every partial sum is kept in IEEE
 * double, in ascending k, on the already-rounded input values.  A product of two
 * float/half/bf16 values is exact in double (at most 48 significant bits), so the
 * only rounding is in the running sum.  The result is returned in double, not in
 * the output type; alongside it, S[i,j] = sum_k |A[i,k]*B[k,j]|, the scale the
 * FP32 tolerance is measured against.
 *
 * Layouts ("SGEMM measured and the three ledgers", section 2: the same bytes read
 * row-major or column-major are transposes of each other; "MTT S4000 FP16 GEMM",
 * section 1: the column-major contest signature):
 *   row-major:    A[i*K + k], B[k*N + j], C[i*N + j]
 *   column-major: A[i + k*M], B[k + j*K], C[i + j*M]
 *
 * Element types: float32 (read as is), IEEE half and bf16 (uint16 bit patterns,
 * decoded bit by bit below; no compiler half type and no CUDA header is used).
 *
 * Loop order: rows i in parallel (OpenMP), then k, then j, with one double
 * accumulator per output of the row.  Each C[i,j] still sums its K products in
 * ascending k, so the result does not depend on the thread count.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { ORACLE_F32 = 0, ORACLE_F16 = 1, ORACLE_BF16 = 2 };
enum { ORACLE_ROW_MAJOR = 0, ORACLE_COL_MAJOR = 1 };

/* IEEE 754 binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
double oracle_decode_f16(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1F;
    int f = h & 0x3FF;
    double v;
    if (e == 0) {
        v = ldexp((double)f, -24);            /* subnormal: f * 2^-10 * 2^-14 */
    } else if (e == 31) {
        v = (f == 0) ? INFINITY : NAN;
    } else {
        v = ldexp((double)(1024 + f), e - 25); /* (1 + f/1024) * 2^(e-15) */
    }
    return sign ? -v : v;
}

/* bfloat16: the upper half of an IEEE binary32 (1 sign, 8 exponent bits with
 * bias 127, 7 fraction bits). */
double oracle_decode_bf16(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 7) & 0xFF;
    int f = h & 0x7F;
    double v;
    if (e == 0) {
        v = ldexp((double)f, -133);           /* subnormal: f * 2^-7 * 2^-126 */
    } else if (e == 255) {
        v = (f == 0) ? INFINITY : NAN;
    } else {
        v = ldexp((double)(128 + f), e - 134); /* (1 + f/128) * 2^(e-127) */
    }
    return sign ? -v : v;
}

static double elem(const void *p, int dtype, int64_t idx)
{
    switch (dtype) {
    case ORACLE_F32: return (double)((const float *)p)[idx];
    case ORACLE_F16: return oracle_decode_f16(((const uint16_t *)p)[idx]);
    default:         return oracle_decode_bf16(((const uint16_t *)p)[idx]);
    }
}

/* Storage offsets of A(i,k), B(k,j) and C(i,j) for the chosen layout. */
static int64_t off_a(int layout, int64_t M, int64_t K, int64_t i, int64_t k)
{
    return layout == ORACLE_ROW_MAJOR ? i * K + k : i + k * M;
}
static int64_t off_b(int layout, int64_t K, int64_t N, int64_t k, int64_t j)
{
    return layout == ORACLE_ROW_MAJOR ? k * N + j : k + j * K;
}
static int64_t off_c(int layout, int64_t M, int64_t N, int64_t i, int64_t j)
{
    return layout == ORACLE_ROW_MAJOR ? i * N + j : i + j * M;
}

static int bad_args(int dtype, int layout, int64_t M, int64_t N, int64_t K)
{
    if (dtype < ORACLE_F32 || dtype > ORACLE_BF16) return 1;
    if (layout != ORACLE_ROW_MAJOR && layout != ORACLE_COL_MAJOR) return 1;
    if (M < 0 || N < 0 || K < 0) return 1;
    return 0;
}

/* One output row i of the product, written to acc[0..N) and sabs[0..N). */
static void one_row(int dtype, int layout, const void *A, const void *B,
                    int64_t M, int64_t N, int64_t K, int64_t i,
                    double *acc, double *sabs)
{
    for (int64_t j = 0; j < N; ++j) { acc[j] = 0.0; sabs[j] = 0.0; }
    for (int64_t k = 0; k < K; ++k) {
        double a = elem(A, dtype, off_a(layout, M, K, i, k));
        for (int64_t j = 0; j < N; ++j) {
            double p = a * elem(B, dtype, off_b(layout, K, N, k, j));
            acc[j] += p;
            sabs[j] += fabs(p);
        }
    }
}

/* Full product.  C and S (S may be NULL) are written in the problem's own layout. */
int oracle_gemm(int dtype, int layout, const void *A, const void *B,
                int64_t M, int64_t N, int64_t K, double *C, double *S)
{
    if (bad_args(dtype, layout, M, N, K)) return 1;
    if (M == 0 || N == 0) return 0;
    int err = 0;
#pragma omp parallel
    {
        double *acc = (double *)malloc(sizeof(double) * (size_t)N);
        double *sab = (double *)malloc(sizeof(double) * (size_t)N);
        if (!acc || !sab) {
#pragma omp atomic write
            err = 2;
        }
#pragma omp for schedule(static)
        for (int64_t i = 0; i < M; ++i) {
            if (!acc || !sab) continue;
            one_row(dtype, layout, A, B, M, N, K, i, acc, sab);
            for (int64_t j = 0; j < N; ++j) {
                C[off_c(layout, M, N, i, j)] = acc[j];
                if (S) S[off_c(layout, M, N, i, j)] = sab[j];
            }
        }
        free(acc);
        free(sab);
    }
    return err;
}

/* Selected rows only: C and S (S may be NULL) are nrows x N, row-major, row r
 * holding output row rows[r]. */
int oracle_gemm_rows(int dtype, int layout, const void *A, const void *B,
                     int64_t M, int64_t N, int64_t K,
                     const int64_t *rows, int64_t nrows, double *C, double *S)
{
    if (bad_args(dtype, layout, M, N, K)) return 1;
    for (int64_t r = 0; r < nrows; ++r)
        if (rows[r] < 0 || rows[r] >= M) return 1;
    int err = 0;
#pragma omp parallel
    {
        double *acc = (double *)malloc(sizeof(double) * (size_t)(N > 0 ? N : 1));
        double *sab = (double *)malloc(sizeof(double) * (size_t)(N > 0 ? N : 1));
        if (!acc || !sab) {
#pragma omp atomic write
            err = 2;
        }
#pragma omp for schedule(dynamic, 1)
        for (int64_t r = 0; r < nrows; ++r) {
            if (!acc || !sab) continue;
            one_row(dtype, layout, A, B, M, N, K, rows[r], acc, sab);
            memcpy(C + r * N, acc, sizeof(double) * (size_t)N);
            if (S) memcpy(S + r * N, sab, sizeof(double) * (size_t)N);
        }
        free(acc);
        free(sab);
    }
    return err;
}

/* Selected entries (ii[t], jj[t]), one dot product each. */
int oracle_gemm_entries(int dtype, int layout, const void *A, const void *B,
                        int64_t M, int64_t N, int64_t K,
                        const int64_t *ii, const int64_t *jj, int64_t n,
                        double *C, double *S)
{
    if (bad_args(dtype, layout, M, N, K)) return 1;
    for (int64_t t = 0; t < n; ++t)
        if (ii[t] < 0 || ii[t] >= M || jj[t] < 0 || jj[t] >= N) return 1;
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < n; ++t) {
        double acc = 0.0, sab = 0.0;
        for (int64_t k = 0; k < K; ++k) {
            double p = elem(A, dtype, off_a(layout, M, K, ii[t], k)) *
                       elem(B, dtype, off_b(layout, K, N, k, jj[t]));
            acc += p;
            sab += fabs(p);
        }
        C[t] = acc;
        if (S) S[t] = sab;
    }
    return 0;
}

/*
 * General form, one problem per batch index b = 0 .. batch-1:
 *
 *     C_b <- alpha * op(A_b) * op(B_b) + beta * C_b
 *
 * ("SGEMM measured and the three ledgers", section 2: the library call with
 * operation flags, leading dimensions and the row-/column-major reading of the
 * same bytes; section 3, kernel K1: C = alpha * acc + beta * C).  op(X) is X or
 * its transpose.  Storage of element (r, c) of a stored matrix with leading
 * dimension ld: row-major X[r*ld + c], column-major X[r + c*ld].  op(A) is
 * M x K: A is stored M x K (op 'N') or K x M (op 'T'); op(B) is K x N: B is
 * stored K x N or N x K; C is M x N.  Matrix b starts stride elements after
 * matrix b-1 (stride 0 reuses one matrix for every b).
 *
 * Outputs, each [batch, M, N] row-major and independent of the layout:
 *   C:  alpha * P + beta * c_in in double;
 *   P:  the plain product sum, sum_k op(A)[i,k] op(B)[k,j] (ascending k);
 *   S:  sum_k |op(A)[i,k] op(B)[k,j]|;
 *   BC: beta * c_in.
 * As in the BLAS convention, C_in is not read when beta == 0 (a NaN there does
 * not reach the result), and A and B are not read when alpha == 0 or K == 0
 * (the product term is then exactly zero).
 */
static int64_t off_stored(int layout, int64_t ld, int64_t r, int64_t c)
{
    return layout == ORACLE_ROW_MAJOR ? r * ld + c : r + c * ld;
}

int oracle_gemm_ex(int dtype, int layout, int op_a, int op_b,
                   int64_t M, int64_t N, int64_t K, double alpha,
                   const void *A, int64_t lda, int64_t stride_a,
                   const void *B, int64_t ldb, int64_t stride_b,
                   double beta, const void *Cin, int64_t ldc, int64_t stride_c,
                   int64_t batch, double *C, double *P, double *S, double *BC)
{
    if (bad_args(dtype, layout, M, N, K) || batch < 0) return 1;
    if ((op_a != 0 && op_a != 1) || (op_b != 0 && op_b != 1)) return 1;
    if (stride_a < 0 || stride_b < 0 || stride_c < 0) return 1;
    const int use_ab = alpha != 0.0 && K > 0;
    const int64_t rows = batch * M;
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        const int64_t b = r / M, i = r % M;
        double *c = C + r * N, *p = P + r * N, *s = S + r * N, *bc = BC + r * N;
        for (int64_t j = 0; j < N; ++j) { p[j] = 0.0; s[j] = 0.0; }
        if (use_ab) {
            const int64_t a0 = b * stride_a, b0 = b * stride_b;
            for (int64_t k = 0; k < K; ++k) {
                /* op(A)[i,k]: stored (i,k) for 'N', stored (k,i) for 'T' */
                const int64_t ia = op_a == 0 ? off_stored(layout, lda, i, k) : off_stored(layout, lda, k, i);
                const double a = elem(A, dtype, a0 + ia);
                for (int64_t j = 0; j < N; ++j) {
                    /* op(B)[k,j]: stored (k,j) for 'N', stored (j,k) for 'T' */
                    const int64_t ib = op_b == 0 ? off_stored(layout, ldb, k, j) : off_stored(layout, ldb, j, k);
                    const double v = a * elem(B, dtype, b0 + ib);
                    p[j] += v;
                    s[j] += fabs(v);
                }
            }
        }
        for (int64_t j = 0; j < N; ++j) {
            bc[j] = beta == 0.0 ? 0.0 : beta * elem(Cin, dtype, b * stride_c + off_stored(layout, ldc, i, j));
            c[j] = (use_ab ? alpha * p[j] : 0.0) + bc[j];
        }
    }
    return 0;
}

/*
 * FP8 E4M3FN ("Chapter 5 Operators and Runtime", section 5.4.3, example 5-7):
 * 1 sign bit, 4 exponent bits (bias 7), 3 fraction bits; largest finite value
 * 448; no infinities; S.1111.111 is NaN.  Subnormals (exponent field 0) are
 * f/8 * 2^-6.
 */
double oracle_decode_e4m3(uint8_t c)
{
    int sign = (c >> 7) & 1;
    int e = (c >> 3) & 0xF;
    int f = c & 0x7;
    double v;
    if (e == 15 && f == 7) {
        v = NAN;
    } else if (e == 0) {
        v = ldexp((double)f, -9);             /* f/8 * 2^-6 */
    } else {
        v = ldexp((double)(8 + f), e - 10);   /* (1 + f/8) * 2^(e-7) */
    }
    return sign ? -v : v;
}

/* Nearest E4M3FN value to x (ties to the even fraction), clamped to +-448 when
 * |x| exceeds it; NaN stays NaN.  Returns the code. */
uint8_t oracle_encode_e4m3(float x)
{
    if (x != x) return 0x7F;
    uint8_t sign = signbit(x) ? 0x80 : 0x00;
    double a = fabs((double)x);
    if (a >= 448.0) return sign | 0x7E;
    if (a == 0.0) return sign;
    int e;
    frexp(a, &e);                      /* a = m * 2^e, 0.5 <= m < 1: binade exponent e-1 */
    int be = e - 1;
    if (be < -6) be = -6;              /* subnormal range shares the spacing of binade -6 */
    double step = ldexp(1.0, be - 3);  /* 3 fraction bits */
    double q = nearbyint(a / step);    /* exact division by a power of two; ties to even */
    double v = q * step;
    if (v >= 448.0) return sign | 0x7E;
    if (v < ldexp(1.0, -6)) return sign | (uint8_t)q;           /* subnormal (or a rounded-up 8 -> normal below) */
    frexp(v, &e);
    be = e - 1;
    uint8_t frac = (uint8_t)(ldexp(v, 3 - be) - 8.0);
    return sign | (uint8_t)((be + 7) << 3) | frac;
}

/*
 * Row-wise quantisation of a half matrix A [M,K] (row-major) to E4M3FN with one
 * scale per row (example 5-7: the scale follows from the whole row's largest
 * magnitude, so the row is read completely before any element is quantised):
 *     amax_i  = max_k |a_ik|
 *     q_ik    = E4M3(a_ik * (448 / amax_i))     (448 / amax_i and the product in FP32)
 *     scale_i = amax_i / 448                    (FP32)
 * so that a_ik ~ q_ik * scale_i.  A row of zeros gives q = 0 and scale 0.
 * The two FP32 operations are written out so that the quantised codes, an
 * integer result decided by floating point, are decided in FP32 exactly as the
 * device does.
 */
int oracle_quantize_rows_e4m3(const uint16_t *A, int64_t M, int64_t K, uint8_t *Q, float *scale)
{
    if (M < 0 || K < 0) return 1;
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < M; ++i) {
        float amax = 0.0f;
        for (int64_t k = 0; k < K; ++k) {
            float a = (float)oracle_decode_f16(A[i * K + k]);
            if (fabsf(a) > amax) amax = fabsf(a);
        }
        if (amax == 0.0f) {
            for (int64_t k = 0; k < K; ++k) Q[i * K + k] = 0;
            scale[i] = 0.0f;
            continue;
        }
        volatile float inv = 448.0f / amax;
        for (int64_t k = 0; k < K; ++k) {
            volatile float x = (float)oracle_decode_f16(A[i * K + k]) * inv;
            Q[i * K + k] = oracle_encode_e4m3(x);
        }
        volatile float sc = amax / 448.0f;
        scale[i] = sc;
    }
    return 0;
}

/*
 * Product of the row-quantised input with E4M3 weights (example 5-8: FP8 input
 * times FP8 weights, FP16 output):
 *     C[i,j] = scale_i * sum_k q_ik * w_kj
 * Q is [M,K] row-major; the weights are given transposed, Wt [N,K] row-major
 * (Wt[j*K + k] = w_kj).  Products and sums in double (each product of two E4M3
 * values is exact); the scale multiplies the finished sum.  S[i,j] =
 * |scale_i| * sum_k |q_ik w_kj|.  C and S are [M,N] row-major; rows select
 * output rows (NULL: all M).
 */
int oracle_gemm_e4m3_rowscale(const uint8_t *Q, const float *scale, const uint8_t *Wt,
                              int64_t M, int64_t N, int64_t K,
                              const int64_t *rows, int64_t nrows, double *C, double *S)
{
    if (M < 0 || N < 0 || K < 0) return 1;
    if (!rows) nrows = M;
    for (int64_t r = 0; r < nrows; ++r)
        if (rows && (rows[r] < 0 || rows[r] >= M)) return 1;
#pragma omp parallel for schedule(dynamic, 4)
    for (int64_t r = 0; r < nrows; ++r) {
        const int64_t i = rows ? rows[r] : r;
        for (int64_t j = 0; j < N; ++j) {
            double acc = 0.0, sab = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                double p = oracle_decode_e4m3(Q[i * K + k]) * oracle_decode_e4m3(Wt[j * K + k]);
                acc += p;
                sab += fabs(p);
            }
            C[r * N + j] = (double)scale[i] * acc;
            S[r * N + j] = fabs((double)scale[i]) * sab;
        }
    }
    return 0;
}

int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Number of OpenMP threads the oracle's later calls use (n >= 1); for timing the
 * oracle on one core.  The results do not depend on it (see the loop order above). */
void oracle_set_num_threads(int n)
{
#ifdef _OPENMP
    if (n >= 1) omp_set_num_threads(n);
#else
    (void)n;
#endif
}
