/*
 * Plain CPU oracle for the fused GEMM epilogue  C = act(A . B + bias).
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or
 * call this file: only the test suite, the smoke check and the benchmark's
 * CPU-baseline leg use it.  It shares no code, header, table or helper with
 * the CUDA library.
 *
 * What it follows:
 *  - "从零开始学习 TileLang：从 Python、PyTorch 到高性能 GPU Kernel 的完整开发教程",
 *    ch.10 §10.1: C[i,j] = sum_{k<K} A[i,k] * B[k,j]; §10.8 "GEMM Epilogue 融合":
 *    the bias is indexed by the output column and added before the ReLU
 *    (relu(a @ b + bias)); §10.7 precision recipe: fp16/bf16 inputs,
 *    fp32 accumulation, fp16/bf16 output.
 *  - "Writing high-performance kernels in TileLang", section "Écrivons un GEMM":
 *    the activation is max(x, 0) applied to the accumulator before the store.
 *  - "TileLang で GPU カーネル設計を解説", §4: bias has shape (N,) in the input dtype;
 *    the GELU epilogue, tanh form written as a sigmoid,
 *    gelu(x) = x / (1 + exp(-1.5957691216 * (x + 0.044715 * x^3))), applied after
 *    the bias (the printed bullet in "x + 0.044715·x•x·x" is read as a product).
 *
 * How: every fp16/bf16 input is decoded exactly to double; each output element
 * is the in-order fp64 sum over k of exact products, then (optionally) plus the
 * bias, then (optionally) the ReLU or the GELU.  The rounding to the output dtype is a
 * separate call (round-to-nearest-even, overflow to +-Inf), so tests can keep
 * the unrounded fp64 value for tolerance checks.  Rows run in parallel under
 * OpenMP when it is available; nothing else is reordered or blocked.
 *
 * Readings taken where the pages are silent:
 *  - ReLU(x) = x if x > 0, +0.0 if x <= 0 (so -0.0 becomes +0.0), NaN stays NaN
 *    (the pages test against torch.relu, which propagates NaN).
 *  - Output dtype = input dtype; rounding is IEEE round-to-nearest-even.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { ORACLE_F16 = 0, ORACLE_BF16 = 1 };
enum { ORACLE_EPI_NONE = 0, ORACLE_EPI_RELU = 1, ORACLE_EPI_BIAS = 2, ORACLE_EPI_BIAS_RELU = 3,
       ORACLE_EPI_GELU = 4, ORACLE_EPI_BIAS_GELU = 5 };

/* The tanh-form GELU as the page prints it (2*sqrt(2/pi) = 1.5957691216...). */
static double gelu_tanh(double x) {
    return x / (1.0 + exp(-1.5957691216 * (x + 0.044715 * x * x * x)));
}

/* Format parameters: mantissa bits (without the hidden bit), exponent bits. */
static void fmt_params(int dtype, int *mbits, int *ebits) {
    if (dtype == ORACLE_BF16) { *mbits = 7; *ebits = 8; }
    else { *mbits = 10; *ebits = 5; }
}

/* Exact decode of a 16-bit IEEE-style binary format to double. */
static double decode16(uint16_t h, int dtype) {
    int mbits, ebits;
    fmt_params(dtype, &mbits, &ebits);
    const int bias = (1 << (ebits - 1)) - 1;
    const int sign = (h >> (mbits + ebits)) & 1;
    const int e = (h >> mbits) & ((1 << ebits) - 1);
    const int m = h & ((1 << mbits) - 1);
    double v;
    if (e == 0) {
        v = ldexp((double)m, 1 - bias - mbits);               /* subnormal or zero */
    } else if (e == (1 << ebits) - 1) {
        v = m ? NAN : INFINITY;
    } else {
        v = ldexp((double)(m | (1 << mbits)), e - bias - mbits);
    }
    return sign ? -v : v;
}

/* Round a double to the nearest 16-bit value, ties to even, overflow to Inf. */
static uint16_t encode16_rne(double x, int dtype) {
    int mbits, ebits;
    fmt_params(dtype, &mbits, &ebits);
    const int bias = (1 << (ebits - 1)) - 1;
    const int emin = 1 - bias, emax = bias;
    const uint16_t sgn = signbit(x) ? (uint16_t)(1u << (mbits + ebits)) : 0;
    const uint16_t expall = (uint16_t)(((1u << ebits) - 1) << mbits);
    if (isnan(x)) return (uint16_t)(sgn | expall | (1u << (mbits - 1)));
    double a = fabs(x);
    if (isinf(a)) return (uint16_t)(sgn | expall);
    if (a == 0.0) return sgn;
    int e2;
    frexp(a, &e2);
    int E = e2 - 1;                        /* a lies in [2^E, 2^(E+1)) */
    if (E < emin) E = emin;                /* subnormal range: fixed quantum */
    const double hidden = ldexp(1.0, mbits);
    double r = nearbyint(ldexp(a, mbits - E));   /* significand in units of the quantum */
    if (r >= 2.0 * hidden) { E += 1; r = hidden; }
    if (E > emax) return (uint16_t)(sgn | expall);
    if (r < hidden) return (uint16_t)(sgn | (uint16_t)r);          /* subnormal */
    return (uint16_t)(sgn | (uint16_t)((E + bias) << mbits) | (uint16_t)(r - hidden));
}

int oracle_decode(const uint16_t *in, double *out, int64_t n, int dtype) {
    if (dtype != ORACLE_F16 && dtype != ORACLE_BF16) return -1;
    for (int64_t i = 0; i < n; ++i) out[i] = decode16(in[i], dtype);
    return 0;
}

int oracle_round(const double *in, uint16_t *out, int64_t n, int dtype) {
    if (dtype != ORACLE_F16 && dtype != ORACLE_BF16) return -1;
    for (int64_t i = 0; i < n; ++i) out[i] = encode16_rne(in[i], dtype);
    return 0;
}

/*
 * out[r*N + j] = epi( sum_k A[i*lda + k] * B[k*ldb + j] (+ bias[j]) ),  i = rows[r]
 * (or i = r when rows == NULL, nrows == M).  Returns 0, or -1 on a bad argument.
 */
int oracle_gemm_epilogue_f64(const uint16_t *A, const uint16_t *B, const uint16_t *bias,
                             double *out, int64_t M, int64_t N, int64_t K,
                             int64_t lda, int64_t ldb, const int64_t *rows, int64_t nrows,
                             int dtype, int epilogue) {
    if (M < 0 || N < 0 || K < 0 || lda < K || ldb < N) return -1;
    if (dtype != ORACLE_F16 && dtype != ORACLE_BF16) return -1;
    if (epilogue < ORACLE_EPI_NONE || epilogue > ORACLE_EPI_BIAS_GELU) return -1;
    const int use_bias = (epilogue == ORACLE_EPI_BIAS || epilogue == ORACLE_EPI_BIAS_RELU ||
                          epilogue == ORACLE_EPI_BIAS_GELU);
    const int use_relu = (epilogue == ORACLE_EPI_RELU || epilogue == ORACLE_EPI_BIAS_RELU);
    const int use_gelu = (epilogue == ORACLE_EPI_GELU || epilogue == ORACLE_EPI_BIAS_GELU);
    if (use_bias && bias == NULL) return -1;
    if (rows == NULL) nrows = M;
    for (int64_t r = 0; r < nrows && rows; ++r)
        if (rows[r] < 0 || rows[r] >= M) return -1;
    if (nrows == 0 || N == 0) return 0;

    /* B decoded once to double: exact. */
    double *Bd = (double *)malloc((size_t)(K > 0 ? K : 1) * (size_t)N * sizeof(double));
    if (!Bd) return -2;
    for (int64_t k = 0; k < K; ++k)
        for (int64_t j = 0; j < N; ++j) Bd[k * N + j] = decode16(B[k * ldb + j], dtype);

#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t r = 0; r < nrows; ++r) {
        const int64_t i = rows ? rows[r] : r;
        double *acc = out + r * N;
        for (int64_t j = 0; j < N; ++j) acc[j] = 0.0;
        for (int64_t k = 0; k < K; ++k) {
            const double a = decode16(A[i * lda + k], dtype);
            const double *brow = Bd + k * N;
            for (int64_t j = 0; j < N; ++j) acc[j] += a * brow[j];
        }
        for (int64_t j = 0; j < N; ++j) {
            double v = acc[j];
            if (use_bias) v += decode16(bias[j], dtype);
            if (use_relu && !isnan(v) && !(v > 0.0)) v = 0.0;
            if (use_gelu) v = gelu_tanh(v);
            acc[j] = v;
        }
    }
    free(Bd);
    return 0;
}

int oracle_max_threads(void) {
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
