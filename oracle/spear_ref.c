/*
 * CPU oracle for the W4 + input-adaptive error-compensator linear.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing in the library links, loads or calls this
 * file; only the tests, the package smoke check and the benchmark's CPU
 * baseline do. It shares no code with the CUDA path.
 *
 * What it computes ("SPEAR: A System for Post-Quantization Error-Adaptive
 * Recovery", section 2.1A, Input-Adaptive Error Compensators): a quantised
 * linear whose effective weight for a token x is
 *
 *     W_eff(x) = W + alpha * B * diag(gamma(A x)) * A,
 *
 * where W is the dequantised 4-bit weight, A (r x K) projects x into a rank-r
 * space, gamma is the input-dependent gate and B (N x r) projects back. Applied
 * to x this is y = W x + alpha * B (gamma(z) (.) z) with z = A x, which is the
 * form evaluated here (section 2.1A, "Mechanism"). The gate is the elementwise
 * sigmoid, the constant 1 (the static low-rank correction W + alpha B A that
 * the paper contrasts with in section 1), or the bottleneck MLP the paper names
 * for gamma (section 2.1A, "Mechanism"): per token,
 *
 *     gamma(z) = sigmoid(W2 relu(W1 z)),  W1 (h x r), W2 (r x h),
 *
 * with relu as the hidden activation (the paper does not name it).
 *
 * Everything is fp64. Inputs are bf16 bit patterns widened exactly.
 * Dequantisation is w = (q - zp) * s with q the 4-bit code, zp the integer zero
 * point of its group and s the bf16 scale of its group (the 4-bit asymmetric
 * group-wise / per-channel setting of section 1 and section 3.1).
 *
 * Build: cc -O2 -fopenmp -shared -fPIC (no -ffast-math).
 *
 * SPEAR_PLANT=<n> compiles a deliberately wrong variant (one planted mistake
 * each) that the pin tests must reject; the default build plants nothing.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif
#ifndef SPEAR_PLANT
#define SPEAR_PLANT 0
#endif

/* bf16 bit pattern -> double, exact. */
static double bf16_to_double(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Code of column k in row n of the packed [N][K/2] byte array: even k in the
 * low nibble, odd k in the high nibble. */
static int code_at(const uint8_t *q, int K, int n, int k) {
    uint8_t byte = q[(size_t)n * (size_t)(K / 2) + (size_t)(k / 2)];
    if (SPEAR_PLANT == 1) return (k % 2 == 0) ? (byte >> 4) : (byte & 0x0F);
    return (k % 2 == 0) ? (byte & 0x0F) : (byte >> 4);
}

static int zero_at(const uint8_t *zp, int n_groups, int n, int g) {
    return zp ? (int)zp[(size_t)n * n_groups + g] : 8; /* no zeros given: symmetric, z = 8 */
}

/* Round a double to the nearest bf16, ties to even, by hand. */
static uint16_t bf16_rne(double v) {
    uint16_t sign = (v < 0.0 || (v == 0.0 && signbit(v))) ? 0x8000u : 0u;
    double a = fabs(v);
    if (a == 0.0) return sign;
    if (isnan(v)) return 0x7FC0u;
    if (isinf(v)) return (uint16_t)(sign | 0x7F80u);
    int e;
    (void)frexp(a, &e);          /* a = m * 2^e, 0.5 <= m < 1 */
    int E = e - 1;               /* a = 1.f * 2^E */
    if (E < -126) E = -126;      /* subnormal range: fixed quantum */
    double quantum = ldexp(1.0, E - 7);
    double t = a / quantum;      /* exact: division by a power of two */
    double fl = floor(t);
    double rem = t - fl;
    uint64_t n = (uint64_t)fl;
    if (SPEAR_PLANT == 6 ? rem >= 0.5 : (rem > 0.5 || (rem == 0.5 && (n & 1u)))) n += 1;
    if (n == 256) { n = 128; E += 1; }
    if (n < 128) return (uint16_t)(sign | (uint16_t)n);      /* subnormal (E == -126) */
    if (E + 127 >= 255) return (uint16_t)(sign | 0x7F80u);   /* overflow */
    return (uint16_t)(sign | (uint16_t)((E + 127) << 7) | (uint16_t)(n - 128));
}

/* Exact fp64 dequantised value of element (n, k). */
static double dequant_at(const uint8_t *q, const uint16_t *s, const uint8_t *zp,
                         int K, int G, int n, int k) {
    int n_groups = K / G;
    int g = (SPEAR_PLANT == 7) ? k / 128 % n_groups : k / G;
    int d = code_at(q, K, n, k) - zero_at(zp, n_groups, n, g);
    if (SPEAR_PLANT == 2) d = code_at(q, K, n, k) + zero_at(zp, n_groups, n, g) - 16;
    return (double)d * bf16_to_double(s[(size_t)n * n_groups + g]);
}

/* The gate applied to z: gamma(z) * z. gate 0 = sigmoid, gate 1 = constant one. */
static double gated(double z, int gate) {
    if (gate == 1) return z;
    if (SPEAR_PLANT == 3) return 1.0 / (1.0 + exp(-z));
    if (SPEAR_PLANT == 8) return z * (1.0 / (1.0 + exp(z)));
    return z * (1.0 / (1.0 + exp(-z)));
}

/* ---------------------------------------------------------------- exports */

/* Bottleneck-MLP gate for M tokens: t = relu(W1 z) (h values), gamma(z) =
 * sigmoid(W2 t) (r values), u = gamma(z) (.) z.
 * W1 bf16 [h][r]; W2 bf16 [r][h]; z, u double [M][r]. */
void oracle_gate_mlp(const double *z, int M, int r, int h, const uint16_t *W1, const uint16_t *W2,
                     double *u) {
    double *t = (double *)malloc(sizeof(double) * (size_t)(h > 0 ? h : 1));
    for (int m = 0; m < M; ++m) {
        const double *zm = z + (size_t)m * r;
        for (int i = 0; i < h; ++i) {
            double acc = 0.0;
            for (int j = 0; j < r; ++j)
                acc += bf16_to_double(W1[SPEAR_PLANT == 11 ? (size_t)j * h + i : (size_t)i * r + j]) * zm[j];
            t[i] = (SPEAR_PLANT == 10 || acc > 0.0) ? acc : 0.0;
        }
        for (int j = 0; j < r; ++j) {
            double acc = 0.0;
            for (int i = 0; i < h; ++i) acc += bf16_to_double(W2[(size_t)j * h + i]) * t[i];
            double g = SPEAR_PLANT == 12 ? acc : 1.0 / (1.0 + exp(-acc));
            u[(size_t)m * r + j] = g * zm[j];
        }
    }
    free(t);
}

/* bf16 dequantised weights, one RNE rounding of the exact (q - z) * s.
 * q uint8 [N][K/2]; s bf16 [N][K/G]; zp uint8 [N][K/G] or NULL; out bf16 [N][K]. */
void oracle_dequant_bf16(const uint8_t *q, const uint16_t *s, const uint8_t *zp,
                         int N, int K, int G, uint16_t *out) {
    #pragma omp parallel for schedule(static)
    for (int n = 0; n < N; ++n)
        for (int k = 0; k < K; ++k)
            out[(size_t)n * K + k] = bf16_rne(dequant_at(q, s, zp, K, G, n, k));
}

/* Same, exact fp64 values. */
void oracle_dequant_f64(const uint8_t *q, const uint16_t *s, const uint8_t *zp,
                        int N, int K, int G, double *out) {
    #pragma omp parallel for schedule(static)
    for (int n = 0; n < N; ++n)
        for (int k = 0; k < K; ++k)
            out[(size_t)n * K + k] = dequant_at(q, s, zp, K, G, n, k);
}

/* EC down-projection z[m][j] = sum_k A[j][k] x[m][k], then u = gamma(z) * z.
 * A bf16 [r][K]; x bf16 [M][K]; z, u double [M][r] (either may be NULL). */
void oracle_ec(const uint16_t *A, const uint16_t *x, int r, int K, int M, int gate,
               double *z_out, double *u_out) {
    #pragma omp parallel for collapse(2) schedule(static)
    for (int m = 0; m < M; ++m)
        for (int j = 0; j < r; ++j) {
            double acc = 0.0;
            for (int k = 0; k < K; ++k)
                acc += bf16_to_double(A[(size_t)j * K + k])
                       * bf16_to_double(x[(size_t)m * K + (SPEAR_PLANT == 9 ? (size_t)(K - 1 - k) : (size_t)k)]);
            if (z_out) z_out[(size_t)m * r + j] = acc;
            if (u_out) u_out[(size_t)m * r + j] = gated(acc, gate);
        }
}

/* Gate only: u[i] = gamma(z[i]) * z[i]. */
void oracle_gate(const double *z, int count, int gate, double *u) {
    for (int i = 0; i < count; ++i) u[i] = gated(z[i], gate);
}

/* Full forward for a set of output rows.
 *   y[m][i] = sum_k W[rows[i]][k] x[m][k] + alpha * sum_j B[rows[i]][j] u[m][j]
 * with u = gamma(A x) (.) (A x). rows == NULL means all N rows (nrows = N).
 * gate 2 (bottleneck MLP) reads gate_hidden, W1 and W2; the others ignore them.
 * rank == 0 (or A/B NULL) means no compensator. y is double [M][nrows].
 * nthreads <= 0 keeps the OpenMP default. */
void oracle_forward(const uint8_t *q, const uint16_t *s, const uint8_t *zp,
                    int N, int K, int G,
                    const uint16_t *A, const uint16_t *B, int rank, double alpha, int gate,
                    const uint16_t *x, int M,
                    const int64_t *rows, int nrows, double *y, int nthreads,
                    int gate_hidden, const uint16_t *W1, const uint16_t *W2) {
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#endif
    int use_ec = rank > 0 && A != NULL && B != NULL;
    double *u = NULL;
    if (use_ec) {
        u = (double *)malloc(sizeof(double) * (size_t)M * rank);
        if (gate == 2) {
            double *zz = (double *)malloc(sizeof(double) * (size_t)M * rank);
            oracle_ec(A, x, rank, K, M, 1, zz, NULL);
            oracle_gate_mlp(zz, M, rank, gate_hidden, W1, W2, u);
            free(zz);
        } else {
            oracle_ec(A, x, rank, K, M, gate, NULL, u);
        }
    }
    double *xd = (double *)malloc(sizeof(double) * (size_t)M * K);
    for (size_t i = 0; i < (size_t)M * K; ++i) xd[i] = bf16_to_double(x[i]);

    #pragma omp parallel
    {
        double *w = (double *)malloc(sizeof(double) * (size_t)K);
        #pragma omp for schedule(dynamic, 4)
        for (int i = 0; i < nrows; ++i) {
            int n = rows ? (int)rows[i] : i;
            for (int k = 0; k < K; ++k) w[k] = dequant_at(q, s, zp, K, G, n, k);
            for (int m = 0; m < M; ++m) {
                const double *xm = xd + (size_t)m * K;
                double acc = 0.0;
                for (int k = 0; k < K; ++k) acc += w[k] * xm[k];
                if (use_ec) {
                    double ec = 0.0;
                    for (int j = 0; j < rank; ++j)
                        ec += bf16_to_double(B[SPEAR_PLANT == 4 ? (size_t)j * N + n : (size_t)n * rank + j])
                              * u[(size_t)m * rank + j];
                    acc += (SPEAR_PLANT == 5 ? 1.0 : alpha) * ec;
                }
                y[(size_t)m * nrows + i] = acc;
            }
        }
        free(w);
    }
    free(xd);
    free(u);
}

/* Threads OpenMP would use (for reporting). */
int oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
