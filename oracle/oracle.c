/*
 * Plain fp64 CPU oracle for the 4/8-bit group-quantised decode projection.
 *
 * TEST INFRASTRUCTURE ONLY. Only tests/, __graft_entry__.smoke() and the
 * cpu_baseline / reference legs of bench.py may load this library. The CUDA
 * library shares no code, header, table or constant with it.
 *
 * Every function here is the plain definition of what the fast path computes,
 * written with naive loops in double precision, no blocking and no reordering
 * beyond the natural index order:
 *
 *   - weight format: MLX affine group quantisation, w = scale*q + bias, one
 *     bf16 scale and one bf16 bias per 64 consecutive K elements, q packed
 *     32/bits values per uint32 along K (uzu page, "Internals 1: models are
 *     assembled from configuration", weight_matrix row of the table: MLX
 *     4/8-bit originals consumed as-is; TensorFold page, box smoke-test table,
 *     "info" row: "4-bit group 64").
 *   - nibble order inside a word is not stated on the pages; the reading used
 *     is least-significant first: element j of a word sits in bits
 *     [bits*j, bits*j + bits).
 *   - projection y[m][n] = sum_k x[m][k] * w[n][k] (W row-major [N][K]).
 *   - RMSNorm folded ahead of a projection (Husky page, "Four implementation
 *     elements of MSI": the preceding normalisation is merged into each
 *     projection kernel): xn = x / sqrt(mean(x^2) + eps) * gamma.
 *   - gate and up processed together with a SwiGLU epilogue (same section):
 *     h = silu(g) * u, silu(g) = g / (1 + exp(-g)).
 *   - MoE routing (uzu page, same table, mlp row: MixtureOfExperts with a
 *     routing function): top-k of the router logits, descending, ties to the
 *     lower expert index, softmax over the k selected logits.
 *   - input randomized Hadamard transform (uzu page, same table, linear row:
 *     an input-side RHT block that spreads quantisation error): the pages give
 *     no block size or layout; the reading used is, per block of `block`
 *     consecutive columns (64 = one quantisation group), xr = H (d .* x) /
 *     sqrt(block) with H the Sylvester-ordered Walsh-Hadamard matrix and d a
 *     +-1 vector stored as bits, least-significant first, bit set = -1.
 *   - NVFP4 weights (TensorFold page, "qualified" model table: NVFP4 checkpoints):
 *     the pages give no layout; the reading is NVIDIA's published NVFP4 format
 *     (E2M1 codes, an E4M3 scale per 16 K elements, an fp32 scale per matrix),
 *     weights only, spelled out above oracle_e2m1 below.
 *
 * Parity pins for every function live in tests/test_oracle_pins.py.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* bf16 -> double is exact: a bf16 is the top half of an IEEE fp32. */
static double bf16_to_double(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* q[n][k] for a row-major [N][K] matrix whose rows are packed along K. */
int oracle_unpack(const uint32_t *wq, int64_t N, int64_t K, int bits, uint8_t *q)
{
    if (bits != 4 && bits != 8)
        return 1;
    const int64_t per_word = 32 / bits;
    if (K % per_word != 0)
        return 1;
    const int64_t words_per_row = K / per_word;
    const uint32_t mask = (1u << bits) - 1u;
    for (int64_t n = 0; n < N; ++n) {
        for (int64_t k = 0; k < K; ++k) {
            uint32_t word = wq[n * words_per_row + k / per_word];
            int shift = (int)(bits * (k % per_word));
            q[n * K + k] = (uint8_t)((word >> shift) & mask);
        }
    }
    return 0;
}

/* w[n][k] = scale[n][k/group] * q[n][k] + bias[n][k/group], in double. */
int oracle_dequant(const uint32_t *wq, const uint16_t *scales, const uint16_t *biases,
                   int64_t N, int64_t K, int bits, int group, double *w)
{
    if (group <= 0 || K % group != 0)
        return 1;
    uint8_t *q = (uint8_t *)malloc((size_t)(N * K));
    if (!q)
        return 2;
    int rc = oracle_unpack(wq, N, K, bits, q);
    if (rc) {
        free(q);
        return rc;
    }
    const int64_t groups = K / group;
    for (int64_t n = 0; n < N; ++n) {
        for (int64_t k = 0; k < K; ++k) {
            double s = bf16_to_double(scales[n * groups + k / group]);
            double b = bf16_to_double(biases[n * groups + k / group]);
            w[n * K + k] = s * (double)q[n * K + k] + b;
        }
    }
    free(q);
    return 0;
}

/*
 * y[m][n] = sum_k x[m][k] * w[n][k] over a quantised W, dequantised one row at
 * a time (the row is the definition above; it is materialised per row only to
 * avoid holding all of W in doubles). absdot[m][n] = sum_k |x[m][k] * w[n][k]|
 * is returned beside it because the parity tolerance is stated in terms of it.
 * x has row stride ldx. absdot may be NULL.
 */
int oracle_qlinear(const double *x, int64_t ldx, int64_t M,
                   const uint32_t *wq, const uint16_t *scales, const uint16_t *biases,
                   int64_t N, int64_t K, int bits, int group,
                   double *y, double *absdot)
{
    if (group <= 0 || K % group != 0 || (bits != 4 && bits != 8))
        return 1;
    const int64_t per_word = 32 / bits;
    const int64_t words_per_row = K / per_word;
    const int64_t groups = K / group;
    double *wrow = (double *)malloc((size_t)K * sizeof(double));
    if (!wrow)
        return 2;
    for (int64_t n = 0; n < N; ++n) {
        int rc = oracle_dequant(wq + n * words_per_row, scales + n * groups,
                                biases + n * groups, 1, K, bits, group, wrow);
        if (rc) {
            free(wrow);
            return rc;
        }
        for (int64_t m = 0; m < M; ++m) {
            double acc = 0.0, acc_abs = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                double p = x[m * ldx + k] * wrow[k];
                acc += p;
                acc_abs += fabs(p);
            }
            y[m * N + n] = acc;
            if (absdot)
                absdot[m * N + n] = acc_abs;
        }
    }
    free(wrow);
    return 0;
}

/* xn[m][k] = x[m][k] / sqrt(sum_k x[m][k]^2 / K + eps) * gamma[k]. */
void oracle_rmsnorm(const double *x, int64_t M, int64_t K, const double *gamma,
                    double eps, double *xn)
{
    for (int64_t m = 0; m < M; ++m) {
        double ss = 0.0;
        for (int64_t k = 0; k < K; ++k)
            ss += x[m * K + k] * x[m * K + k];
        double denom = sqrt(ss / (double)K + eps);
        for (int64_t k = 0; k < K; ++k)
            xn[m * K + k] = x[m * K + k] / denom * gamma[k];
    }
}

/* silu(g) = g / (1 + exp(-g)), evaluated without overflow for large |g|. */
static double silu(double g)
{
    if (g >= 0.0)
        return g / (1.0 + exp(-g));
    double e = exp(g);
    return g * e / (1.0 + e);
}

/* h[i] = silu(g[i]) * u[i]. */
void oracle_swiglu(const double *g, const double *u, int64_t n, double *h)
{
    for (int64_t i = 0; i < n; ++i)
        h[i] = silu(g[i]) * u[i];
}

/*
 * Router: per row, the top_k experts by logit (descending; equal logits go to
 * the lower expert index), then the softmax of the selected logits:
 * w_j = exp(l_j - l_max) / sum_i exp(l_i - l_max). Selection is a repeated
 * linear scan for the best remaining candidate; comparisons are on the fp32
 * logits themselves.
 */
int oracle_topk_softmax(const float *logits, int64_t M, int64_t E, int64_t top_k,
                        int32_t *idx, double *w)
{
    if (top_k <= 0 || top_k > E)
        return 1;
    unsigned char *taken = (unsigned char *)malloc((size_t)E);
    if (!taken)
        return 2;
    for (int64_t m = 0; m < M; ++m) {
        const float *l = logits + m * E;
        memset(taken, 0, (size_t)E);
        for (int64_t j = 0; j < top_k; ++j) {
            int64_t best = -1;
            for (int64_t e = 0; e < E; ++e) {
                if (taken[e])
                    continue;
                if (best < 0 || l[e] > l[best])
                    best = e; /* strict '>' keeps the lower index on ties */
            }
            taken[best] = 1;
            idx[m * top_k + j] = (int32_t)best;
        }
        double lmax = (double)l[idx[m * top_k]];
        double denom = 0.0;
        for (int64_t j = 0; j < top_k; ++j)
            denom += exp((double)l[idx[m * top_k + j]] - lmax);
        for (int64_t j = 0; j < top_k; ++j)
            w[m * top_k + j] = exp((double)l[idx[m * top_k + j]] - lmax) / denom;
    }
    free(taken);
    return 0;
}

/* Input randomized Hadamard transform, row by row and block by block:
 * out[m][b*block + i] = sum_j H[i][j] * d[b*block + j] * x[m][b*block + j] / sqrt(block),
 * H[i][j] = (-1)^popcount(i & j), computed with the textbook in-place butterflies
 * (stride 1, 2, 4, ...: (a, b) -> (a + b, a - b)), which give exactly that order.
 * signs: bit k % 8 of byte k / 8 set means d[k] = -1. block: a power of two
 * dividing K. Returns nonzero on a bad block size. */
int oracle_rht(const double *x, int64_t M, int64_t K, const uint8_t *signs, int64_t block, double *out)
{
    if (block < 1 || (block & (block - 1)) != 0 || K % block != 0)
        return 1;
    const double scale = 1.0 / sqrt((double)block);
    for (int64_t m = 0; m < M; ++m) {
        for (int64_t k0 = 0; k0 < K; k0 += block) {
            double *v = out + m * K + k0;
            for (int64_t j = 0; j < block; ++j) {
                const int64_t k = k0 + j;
                const int neg = (signs[k / 8] >> (k % 8)) & 1;
                v[j] = neg ? -x[m * K + k] : x[m * K + k];
            }
            for (int64_t h = 1; h < block; h *= 2)
                for (int64_t i = 0; i < block; i += 2 * h)
                    for (int64_t j = i; j < i + h; ++j) {
                        const double a = v[j], b = v[j + h];
                        v[j] = a + b;
                        v[j + h] = a - b;
                    }
            for (int64_t j = 0; j < block; ++j)
                v[j] *= scale;
        }
    }
    return 0;
}

/* ---------------------------------------------------------------- NVFP4 weight code
 *
 * The TensorFold page lists NVFP4 checkpoints among the weight formats it serves but
 * gives no layout. The reading used is NVIDIA's published NVFP4 format, weights only
 * (activations stay bf16, as for every other code here):
 *   - element: 4-bit E2M1, bit 3 sign, bits 2-1 exponent (bias 1), bit 0 mantissa;
 *     exponent 0 is subnormal (0 or 0.5);
 *   - block scale: one E4M3 byte per 16 consecutive K elements, bit 7 sign, bits
 *     6-3 exponent (bias 7), bits 2-0 mantissa, exponent 0 subnormal, S.1111.111
 *     NaN, no infinities;
 *   - one fp32 scale per matrix: w[n][k] = global * e4m3(scale[n][k/16]) * e2m1(q[n][k]);
 *   - codes two per byte along K, the even column in the low nibble. */

double oracle_e2m1(int code)
{
    const int sign = (code >> 3) & 1, e = (code >> 1) & 3, m = code & 1;
    const double v = e == 0 ? 0.5 * m : ldexp(1.0 + 0.5 * m, e - 1);
    return sign ? -v : v;
}

double oracle_e4m3(int code)
{
    const int sign = (code >> 7) & 1, e = (code >> 3) & 15, m = code & 7;
    double v;
    if (e == 15 && m == 7)
        v = NAN;
    else if (e == 0)
        v = ldexp(m / 8.0, -6);
    else
        v = ldexp(1.0 + m / 8.0, e - 7);
    return sign ? -v : v;
}

/* w[n][k] in double, [N][K]. codes uint8 [N][K/2], scales uint8 [N][K/16]. */
int oracle_nvfp4_dequant(const uint8_t *codes, const uint8_t *scales, double global, int64_t N, int64_t K,
                         double *w)
{
    if (K <= 0 || K % 16 != 0)
        return 1;
    for (int64_t n = 0; n < N; ++n)
        for (int64_t k = 0; k < K; ++k) {
            const uint8_t byte = codes[n * (K / 2) + k / 2];
            const int q = (k % 2) ? byte >> 4 : byte & 15;
            w[n * K + k] = global * oracle_e4m3(scales[n * (K / 16) + k / 16]) * oracle_e2m1(q);
        }
    return 0;
}

/* y[m][n] = sum_k x[m][k] * w[n][k] over NVFP4 weights, one dequantised row at a time
 * (as oracle_qlinear); absdot[m][n] = sum_k |x[m][k] * w[n][k]| (may be NULL). */
int oracle_nvfp4_qlinear(const double *x, int64_t ldx, int64_t M, const uint8_t *codes, const uint8_t *scales,
                         double global, int64_t N, int64_t K, double *y, double *absdot)
{
    if (K <= 0 || K % 16 != 0)
        return 1;
    double *wrow = (double *)malloc((size_t)K * sizeof(double));
    if (!wrow)
        return 2;
    for (int64_t n = 0; n < N; ++n) {
        oracle_nvfp4_dequant(codes + n * (K / 2), scales + n * (K / 16), global, 1, K, wrow);
        for (int64_t m = 0; m < M; ++m) {
            double acc = 0.0, acc_abs = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                const double p = x[m * ldx + k] * wrow[k];
                acc += p;
                acc_abs += fabs(p);
            }
            y[m * N + n] = acc;
            if (absdot)
                absdot[m * N + n] = acc_abs;
        }
    }
    free(wrow);
    return 0;
}
