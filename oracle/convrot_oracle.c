/*
 * Oracle for the INT8 convrot linear layer.
 *
 * TEST INFRASTRUCTURE ONLY. This file is a plain, slow, fp64 CPU statement of
 * what the layer computes, written from the page "INT8 Convrot Safetensors"
 * (stable-diffusion.cpp docs, int8_convrot.md). Only the test-suite, the
 * package's smoke check and the benchmark's CPU-baseline leg may load it. It
 * shares no code, header, table or helper with the CUDA library, and the CUDA
 * library never calls it.
 *
 * Every step follows the page's formulas in the page's order, with no
 * blocking, fusion or reordering:
 *
 *   H4            "How INT8 convrot works": the printed 4x4 matrix / 2.
 *   R_G           "How INT8 convrot works": the normalized Kronecker power of
 *                 H4 for G = 4^n, applied to every contiguous group of G
 *                 input features (block-diagonal R).
 *   X_rot = X R   "How INT8 convrot works" / "Runtime activation quantization".
 *   s, Q          "Weight quantization" and "Runtime activation quantization":
 *                 s = max_i |rot[i]| / 127, Q = clamp(round(rot / s), -127, 127).
 *   A = Q_x Q_w^T "Runtime activation quantization": signed 32-bit sums.
 *   Y             "Runtime activation quantization": A * s_x[r] * s_w[o] + b[o].
 *
 * Readings where the page is silent (each one is listed in the design notes):
 *   - "round" is round half away from zero (C's round()).
 *   - The scales are stored as fp32 ("floating-point" scales); the pre-round
 *     value divides the fp64 rotated value by that stored fp32 scale.
 *   - A row whose rotated values are all zero has s = 0 and Q = 0.
 *   - The bias is fp32 and may be absent (then it is 0).
 *
 * Two rotation routines exist. oracle_rotate_dense multiplies each group by
 * the dense matrix R_G (the definition). oracle_rotate_fast uses the
 * mixed-product property of the Kronecker product: H4 (x) ... (x) H4 applied
 * to a vector is H4 applied along each base-4 digit of the index in turn.
 * The tests check each against the other and both against a closed form.
 *
 * Rows are independent; when compiled with -fopenmp the row loops run in
 * parallel. Results do not depend on the thread count.
 */
#define _GNU_SOURCE
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* The matrix printed in "How INT8 convrot works", before the division by 2. */
static const double kH4Printed[4][4] = {
    {1, 1, 1, -1},
    {1, 1, -1, 1},
    {1, -1, 1, 1},
    {-1, 1, 1, 1},
};

/* Returns n if G == 4^n with n >= 1, else -1. */
int oracle_log4(int64_t G)
{
    int n = 0;
    if (G < 4) return -1;
    while (G > 1) {
        if (G % 4 != 0) return -1;
        G /= 4;
        n++;
    }
    return n;
}

/* H4 row-major into out[16]: the printed matrix divided by 2. */
void oracle_h4(double *out)
{
    for (int i = 0; i < 4; i++)
        for (int j = 0; j < 4; j++) out[i * 4 + j] = kH4Printed[i][j] / 2.0;
}

/*
 * Dense R_G = H4 (x) H4 (x) ... (x) H4 (n factors), G x G row-major.
 * Built by the recursion M_1 = H4, M_{t+1} = kron(M_t, H4).
 * Returns 0, or -1 if G is not a power of four with n >= 1.
 */
int oracle_rotation_matrix(int64_t G, double *R)
{
    int n = oracle_log4(G);
    if (n < 0) return -1;
    double h4[16];
    oracle_h4(h4);
    double *cur = (double *)malloc(sizeof(double) * (size_t)G * (size_t)G);
    double *nxt = (double *)malloc(sizeof(double) * (size_t)G * (size_t)G);
    if (!cur || !nxt) {
        free(cur);
        free(nxt);
        return -1;
    }
    int64_t d = 4;
    memcpy(cur, h4, sizeof(h4));
    for (int t = 1; t < n; t++) {
        /* kron(cur[d x d], H4) -> nxt[4d x 4d]: nxt[4a+c][4b+e] = cur[a][b] * H4[c][e] */
        int64_t D = d * 4;
        for (int64_t a = 0; a < d; a++)
            for (int64_t b = 0; b < d; b++)
                for (int c = 0; c < 4; c++)
                    for (int e = 0; e < 4; e++)
                        nxt[(4 * a + c) * D + (4 * b + e)] = cur[a * d + b] * h4[c * 4 + e];
        double *tmp = cur;
        cur = nxt;
        nxt = tmp;
        d = D;
    }
    memcpy(R, cur, sizeof(double) * (size_t)G * (size_t)G);
    free(cur);
    free(nxt);
    return 0;
}

/*
 * X_rot = X R with R block-diagonal (one R_G per contiguous group), by the
 * definition: xr[r][g*G + i] = sum_j X[r][g*G + j] * R_G[j][i].
 * X is fp32 [m, ldx]; Xrot is fp64 [m, k] (dense, leading dimension k).
 */
void oracle_rotate_dense(const float *X, int64_t m, int64_t k, int64_t ldx, int64_t G,
                         const double *RG, double *Xrot)
{
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < m; r++) {
        const float *x = X + r * ldx;
        double *y = Xrot + r * k;
        for (int64_t g = 0; g < k / G; g++) {
            for (int64_t i = 0; i < G; i++) {
                double acc = 0.0;
                for (int64_t j = 0; j < G; j++) acc += (double)x[g * G + j] * RG[j * G + i];
                y[g * G + i] = acc;
            }
        }
    }
}

/*
 * Same X_rot by the Kronecker mixed-product property: for each base-4 digit
 * position p of the in-group index, replace every 4-tuple of entries that
 * differ only in digit p by H4 applied to it. (R_G is symmetric, so applying
 * it to a row vector from the right equals applying it to a column vector.)
 */
void oracle_rotate_fast(const float *X, int64_t m, int64_t k, int64_t ldx, int64_t G,
                        double *Xrot)
{
    int n = oracle_log4(G);
    double h4[16];
    oracle_h4(h4);
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < m; r++) {
        double *y = Xrot + r * k;
        for (int64_t i = 0; i < k; i++) y[i] = (double)X[r * ldx + i];
        for (int64_t g = 0; g < k / G; g++) {
            double *v = y + g * G;
            int64_t stride = 1;
            for (int p = 0; p < n; p++) {
                for (int64_t base = 0; base < G; base++) {
                    if ((base / stride) % 4 != 0) continue; /* digit p of base must be 0 */
                    double in[4], out[4];
                    for (int c = 0; c < 4; c++) in[c] = v[base + c * stride];
                    for (int c = 0; c < 4; c++) {
                        double acc = 0.0;
                        for (int e = 0; e < 4; e++) acc += in[e] * h4[e * 4 + c];
                        out[c] = acc;
                    }
                    for (int c = 0; c < 4; c++) v[base + c * stride] = out[c];
                }
                stride *= 4;
            }
        }
    }
}

/* Round half away from zero, then clamp to [-127, 127]. */
static int8_t quant_code(double v)
{
    double q = round(v);
    if (q > 127.0) q = 127.0;
    if (q < -127.0) q = -127.0;
    return (int8_t)q;
}

/*
 * Per-row scale and int8 codes from rotated rows ("Weight quantization",
 * "Runtime activation quantization"):
 *   scale[r] = (float)(max_i |rot[r][i]| / 127)
 *   v[r][i]  = rot[r][i] / (double)scale[r]       (pre-round value)
 *   Q[r][i]  = clamp(round(v[r][i]), -127, 127)
 * rot is fp64 [m, k]; Q is int8 [m, ldq]; entries k..ldq-1 of each Q row are
 * left untouched. pre_round may be NULL; else fp64 [m, k].
 * A zero row (or a scale that rounds to zero in fp32) gives scale 0, v 0, Q 0.
 */
void oracle_quantize_rows(const double *rot, int64_t m, int64_t k, float *scale, int8_t *Q,
                          int64_t ldq, double *pre_round)
{
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < m; r++) {
        const double *x = rot + r * k;
        double amax = 0.0;
        for (int64_t i = 0; i < k; i++) {
            double a = fabs(x[i]);
            if (a > amax) amax = a;
        }
        float s = (float)(amax / 127.0);
        scale[r] = s;
        for (int64_t i = 0; i < k; i++) {
            double v = (s == 0.0f) ? 0.0 : x[i] / (double)s;
            if (pre_round) pre_round[r * k + i] = v;
            Q[r * ldq + i] = quant_code(v);
        }
    }
}

/*
 * A[r][o] = sum_i Qx[r][i] * Qw[o][i] over i < k ("Runtime activation
 * quantization"), summed in int64 and stored as int32.
 * Returns 0, or -1 if any sum is outside the signed 32-bit range (the page
 * accumulates in signed 32-bit integers, so such a K is not representable).
 */
int oracle_gemm_i32(const int8_t *Qx, int64_t m, int64_t ldqx, const int8_t *Qw, int64_t n,
                    int64_t ldqw, int64_t k, int32_t *A, int64_t lda)
{
    int bad = 0;
#pragma omp parallel for schedule(static) reduction(| : bad)
    for (int64_t r = 0; r < m; r++) {
        for (int64_t o = 0; o < n; o++) {
            int64_t acc = 0;
            for (int64_t i = 0; i < k; i++) acc += (int64_t)Qx[r * ldqx + i] * (int64_t)Qw[o * ldqw + i];
            if (acc > INT32_MAX || acc < INT32_MIN) bad = 1;
            A[r * lda + o] = (int32_t)acc;
        }
    }
    return bad ? -1 : 0;
}

/*
 * Y[r][o] = A[r][o] * s_x[r] * s_w[o] + b[o], evaluated in fp64 and stored
 * as fp32 ("Runtime activation quantization"). bias may be NULL. Y_f64 may be
 * NULL; else it receives the fp64 values [m, n] before the fp32 store.
 */
void oracle_reconstruct(const int32_t *A, int64_t lda, int64_t m, int64_t n, const float *sx,
                        const float *sw, const float *bias, float *Y, int64_t ldy, double *Y_f64)
{
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < m; r++) {
        for (int64_t o = 0; o < n; o++) {
            double y = (double)A[r * lda + o] * (double)sx[r] * (double)sw[o];
            if (bias) y += (double)bias[o];
            if (Y_f64) Y_f64[r * n + o] = y;
            Y[r * ldy + o] = (float)y;
        }
    }
}

/*
 * Activation after the linear, for the up projection of a DiT MLP (the page's
 * layer is a plain linear; the MLP applies GELU to its output before the down
 * projection packs it). GELU(v) = v * Phi(v), Phi the standard normal CDF
 * (Hendrycks and Gimpel, "Gaussian Error Linear Units"):
 *   act 1: 0.5 v (1 + erf(v / sqrt 2))                       (exact form)
 *   act 2: 0.5 v (1 + tanh(sqrt(2 / pi) (v + 0.044715 v^3)))  (their tanh approximation)
 *   act 0: v
 * Applied in place to count fp64 values.
 */
void oracle_activation(double *v, int64_t count, int act)
{
    for (int64_t i = 0; i < count; i++) {
        const double x = v[i];
        if (act == 1)
            v[i] = 0.5 * x * (1.0 + erf(x / sqrt(2.0)));
        else if (act == 2)
            v[i] = 0.5 * x * (1.0 + tanh(sqrt(2.0 / M_PI) * (x + 0.044715 * x * x * x)));
    }
}

/*
 * Runtime LoRA correction ("Backend support", paragraph on adapters): from the
 * original, unrotated activation, D = scale * (X A^T) B^T, with A [r, k]
 * (down) and B [n, r] (up), in fp64. T [m, r] receives X A^T (may be NULL).
 * D is [m, n] with row pitch n.
 */
void oracle_lora_delta(const float *X, int64_t m, int64_t k, int64_t ldx, const float *A, int64_t r,
                       const float *B, int64_t n, double scale, double *T, double *D)
{
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < m; i++) {
        double t[256];
        double *ti = T ? T + i * r : t;
        for (int64_t j = 0; j < r; j++) {
            double acc = 0.0;
            for (int64_t c = 0; c < k; c++) acc += (double)X[i * ldx + c] * (double)A[j * k + c];
            ti[j] = acc;
        }
        for (int64_t o = 0; o < n; o++) {
            double acc = 0.0;
            for (int64_t j = 0; j < r; j++) acc += ti[j] * (double)B[o * r + j];
            D[i * n + o] = scale * acc;
        }
    }
}

/*
 * Whole pack of rows: rotate (fast form) then quantize. Used for the
 * activation pack and for the offline weight quantization, which the page
 * defines with the same formulas. Q is int8 [m, ldq]; columns k..ldq-1 are
 * set to zero. pre_round may be NULL. Returns 0, or -1 on a bad G or
 * allocation failure.
 */
int oracle_pack_rows(const float *X, int64_t m, int64_t k, int64_t ldx, int64_t G, float *scale,
                     int8_t *Q, int64_t ldq, double *pre_round)
{
    if (oracle_log4(G) < 0 || k % G != 0) return -1;
    double *rot = (double *)malloc(sizeof(double) * (size_t)(m > 0 ? m : 1) * (size_t)k);
    if (!rot) return -1;
    oracle_rotate_fast(X, m, k, ldx, G, rot);
    oracle_quantize_rows(rot, m, k, scale, Q, ldq, pre_round);
    for (int64_t r = 0; r < m; r++)
        for (int64_t i = k; i < ldq; i++) Q[r * ldq + i] = 0;
    free(rot);
    return 0;
}

#ifdef _OPENMP
#include <omp.h>
#endif

/* Threads the row loops above will use (1 without OpenMP). */
int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
