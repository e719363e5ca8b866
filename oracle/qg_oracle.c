/*
 * CPU oracle for the Q8_0 / bf16 decode matrix-vector path.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the slow, plain statement of what the
 * decode path computes.  Only the test suite, the smoke check and the benchmark's
 * CPU-baseline leg may load it.  It shares no code, header or table with the CUDA
 * library, and the CUDA library never calls it.
 *
 * Sources (web pages; sections named as they appear on the page):
 *   [Phobos]  "Filling in the blanks: Inference using Phobos"
 *   [Herbert] "One level down: #002 the same compiler on a GPU"
 *
 * What the pages fix, and what is a reading (the readings are listed again in the
 * design notes at the repository root):
 *   - A Q8_0 block is 32 int8 values that carry one scale ([Phobos] Fast Decode).
 *     The scale is IEEE binary16 (reading; the page names the format only).
 *   - Decode does the dot products in int8 end to end and applies each block's
 *     scale once per 32 values ([Phobos] Fast Decode).
 *   - Activation quantization (reading): d = max|x| / 127 in f32,
 *     q = round-half-away-from-zero(x / d) in f32, stored scale = fp16(d).
 *   - RMSNorm (reading): r = 1 / sqrt(mean(x^2) + eps), evaluated in f64 and
 *     rounded once to f32; x_hat = (x * r) * gamma in f32.
 *   - bf16 weights and activations with f32 accumulation ([Herbert] The
 *     numerical contract); the oracle accumulates in f64, where every bf16*bf16
 *     product is exact.
 *   - SiLU(gate) * up on the stacked halves and the folded residual add
 *     ([Herbert] Emitting for a GPU; [Phobos] Fast Decode).
 *
 * Everything real-valued is evaluated in f64.  Each block term d_w * d_x * S_b is
 * exact in f64 (11 + 11 + 20 significant bits), so a GEMV output is the f64 sum
 * of exact terms, and ``a`` (the sum of the terms' magnitudes) is returned beside
 * it for the tolerance model of the tests.
 *
 * Build: cc -O2 -ffp-contract=off -fPIC -shared -o liboracle.so qg_oracle.c -lm
 * (no FMA contraction, no fast-math: every f32 operation is one IEEE operation).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define QK 32

/* ------------------------------------------------------------------------ */
/* IEEE 754 binary16 and bfloat16 from their definitions                     */
/* ------------------------------------------------------------------------ */

/* Round the finite, non-negative value v to a multiple of quantum q, ties to
 * even multiple.  v / q is exact in f64 for the ranges used here (q is a power
 * of two and v is an f32 value). */
static double round_to_quantum_rne(double v, double q)
{
    double m = v / q;
    double f = floor(m);
    double frac = m - f;
    if (frac > 0.5 || (frac == 0.5 && fmod(f, 2.0) != 0.0))
        f += 1.0;
    return f * q;
}

/* Encode a finite non-negative value that is exactly representable in a binary
 * format with `mbits` stored fraction bits and exponent bias `bias`.  Returns the
 * magnitude bits, or the infinity pattern when the exponent is out of range. */
static uint32_t encode_exact(double v, int mbits, int bias, int emax_field)
{
    if (v == 0.0)
        return 0;
    double min_normal = ldexp(1.0, 1 - bias);
    if (v < min_normal) { /* subnormal: v = frac * 2^(1-bias-mbits) */
        return (uint32_t)(v / ldexp(1.0, 1 - bias - mbits));
    }
    int e2;
    double m = frexp(v, &e2); /* v = m * 2^e2, m in [0.5, 1) */
    int e = e2 - 1;           /* v = (2m) * 2^e, 2m in [1, 2) */
    int field = e + bias;
    if (field >= emax_field)
        return (uint32_t)emax_field << mbits; /* infinity */
    uint32_t frac = (uint32_t)((2.0 * m - 1.0) * ldexp(1.0, mbits));
    return ((uint32_t)field << mbits) | frac;
}

/* f32 -> binary16 bits, round to nearest, ties to even; subnormals kept,
 * overflow to infinity, NaN kept as a quiet NaN. */
uint16_t orc_f32_to_f16(float x)
{
    uint32_t u;
    memcpy(&u, &x, 4);
    uint16_t sign = (uint16_t)((u >> 16) & 0x8000u);
    if (isnan(x))
        return (uint16_t)(sign | 0x7e00u | ((u >> 13) & 0x3ffu));
    double a = fabs((double)x);
    if (isinf(x))
        return (uint16_t)(sign | 0x7c00u);
    /* quantum of the binade of a (binary16: 10 fraction bits, min exponent -14) */
    double q;
    if (a < ldexp(1.0, -14)) {
        q = ldexp(1.0, -24);
    } else {
        int e2;
        frexp(a, &e2);
        q = ldexp(1.0, (e2 - 1) - 10);
    }
    double r = round_to_quantum_rne(a, q);
    return (uint16_t)(sign | encode_exact(r, 10, 15, 31));
}

double orc_f16_to_f64(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int field = (h >> 10) & 0x1f;
    int frac = h & 0x3ff;
    double v;
    if (field == 0)
        v = ldexp((double)frac, -24);
    else if (field == 31)
        v = frac ? NAN : INFINITY;
    else
        v = ldexp(1024.0 + frac, field - 25);
    return sign ? -v : v;
}

/* f32 -> bfloat16 bits (8 exponent bits, 7 fraction bits), round to nearest,
 * ties to even; subnormals kept, overflow to infinity, NaN kept quiet. */
uint16_t orc_f32_to_bf16(float x)
{
    uint32_t u;
    memcpy(&u, &x, 4);
    uint16_t sign = (uint16_t)((u >> 16) & 0x8000u);
    if (isnan(x))
        return (uint16_t)(sign | 0x7fc0u | ((u >> 16) & 0x3fu));
    if (isinf(x))
        return (uint16_t)(sign | 0x7f80u);
    double a = fabs((double)x);
    double q;
    if (a < ldexp(1.0, -126)) {
        q = ldexp(1.0, -133);
    } else {
        int e2;
        frexp(a, &e2);
        q = ldexp(1.0, (e2 - 1) - 7);
    }
    double r = round_to_quantum_rne(a, q);
    return (uint16_t)(sign | encode_exact(r, 7, 127, 255));
}

double orc_bf16_to_f64(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4); /* bf16 is the top half of an f32 pattern */
    return (double)f;
}

/* Array forms of the converters (same definitions, element by element). */
void orc_f32_to_f16_array(const float *x, int64_t n, uint16_t *out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = orc_f32_to_f16(x[i]);
}

void orc_f32_to_bf16_array(const float *x, int64_t n, uint16_t *out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = orc_f32_to_bf16(x[i]);
}

void orc_f16_to_f64_array(const uint16_t *h, int64_t n, double *out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = orc_f16_to_f64(h[i]);
}

/* ------------------------------------------------------------------------ */
/* Q8_0 weight layout: canonical 34-byte blocks -> value and scale planes     */
/* ------------------------------------------------------------------------ */

/* [Phobos] GPU Performance Heisenbugs: weights are re-laid out so that decode
 * reads whole cache lines.  Canonical block = { fp16 d (little-endian), int8
 * qs[32] }; planes = qs[n][k] and d[n][k/32].  A pure byte permutation. */
void orc_q8_0_pack(const uint8_t *blocks, int64_t n_rows, int64_t k, int8_t *qs, uint16_t *d)
{
    int64_t nb = k / QK;
    for (int64_t n = 0; n < n_rows; ++n) {
        for (int64_t b = 0; b < nb; ++b) {
            const uint8_t *blk = blocks + (n * nb + b) * 34;
            d[n * nb + b] = (uint16_t)(blk[0] | ((uint16_t)blk[1] << 8));
            for (int i = 0; i < QK; ++i)
                qs[n * k + b * QK + i] = (int8_t)blk[2 + i];
        }
    }
}

/* ------------------------------------------------------------------------ */
/* Activation quantization to Q8_0                                            */
/* ------------------------------------------------------------------------ */

/* One 32-value block: d = max|v| / 127 (f32), q = round half away from zero of
 * v / d (one IEEE f32 division), clamped to [-127, 127]; d == 0 gives q = 0.
 * The stored scale is fp16(d).  [Phobos] Fast Decode: an activation is
 * quantized once to Q8_0 and shared by every projection that reads it. */
static void quantize_block(const float *v, int8_t *q, uint16_t *d_out)
{
    float amax = 0.0f;
    for (int i = 0; i < QK; ++i) {
        float a = fabsf(v[i]);
        if (a > amax)
            amax = a;
    }
    float d = amax / 127.0f;
    for (int i = 0; i < QK; ++i) {
        float t = (d != 0.0f) ? v[i] / d : 0.0f;
        float r = roundf(t); /* C roundf: halfway cases away from zero */
        if (r > 127.0f)
            r = 127.0f;
        if (r < -127.0f)
            r = -127.0f;
        q[i] = (int8_t)r;
    }
    *d_out = orc_f32_to_f16(d);
}

void orc_quantize_q8_0(const float *x, int64_t rows, int64_t k, int8_t *q, uint16_t *d)
{
    int64_t nb = k / QK;
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t b = 0; b < nb; ++b)
            quantize_block(x + r * k + b * QK, q + r * k + b * QK, d + r * nb + b);
}

/* ------------------------------------------------------------------------ */
/* RMSNorm                                                                    */
/* ------------------------------------------------------------------------ */

/* r = 1 / sqrt(mean(x^2) + eps), in f64 (every square of an f32 is exact in
 * f64), rounded once to f32.  [Herbert] Emitting for a GPU: the normalization
 * is fused with the projection that follows it; [Phobos] Q4_K_M: the fast norm
 * kernel.  Neither page fixes eps or the precision: those are readings. */
float orc_rms_inv(const float *x, int64_t k, float eps)
{
    double s = 0.0;
    for (int64_t i = 0; i < k; ++i)
        s += (double)x[i] * (double)x[i];
    double mean = s / (double)k;
    double r = 1.0 / sqrt(mean + (double)eps);
    return (float)r;
}

/* x_hat_i = (x_i * r) * gamma_i, two f32 multiplies; then Q8_0 quantization of
 * x_hat.  r_out and xhat_out may be NULL. */
void orc_rmsnorm_quantize(const float *x, const float *gamma, int64_t k, float eps,
                          int8_t *q, uint16_t *d, float *r_out, float *xhat_out)
{
    float r = orc_rms_inv(x, k, eps);
    float blk[QK];
    for (int64_t b = 0; b < k / QK; ++b) {
        for (int i = 0; i < QK; ++i) {
            float xr = x[b * QK + i] * r;
            blk[i] = xr * gamma[b * QK + i];
            if (xhat_out)
                xhat_out[b * QK + i] = blk[i];
        }
        quantize_block(blk, q + b * QK, d + b);
    }
    if (r_out)
        *r_out = r;
}

/* ------------------------------------------------------------------------ */
/* Block dots and the block-scaled GEMV                                       */
/* ------------------------------------------------------------------------ */

/* S[beta][n][b] = sum_{i<32} w_q[n][32b+i] * x_q[beta][32b+i], exact in int32
 * (|S| <= 32 * 127 * 127).  [Phobos] Fast Decode: the math runs in int8 end to
 * end (dp4a), one scale per 32 values. */
void orc_block_dots(const int8_t *wq, int64_t n_rows, int64_t k, const int8_t *xq,
                    int64_t batch, int32_t *s)
{
    int64_t nb = k / QK;
    for (int64_t be = 0; be < batch; ++be)
        for (int64_t n = 0; n < n_rows; ++n)
            for (int64_t b = 0; b < nb; ++b) {
                int32_t acc = 0;
                for (int i = 0; i < QK; ++i)
                    acc += (int32_t)wq[n * k + b * QK + i] * (int32_t)xq[be * k + b * QK + i];
                s[(be * n_rows + n) * nb + b] = acc;
            }
}

/* y[beta][n] = sum_b d_w[n][b] * d_x[beta][b] * S_b  (f64; each term exact),
 * a[beta][n] = sum_b |d_w[n][b] * d_x[beta][b] * S_b|.
 * [Phobos] Fast Decode: a warp owns an output row and does the whole
 * multiply-and-add for it, including the scales.  Also the prefill form with
 * batch = prompt rows ([Phobos] Fast Decode: prompt processing reuses every
 * weight once per prompt row). */
void orc_gemv_q8_0(const int8_t *wq, const uint16_t *wd, int64_t n_rows, int64_t k,
                   const int8_t *xq, const uint16_t *xd, int64_t batch, double *y, double *a)
{
    int64_t nb = k / QK;
    for (int64_t be = 0; be < batch; ++be) {
        for (int64_t n = 0; n < n_rows; ++n) {
            double sum = 0.0, mag = 0.0;
            for (int64_t b = 0; b < nb; ++b) {
                int32_t s = 0;
                for (int i = 0; i < QK; ++i)
                    s += (int32_t)wq[n * k + b * QK + i] * (int32_t)xq[be * k + b * QK + i];
                double term = orc_f16_to_f64(wd[n * nb + b]) * orc_f16_to_f64(xd[be * nb + b]) * (double)s;
                sum += term;
                mag += fabs(term);
            }
            y[be * n_rows + n] = sum;
            if (a)
                a[be * n_rows + n] = mag;
        }
    }
}

/* ------------------------------------------------------------------------ */
/* Epilogues                                                                  */
/* ------------------------------------------------------------------------ */

/* silu(g) = g / (1 + exp(-g)); h = silu(g) * u, in f64.  The gate rows are the
 * first half of the stacked output and the up rows the second half ([Herbert]
 * Emitting for a GPU: gate and up computed in one projection). */
void orc_silu_mul(const double *g, const double *u, int64_t n, double *h)
{
    for (int64_t i = 0; i < n; ++i)
        h[i] = g[i] / (1.0 + exp(-g[i])) * u[i];
}

/* Rotation of the normalised activation ([Phobos] PrismML Ternary-Bonsai-2-27B:
 * the format applies a Hadamard matrix transform to the activation, which
 * spreads outliers over the block, and the rotated activation is computed once
 * and shared by every projection that reads the same input).  Reading: the
 * Walsh-Hadamard matrix of order 128 (the format's block of 128 weights) in
 * Sylvester order, unnormalised (entries +1 / -1, H H^T = 128 I), applied to
 * each consecutive block of 128 values:
 *   z[128 b + i] = sum_j (-1)^popcount(i & j) x[128 b + j],
 * evaluated term by term in f64 from the definition (n a multiple of 128). */
void orc_hadamard128(const float *x, int64_t n, double *z)
{
    for (int64_t b = 0; b < n / 128; ++b) {
        for (int i = 0; i < 128; ++i) {
            double sum = 0.0;
            for (int j = 0; j < 128; ++j) {
                int bits = i & j, par = 0;
                while (bits) {
                    par ^= bits & 1;
                    bits >>= 1;
                }
                const double v = (double)x[128 * b + j];
                sum += par ? -v : v;
            }
            z[128 * b + i] = sum;
        }
    }
}

/* Residual folded into the last product ([Phobos] Fast Decode): out[n] =
 * res[n] + y[n] in f64 (res is f32, so exact in f64; y is the exact f64 value of
 * the block-scaled sum). */
void orc_residual_add(const float *res, const double *y, int64_t n, double *out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = (double)res[i] + y[i];
}

/* One decode feed-forward block, every step in the pages' order ([Phobos] Fast
 * Decode: quantize the activation once and share it between the stacked
 * projections, fold the residual add into the last matmul; [Herbert] Emitting
 * for a GPU: norm in front of the stacked gate|up, activation behind it):
 *   q, d   = Q8_0(RMSNorm(x) * gamma)                    (orc_rmsnorm_quantize)
 *   g | u  = stacked gate|up rows [0, F) | [F, 2F)        (orc_gemv_q8_0, f64)
 *   h      = f32(silu(g) * u)                             (orc_silu_mul, then one f32 rounding)
 *   hq, hd = Q8_0(h)                                      (orc_quantize_q8_0)
 *   out    = x + down(hq, hd)                             (orc_gemv_q8_0, orc_residual_add)
 * Outputs (caller-allocated): xq int8[k], xd u16[k/32], r f32[1], gu f64[2F],
 * a_gu f64[2F], h64 f64[F], h f32[F], hq int8[F], hd u16[F/32], y f64[k],
 * a_y f64[k], out f64[k]. */
void orc_decode_ffn(const float *x, const float *gamma, int64_t k, int64_t ffn, float eps,
                    const int8_t *gu_qs, const uint16_t *gu_d, const int8_t *dn_qs,
                    const uint16_t *dn_d, int8_t *xq, uint16_t *xd, float *r, double *gu,
                    double *a_gu, double *h64, float *h, int8_t *hq, uint16_t *hd, double *y,
                    double *a_y, double *out)
{
    float *xhat = (float *)calloc((size_t)k, sizeof(float));
    if (!xhat)
        return;
    orc_rmsnorm_quantize(x, gamma, k, eps, xq, xd, r, xhat);
    free(xhat);
    orc_gemv_q8_0(gu_qs, gu_d, 2 * ffn, k, xq, xd, 1, gu, a_gu);
    orc_silu_mul(gu, gu + ffn, ffn, h64);
    for (int64_t i = 0; i < ffn; ++i)
        h[i] = (float)h64[i];
    orc_quantize_q8_0(h, 1, ffn, hq, hd);
    orc_gemv_q8_0(dn_qs, dn_d, k, ffn, hq, hd, 1, y, a_y);
    orc_residual_add(x, y, k, out);
}

/* ------------------------------------------------------------------------ */
/* bf16 projection with the norm in front                                     */
/* ------------------------------------------------------------------------ */

/* [Herbert] The numerical contract: bf16 weights and activations, f32
 * accumulators.  With gamma != NULL the input is RMSNorm'd first ([Herbert]
 * Emitting for a GPU): x_hat = bf16((x * r) * gamma) with r from orc_rms_inv
 * over the f32 values of x; without gamma x_hat = x.  y[n] = sum_k w[n][k] *
 * x_hat[k] in f64 (each bf16 product is exact), a[n] = sum_k |w x_hat|. */
void orc_gemv_bf16(const uint16_t *w, int64_t n_rows, int64_t k, const uint16_t *x,
                   const uint16_t *gamma, float eps, uint16_t *xhat, float *r_out,
                   double *y, double *a)
{
    /* xhat: caller-provided bf16[k] that receives the normalised input */
    float r = 1.0f;
    if (gamma) {
        float *xf = (float *)calloc((size_t)k, sizeof(float));
        if (!xf)
            return;
        for (int64_t i = 0; i < k; ++i)
            xf[i] = (float)orc_bf16_to_f64(x[i]);
        r = orc_rms_inv(xf, k, eps);
        for (int64_t i = 0; i < k; ++i) {
            float xr = xf[i] * r;
            float t = xr * (float)orc_bf16_to_f64(gamma[i]);
            xhat[i] = orc_f32_to_bf16(t);
        }
        free(xf);
    } else {
        for (int64_t i = 0; i < k; ++i)
            xhat[i] = x[i];
    }
    if (r_out)
        *r_out = r;
    for (int64_t n = 0; n < n_rows; ++n) {
        double sum = 0.0, mag = 0.0;
        for (int64_t i = 0; i < k; ++i) {
            double p = orc_bf16_to_f64(w[n * k + i]) * orc_bf16_to_f64(xhat[i]);
            sum += p;
            mag += fabs(p);
        }
        y[n] = sum;
        if (a)
            a[n] = mag;
    }
}
