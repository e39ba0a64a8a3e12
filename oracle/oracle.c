/*
 * W4A16 group-quantized linear: plain CPU oracle (fp64, single thread).
 *
 * TEST INFRASTRUCTURE ONLY. Nothing in the product path may link, load or
 * call this file; only the test suite, the smoke check and the CPU-baseline
 * leg of the benchmark do. It shares no code, header, table or helper with
 * the CUDA library: the fp16 conversions below are written out here from
 * the IEEE 754 binary16 definition.
 *
 * What it computes (LLM170, introduction: "W4A16 (int4 sym g128, f16
 * activations)"; group 32 for the MoE models; Repository layout: "kernel
 * outputs must match the CPU reference"):
 *
 *   q[n,k]    = ((qw[n, k/2] >> (4 * (k mod 2))) & 0xF) - 8      (int4 sym)
 *   W^[n,k]   = s[n, k/g] * q[n,k]                              (g per group)
 *   y[m,n]    = sum_k x[m,k] * W^[n,k]        (fp64, k ascending)
 *
 * and the symmetric group quantizer that produces (qw, s) from fp32 weights:
 *   amax = max_k |w| over the group (fp32), s = fp16_rn(fp32(amax / 7)),
 *   q = clamp(rint(w / s), -8, 7) in fp32, all-zero group -> s = 0, q = 0,
 *   stored as the nibble q + 8, even k in the low nibble.
 *
 * Build: plain C99, no fast-math, -ffp-contract=off (no fused multiply-add
 * contraction), so that x86-64 and aarch64 hosts give bit-identical results.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ---------------------------------------------------------------- fp16 -- */

/* binary16 -> double, exact for every bit pattern (NaN stays NaN). */
double oracle_half_to_double(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1F;
    int f = h & 0x3FF;
    double v;
    if (e == 0)
        v = ldexp((double)f, -24);              /* zero or subnormal: f * 2^-24 */
    else if (e == 31)
        v = f ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + f), e - 25);  /* (1.f) * 2^(e-15) */
    return sign ? -v : v;
}

/* float -> binary16, round to nearest, ties to even; overflow -> +-inf. */
uint16_t oracle_float_to_half_rn(float fv)
{
    double v = (double)fv;                     /* exact */
    uint16_t sign = signbit(v) ? 0x8000 : 0;
    double a = fabs(v);
    if (isnan(v))
        return (uint16_t)(sign | 0x7E00);
    if (isinf(v))
        return (uint16_t)(sign | 0x7C00);
    if (a < ldexp(1.0, -14)) {
        /* subnormal range: multiples of 2^-24; rint rounds half to even.
         * A result of 1024 is exactly the smallest normal's bit pattern. */
        double r = rint(ldexp(a, 24));
        return (uint16_t)(sign | (uint16_t)r);
    }
    int E;
    (void)frexp(a, &E);                        /* a = m * 2^E, m in [0.5, 1) */
    int e = E - 1;                             /* a in [2^e, 2^(e+1)) */
    double r = rint(ldexp(a, 10 - e));         /* significand in [1024, 2048] */
    if (r == 2048.0) {
        r = 1024.0;
        e += 1;
    }
    if (e > 15)
        return (uint16_t)(sign | 0x7C00);
    return (uint16_t)(sign | (uint16_t)((e + 15) << 10) | (uint16_t)(r - 1024.0));
}

/* bulk helpers for the tests */
void oracle_half_to_double_n(const uint16_t* h, int64_t n, double* out)
{
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_half_to_double(h[i]);
}

void oracle_float_to_half_rn_n(const float* f, int64_t n, uint16_t* out)
{
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_float_to_half_rn(f[i]);
}

/* ------------------------------------------------------------ quantizer -- */

/* Symmetric int4 quantizer, one fp16 scale per group of g consecutive k.
 * w: fp32 [N, K] row-major. qw: uint8 [N, K/2]. s: fp16 bits [N, K/g]. */
void oracle_quantize(const float* w, int64_t N, int64_t K, int32_t g,
                     uint8_t* qw, uint16_t* s)
{
    int64_t G = K / g;
    for (int64_t n = 0; n < N; ++n) {
        const float* wr = w + n * K;
        memset(qw + n * (K / 2), 0, (size_t)(K / 2));
        for (int64_t j = 0; j < G; ++j) {
            float amax = 0.0f;
            for (int64_t k = j * g; k < (j + 1) * g; ++k) {
                float a = fabsf(wr[k]);
                if (a > amax) amax = a;
            }
            float t = amax / 7.0f;             /* fp32 quotient */
            uint16_t sh = oracle_float_to_half_rn(t);
            s[n * G + j] = sh;
            float sf = (float)oracle_half_to_double(sh);
            for (int64_t k = j * g; k < (j + 1) * g; ++k) {
                int q = 0;
                if (sf != 0.0f) {
                    float r = wr[k] / sf;      /* fp32 quotient */
                    float rr = rintf(r);       /* half to even */
                    if (rr > 7.0f) rr = 7.0f;
                    if (rr < -8.0f) rr = -8.0f;
                    q = (int)rr;
                }
                uint8_t nib = (uint8_t)(q + 8);
                qw[n * (K / 2) + k / 2] |= (uint8_t)(nib << (4 * (k & 1)));
            }
        }
    }
}

/* q[n,k] in [-8, 7] from the packed bytes. */
void oracle_unpack(const uint8_t* qw, int64_t N, int64_t K, int8_t* q)
{
    for (int64_t n = 0; n < N; ++n)
        for (int64_t k = 0; k < K; ++k) {
            uint8_t b = qw[n * (K / 2) + k / 2];
            int nib = (b >> (4 * (k & 1))) & 0xF;
            q[n * K + k] = (int8_t)(nib - 8);
        }
}

/* Inverse of oracle_unpack: bytes from q in [-8, 7]. */
void oracle_pack_q(const int8_t* q, int64_t N, int64_t K, uint8_t* qw)
{
    for (int64_t n = 0; n < N; ++n)
        for (int64_t j = 0; j < K / 2; ++j) {
            int lo = q[n * K + 2 * j] + 8;
            int hi = q[n * K + 2 * j + 1] + 8;
            qw[n * (K / 2) + j] = (uint8_t)((lo & 0xF) | ((hi & 0xF) << 4));
        }
}

/* W^[n,k] = s[n, k/g] * q[n,k] in fp64 (exact: 11-bit times 4-bit). */
void oracle_dequantize(const uint8_t* qw, const uint16_t* s, int64_t N, int64_t K,
                       int32_t g, double* w_hat)
{
    int64_t G = K / g;
    for (int64_t n = 0; n < N; ++n)
        for (int64_t k = 0; k < K; ++k) {
            uint8_t b = qw[n * (K / 2) + k / 2];
            int q = ((b >> (4 * (k & 1))) & 0xF) - 8;
            w_hat[n * K + k] = oracle_half_to_double(s[n * G + k / g]) * (double)q;
        }
}

/* ---------------------------------------------------------------- linear -- */

/* y[m,n] = sum_k x[m,k] * W^[n,k], fp64, k ascending. If absdot is not NULL
 * it receives sum_k |x[m,k] * W^[n,k]| (the scale of the rounding bound).
 * x: fp16 bits [M, K]; y, absdot: fp64 [M, N]. */
void oracle_linear(const uint16_t* x, const uint8_t* qw, const uint16_t* s,
                   int64_t M, int64_t N, int64_t K, int32_t g,
                   double* y, double* absdot)
{
    double* xd = (double*)malloc(sizeof(double) * (size_t)(M * K));
    double* wr = (double*)malloc(sizeof(double) * (size_t)K);
    if (!xd || !wr) {
        free(xd);
        free(wr);
        return;
    }
    for (int64_t i = 0; i < M * K; ++i) xd[i] = oracle_half_to_double(x[i]);
    for (int64_t n = 0; n < N; ++n) {
        oracle_dequantize(qw + n * (K / 2), s + n * (K / g), 1, K, g, wr);
        for (int64_t m = 0; m < M; ++m) {
            const double* xr = xd + m * K;
            double acc = 0.0, aacc = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                double p = xr[k] * wr[k];
                acc += p;
                aacc += fabs(p);
            }
            y[m * N + n] = acc;
            if (absdot) absdot[m * N + n] = aacc;
        }
    }
    free(xd);
    free(wr);
}

/* Grouped (routed-expert) linear: rows offsets[e] <= r < offsets[e+1] of the
 * expert-sorted activations use expert e's weights.
 * x: fp16 [R, K]; qw: [E, N, K/2]; s: [E, N, K/g]; offsets: int32 [E+1]
 * (offsets[0] = 0, non-decreasing, offsets[E] = R); y, absdot: fp64 [R, N]. */
void oracle_grouped_linear(const uint16_t* x, const uint8_t* qw, const uint16_t* s,
                           const int32_t* offsets, int32_t E, int64_t R, int64_t N,
                           int64_t K, int32_t g, double* y, double* absdot)
{
    (void)R;
    for (int32_t e = 0; e < E; ++e) {
        int64_t r0 = offsets[e], r1 = offsets[e + 1];
        if (r1 <= r0) continue;
        oracle_linear(x + r0 * K, qw + (int64_t)e * N * (K / 2), s + (int64_t)e * N * (K / g),
                      r1 - r0, N, K, g, y + r0 * N, absdot ? absdot + r0 * N : NULL);
    }
}
