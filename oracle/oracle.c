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
 * GGUF block formats (infr README, "Also validated for correctness": Q4_K_M
 * among the formats decoded on the GPU byte-identically to the CPU dequant;
 * footnote 3: routed expert banks stored as Q5_1; LLM170 README, status:
 * "q5_1 down" and "q4_K" MoE tiles). The pages name the formats but print no
 * layout; the layouts below are the block types of the ggml tensor library
 * that GGUF files carry (GGUF specification, ggml repository docs/gguf.md;
 * Q4_K from the k-quants change, llama.cpp pull request 1684). A row of K
 * weights is K/256 Q4_K blocks or K/32 Q5_1 blocks, rows one after another.
 *
 *   Q4_K, 256 weights in 144 bytes: fp16 d, fp16 dmin, 12 bytes holding
 *   eight 6-bit sub-block scales sc[j] and eight 6-bit minimums mn[j] (one
 *   pair per 32 weights), then 128 bytes of 4-bit q. Weight i has
 *   W^ = d * sc[i/32] * q - dmin * mn[i/32].
 *   Q5_1, 32 weights in 24 bytes: fp16 d, fp16 m, a 32-bit word of fifth
 *   bits, 16 bytes of low nibbles. W^ = d * q + m, q in [0, 31].
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

/* ------------------------------------------------------ GGUF block formats -- */

#define ORACLE_Q4_K 1
#define ORACLE_Q5_1 2

/* Weights and bytes per block; 0 for an unknown format. */
static int block_weights(int32_t fmt) { return fmt == ORACLE_Q4_K ? 256 : fmt == ORACLE_Q5_1 ? 32 : 0; }
static int block_bytes(int32_t fmt) { return fmt == ORACLE_Q4_K ? 144 : fmt == ORACLE_Q5_1 ? 24 : 0; }

/* Bytes of one row of K weights, or -1 if the format is unknown or K is not
 * a whole number of blocks. */
int64_t oracle_blocks_row_bytes(int32_t fmt, int64_t K)
{
    int bw = block_weights(fmt);
    if (bw == 0 || K < 0 || K % bw != 0) return -1;
    return K / bw * block_bytes(fmt);
}

static uint16_t le16(const uint8_t* p) { return (uint16_t)(p[0] | (p[1] << 8)); }

/* Sub-block j of a Q4_K block: its 6-bit scale and minimum. The twelve bytes
 * hold, for j < 4, sc[j] in the low 6 bits of byte j and mn[j] in the low 6
 * bits of byte j + 4; for j >= 4 the low 4 bits of sc[j] and of mn[j] are the
 * low and high nibble of byte j + 4, and their top 2 bits sit in the top 2
 * bits of byte j - 4 (sc) and byte j (mn). */
static void q4k_scale_min(const uint8_t* b12, int j, int* sc, int* mn)
{
    if (j < 4) {
        *sc = b12[j] & 63;
        *mn = b12[j + 4] & 63;
    } else {
        *sc = (b12[j + 4] & 0x0F) | ((b12[j - 4] >> 6) << 4);
        *mn = (b12[j + 4] >> 4) | ((b12[j] >> 6) << 4);
    }
}

/* One block as W^[i] = a[i] * q[i] + b[i]: the unsigned integer q and the
 * fp64 step a and offset b (exact products of fp16 values and small
 * integers). */
static void block_terms(int32_t fmt, const uint8_t* blk, int* q, double* a, double* b)
{
    if (fmt == ORACLE_Q4_K) {
        double d = oracle_half_to_double(le16(blk));
        double dmin = oracle_half_to_double(le16(blk + 2));
        const uint8_t* qs = blk + 16;
        for (int i = 0; i < 256; ++i) {
            /* 64 weights per 32 bytes: the first 32 in the low nibbles,
             * the next 32 in the high nibbles of the same bytes */
            int chunk = i / 64, r = i % 64;
            uint8_t byte = qs[32 * chunk + (r % 32)];
            int sc, mn;
            q4k_scale_min(blk + 4, i / 32, &sc, &mn);
            q[i] = r < 32 ? (byte & 0x0F) : (byte >> 4);
            a[i] = d * (double)sc;
            b[i] = -(dmin * (double)mn);
        }
    } else {
        double d = oracle_half_to_double(le16(blk));
        double m = oracle_half_to_double(le16(blk + 2));
        uint32_t qh = (uint32_t)blk[4] | ((uint32_t)blk[5] << 8) | ((uint32_t)blk[6] << 16) |
                      ((uint32_t)blk[7] << 24);
        const uint8_t* qs = blk + 8;
        for (int i = 0; i < 32; ++i) {
            /* weight i: low nibble of byte i (i < 16) or high nibble of byte
             * i - 16, plus bit i of qh as the fifth bit */
            int nib = i < 16 ? (qs[i] & 0x0F) : (qs[i - 16] >> 4);
            q[i] = nib | (int)(((qh >> i) & 1u) << 4);
            a[i] = d;
            b[i] = m;
        }
    }
}

/* W^ [N, K] in fp64 from the blocks [N, row_bytes]. */
void oracle_blocks_decode(int32_t fmt, const uint8_t* w, int64_t N, int64_t K, double* w_hat)
{
    int bw = block_weights(fmt), bb = block_bytes(fmt);
    int q[256];
    double a[256], b[256];
    for (int64_t n = 0; n < N; ++n)
        for (int64_t kb = 0; kb < K / bw; ++kb) {
            block_terms(fmt, w + (n * (K / bw) + kb) * bb, q, a, b);
            for (int i = 0; i < bw; ++i) w_hat[n * K + kb * bw + i] = a[i] * (double)q[i] + b[i];
        }
}

/* The same weights in fp32 as a CPU dequantizer forms them: step a and
 * offset b in fp32 (exact), then a * q (exact) plus b, rounded once. */
void oracle_blocks_decode_f32(int32_t fmt, const uint8_t* w, int64_t N, int64_t K, float* out)
{
    int bw = block_weights(fmt), bb = block_bytes(fmt);
    int q[256];
    double a[256], b[256];
    for (int64_t n = 0; n < N; ++n)
        for (int64_t kb = 0; kb < K / bw; ++kb) {
            block_terms(fmt, w + (n * (K / bw) + kb) * bb, q, a, b);
            for (int i = 0; i < bw; ++i) {
                float af = (float)a[i], bf = (float)b[i];
                float p = af * (float)q[i];
                out[n * K + kb * bw + i] = p + bf;
            }
        }
}

/* y[m,n] = sum_k x[m,k] * W^[n,k] in fp64, k ascending; absterm (if not NULL)
 * = sum_k |x[m,k]| * (|a q| + |b|), the size of the two parts a block format
 * adds up (for a format without offset it is sum_k |x W^|).
 * x: fp16 bits [M, K]; w: blocks [N, row_bytes]; y, absterm: fp64 [M, N]. */
void oracle_blocks_linear(int32_t fmt, const uint16_t* x, const uint8_t* w, int64_t M, int64_t N, int64_t K,
                          double* y, double* absterm)
{
    int bw = block_weights(fmt), bb = block_bytes(fmt);
    double* xd = (double*)malloc(sizeof(double) * (size_t)(M * K + 1));
    double* wr = (double*)malloc(sizeof(double) * (size_t)(K + 1));
    double* ar = (double*)malloc(sizeof(double) * (size_t)(K + 1));
    if (!xd || !wr || !ar) {
        free(xd);
        free(wr);
        free(ar);
        return;
    }
    int q[256];
    double a[256], b[256];
    for (int64_t i = 0; i < M * K; ++i) xd[i] = oracle_half_to_double(x[i]);
    for (int64_t n = 0; n < N; ++n) {
        for (int64_t kb = 0; kb < K / bw; ++kb) {
            block_terms(fmt, w + (n * (K / bw) + kb) * bb, q, a, b);
            for (int i = 0; i < bw; ++i) {
                wr[kb * bw + i] = a[i] * (double)q[i] + b[i];
                ar[kb * bw + i] = fabs(a[i] * (double)q[i]) + fabs(b[i]);
            }
        }
        for (int64_t m = 0; m < M; ++m) {
            const double* xr = xd + m * K;
            double acc = 0.0, aacc = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                acc += xr[k] * wr[k];
                aacc += fabs(xr[k]) * ar[k];
            }
            y[m * N + n] = acc;
            if (absterm) absterm[m * N + n] = aacc;
        }
    }
    free(xd);
    free(wr);
    free(ar);
}
