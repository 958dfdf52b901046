/*
 * oracle.c -- the CPU oracle. TEST INFRASTRUCTURE ONLY (see oracle.h).
 *
 * Plain single-threaded C, written from definitions:
 *  - the IEEE-754 binary16 / bfloat16 and OCP FP8 E4M3 / FP4 E2M1 number formats;
 *  - BlockToFloat dequantization, i.e. the CPU reference the on-core decode was
 *    held bit-exact against ("feat(BACKEND-TENSTORRENT-KEEPQUANT): the 27B arm —
 *    on-core decode residency, TT grouped keep-quant GEMM, e2e gate", the W4
 *    residency paragraph: the word-shadow decode matched the CPU BlockToFloat bit
 *    for bit);
 *  - the matmul seam Y = X . W^T with W packed, one matrix (E = 1) or a stacked
 *    expert tower weight[E*N, K] (same issue, scope item 2 and the "Re-anchor"
 *    comment);
 *  - dequantize-then-matvec as the reference a fused kernel is compared with
 *    ("A 320B MoE on a free Kaggle TPU", section "What I actually ran");
 *  - NVFP4 E2M1 codes with E4M3 block scales and row-scaled FP8 weights, and the
 *    activation quantizer for W4A4 prefill ("I Built a Custom Blackwell Kernel for
 *    Qwen3.8-27B", section "What the custom path actually does").
 * Byte sizes: Q8_0 34 B / 32 values, Q6_K 210 B / 256 ("#3030", "Budget on the
 * 32 GB P150"); Q4_K 144 B / 256 (fp16 d, fp16 dmin, 12 B of 6-bit scales and
 * mins, 128 B of nibbles), Q5_K 176 B / 256 (the 5-bit member of the same K-quant
 * family, named with Q4_K/Q6_K/Q8_0 in "#3030" scope item 1 and owed by the
 * grouped kernel in its "Re-anchor" comment; the pages print no layout for it, so
 * it is Q4_K's header and nibbles plus one 32-byte plane of fifth bits), NVFP4 16-value blocks with an E4M3 scale and one fp32
 * tensor scale, FP8 E4M3 with one fp32 scale per row. IQ4_XS 136 B / 256 ("A 320B MoE
 * on a free Kaggle TPU", section "What '3-bit' costs, measured": the GGUF block
 * sizes of the codebook formats): a weight is an entry of the matrix's 16-value
 * codebook times its sub-block scale. IQ3_S 110 B / 256 and IQ2_S 82 B / 256 (same
 * section; "The kernel, and why 64 tok/s is not a bandwidth number": a group of
 * weights is one entry of the format's grid, 1,024 entries of 8 weights for IQ2_S,
 * groups of four for IQ3_S, with sign bits).
 *
 * Where the pages give no bit-level layout, the reading taken is the one written
 * in oracle.h (the plainest one consistent with the printed sizes).
 */
#include "oracle.h"
#include <math.h>
#include <string.h>
#include <stdlib.h>

/* ----------------------------------------------------------------------------
 * Rounding to a small binary floating-point format, round-to-nearest-even.
 * p = significand bits including the implicit one, emin = exponent of the
 * smallest normal binade. Works on a non-negative magnitude; the result is the
 * nearest representable magnitude (possibly one binade up after a carry).
 * Every fp32 input divided by a power of two is exact in double, and rint()
 * under the default rounding mode rounds ties to the even integer, i.e. to the
 * even significand.
 * -------------------------------------------------------------------------- */
static double rne_to_format(double a, int p, int emin) {
    if (a == 0.0) return 0.0;
    int ex;
    frexp(a, &ex);            /* a = f * 2^ex, f in [0.5, 1) */
    int e = ex - 1;           /* floor(log2 a) */
    if (e < emin) e = emin;   /* subnormal range keeps the quantum of emin */
    double q = ldexp(1.0, e - (p - 1));
    return rint(a / q) * q;
}

/* ---- IEEE binary16 ------------------------------------------------------- */
float or_fp16_to_f32(uint16_t h) {
    int s = h >> 15, e = (h >> 10) & 31, m = h & 1023;
    double v;
    if (e == 0) v = ldexp((double)m, -24);
    else if (e == 31) v = (m == 0) ? INFINITY : NAN;
    else v = ldexp(1.0 + m / 1024.0, e - 15);
    return (float)(s ? -v : v);
}

uint16_t or_f32_to_fp16(float f) {
    uint16_t s = signbit(f) ? 0x8000 : 0;
    if (isnan(f)) return 0x7E00;
    double a = fabs((double)f);
    if (isinf(f)) return s | 0x7C00;
    double r = rne_to_format(a, 11, -14);
    if (r > 65504.0) return s | 0x7C00;            /* overflow to infinity */
    if (r == 0.0) return s;
    if (r < ldexp(1.0, -14)) return s | (uint16_t)(r / ldexp(1.0, -24));
    int ex; frexp(r, &ex); int e = ex - 1;
    uint16_t m = (uint16_t)((r / ldexp(1.0, e) - 1.0) * 1024.0);
    return s | (uint16_t)((e + 15) << 10) | m;
}

/* ---- bfloat16: the top half of an fp32 ----------------------------------- */
/* round-to-nearest-even of a double to bfloat16 (8 significand bits, fp32's exponent
 * range); overflow to infinity */
uint16_t or_f64_to_bf16(double v) {
    if (v != v) return 0x7FC0;
    uint16_t sign = (v < 0 || (v == 0 && 1.0 / v < 0)) ? 0x8000 : 0;
    double a = fabs(v);
    double r = rne_to_format(a, 8, -126);
    if (r >= ldexp(1.0, 128)) return (uint16_t)(sign | 0x7F80);
    if (r == 0.0) return sign;
    float f = (float)r;                     /* exact: r has at most 8 significant bits */
    uint32_t u;
    memcpy(&u, &f, 4);
    return (uint16_t)(sign | ((u >> 16) & 0x7FFF));
}

float or_bf16_to_f32(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

/* ---- OCP FP8 E4M3: bias 7, 3 mantissa bits, S.1111.111 = NaN, max 448 ---- */
float or_e4m3_to_f32(uint8_t c) {
    int s = c >> 7, e = (c >> 3) & 15, m = c & 7;
    double v;
    if (e == 15 && m == 7) return NAN;
    if (e == 0) v = ldexp((double)m, -9);            /* 2^-6 * m/8 */
    else v = ldexp(1.0 + m / 8.0, e - 7);
    return (float)(s ? -v : v);
}

uint8_t or_f32_to_e4m3(float f) {                    /* RNE, saturate to +-448 */
    uint8_t s = signbit(f) ? 0x80 : 0;
    if (isnan(f)) return 0x7F;
    double r = rne_to_format(fabs((double)f), 4, -6);
    if (r > 448.0) r = 448.0;
    if (r == 0.0) return s;
    if (r < ldexp(1.0, -6)) return s | (uint8_t)(r / ldexp(1.0, -9));
    int ex; frexp(r, &ex); int e = ex - 1;
    uint8_t m = (uint8_t)((r / ldexp(1.0, e) - 1.0) * 8.0);
    return s | (uint8_t)((e + 7) << 3) | m;
}

/* ---- OCP FP4 E2M1: bias 1, 1 mantissa bit, max 6, no inf/NaN ------------- */
float or_e2m1_to_f32(uint8_t c) {
    int s = (c >> 3) & 1, e = (c >> 1) & 3, m = c & 1;
    double v = (e == 0) ? 0.5 * m : ldexp(1.0 + m / 2.0, e - 1);
    return (float)(s ? -v : v);
}

uint8_t or_f32_to_e2m1(float f) {                    /* RNE, saturate to +-6 */
    uint8_t s = signbit(f) ? 0x8 : 0;
    double r = rne_to_format(fabs((double)f), 2, 0);
    if (r > 6.0) r = 6.0;
    if (r == 0.0) return s;
    if (r < 1.0) return s | 1;                       /* the subnormal 0.5 */
    int ex; frexp(r, &ex); int e = ex - 1;
    uint8_t m = (uint8_t)((r / ldexp(1.0, e) - 1.0) * 2.0);
    return s | (uint8_t)((e + 1) << 1) | m;
}

/* ---- sizes ---------------------------------------------------------------- */
int64_t or_block_values(int fmt) {
    switch (fmt) {
    case OR_Q8_0: return 32;
    case OR_Q4_K: return 256;
    case OR_Q5_K: return 256;
    case OR_Q6_K: return 256;
    case OR_NVFP4: return 16;
    case OR_FP8_ROW: return 1;
    case OR_IQ4_XS: return 256;
    case OR_IQ3_S: return 256;
    case OR_IQ2_S: return 256;
    default: return 0;
    }
}

int64_t or_canon_bytes(int fmt, int64_t rows, int64_t K) {
    switch (fmt) {
    case OR_Q8_0: return rows * (K / 32) * 34;
    case OR_Q4_K: return rows * (K / 256) * 144;
    case OR_Q5_K: return rows * (K / 256) * 176;
    case OR_Q6_K: return rows * (K / 256) * 210;
    case OR_NVFP4: return rows * (K / 2) + rows * (K / 16) + 4;
    case OR_FP8_ROW: return rows * K + rows * 4;
    case OR_IQ4_XS: return rows * (K / 256) * 136 + 16;
    case OR_IQ3_S: return or_grid_bytes(fmt) + rows * (K / 256) * 110;
    case OR_IQ2_S: return or_grid_bytes(fmt) + rows * (K / 256) * 82;
    default: return -1;
    }
}

int64_t or_grid_bytes(int fmt) {
    return fmt == OR_IQ3_S ? 512 * 4 : (fmt == OR_IQ2_S ? 1024 * 8 : 0);
}

static uint16_t rd16(const uint8_t* p) { return (uint16_t)(p[0] | (p[1] << 8)); }
static void wr16(uint8_t* p, uint16_t v) { p[0] = (uint8_t)v; p[1] = (uint8_t)(v >> 8); }
static float rdf32(const uint8_t* p) { float f; memcpy(&f, p, 4); return f; }
static void wrf32(uint8_t* p, float f) { memcpy(p, &f, 4); }

static float clampf(float v, float lo, float hi) { return v < lo ? lo : (v > hi ? hi : v); }

/* 6-bit field f (0..15) of the 96-bit little-endian scale bitstream of Q4_K */
static int q4k_field(const uint8_t* sc12, int f) {
    int v = 0;
    for (int b = 0; b < 6; b++) {
        int bit = 6 * f + b;
        v |= ((sc12[bit >> 3] >> (bit & 7)) & 1) << b;
    }
    return v;
}
static void q4k_set_field(uint8_t* sc12, int f, int v) {
    for (int b = 0; b < 6; b++) {
        int bit = 6 * f + b;
        if ((v >> b) & 1) sc12[bit >> 3] |= (uint8_t)(1 << (bit & 7));
    }
}

/* ---------------------------------------------------------------------------
 * Encoders (synthetic-data generation). Non-iterative round-to-nearest
 * quantizers, fp32 arithmetic in the order written.
 * ------------------------------------------------------------------------- */
static void enc_q8_0_block(const float* x, uint8_t* blk) {
    float amax = 0.0f;
    for (int i = 0; i < 32; i++) { float a = fabsf(x[i]); if (a > amax) amax = a; }
    uint16_t d = or_f32_to_fp16(amax / 127.0f);
    float dd = or_fp16_to_f32(d);
    wr16(blk, d);
    for (int i = 0; i < 32; i++) {
        float q = (dd == 0.0f) ? 0.0f : clampf(nearbyintf(x[i] / dd), -127.0f, 127.0f);
        blk[2 + i] = (uint8_t)(int8_t)q;
    }
}

static void enc_q4_k_block(const float* x, uint8_t* blk) {
    float s[8], mn[8], smax = 0.0f, mmax = 0.0f;
    for (int j = 0; j < 8; j++) {
        float lo = 0.0f, hi = x[32 * j];
        for (int i = 0; i < 32; i++) {
            float v = x[32 * j + i];
            if (v < lo) lo = v;
            if (v > hi) hi = v;
        }
        s[j] = (hi - lo) / 15.0f;
        mn[j] = -lo;
        if (s[j] > smax) smax = s[j];
        if (mn[j] > mmax) mmax = mn[j];
    }
    uint16_t d = or_f32_to_fp16(smax / 63.0f), dmin = or_f32_to_fp16(mmax / 63.0f);
    float dd = or_fp16_to_f32(d), dm = or_fp16_to_f32(dmin);
    memset(blk, 0, 144);
    wr16(blk, d);
    wr16(blk + 2, dmin);
    for (int j = 0; j < 8; j++) {
        int sc = (dd == 0.0f) ? 0 : (int)clampf(nearbyintf(s[j] / dd), 0.0f, 63.0f);
        int mq = (dm == 0.0f) ? 0 : (int)clampf(nearbyintf(mn[j] / dm), 0.0f, 63.0f);
        q4k_set_field(blk + 4, j, sc);
        q4k_set_field(blk + 4, 8 + j, mq);
        float den = dd * (float)sc;
        float off = dm * (float)mq;
        for (int i = 0; i < 32; i++) {
            int e = 32 * j + i;
            float num = x[e] + off;
            int q = (den == 0.0f) ? 0 : (int)clampf(nearbyintf(num / den), 0.0f, 15.0f);
            blk[16 + e / 2] |= (uint8_t)(q << (4 * (e & 1)));
        }
    }
}

/* Q5_K: Q4_K's quantizer with 32 levels per sub-block instead of 16 */
static void enc_q5_k_block(const float* x, uint8_t* blk) {
    float s[8], mn[8], smax = 0.0f, mmax = 0.0f;
    for (int j = 0; j < 8; j++) {
        float lo = 0.0f, hi = x[32 * j];
        for (int i = 0; i < 32; i++) {
            float v = x[32 * j + i];
            if (v < lo) lo = v;
            if (v > hi) hi = v;
        }
        s[j] = (hi - lo) / 31.0f;
        mn[j] = -lo;
        if (s[j] > smax) smax = s[j];
        if (mn[j] > mmax) mmax = mn[j];
    }
    uint16_t d = or_f32_to_fp16(smax / 63.0f), dmin = or_f32_to_fp16(mmax / 63.0f);
    float dd = or_fp16_to_f32(d), dm = or_fp16_to_f32(dmin);
    memset(blk, 0, 176);
    wr16(blk, d);
    wr16(blk + 2, dmin);
    for (int j = 0; j < 8; j++) {
        int sc = (dd == 0.0f) ? 0 : (int)clampf(nearbyintf(s[j] / dd), 0.0f, 63.0f);
        int mq = (dm == 0.0f) ? 0 : (int)clampf(nearbyintf(mn[j] / dm), 0.0f, 63.0f);
        q4k_set_field(blk + 4, j, sc);
        q4k_set_field(blk + 4, 8 + j, mq);
        float den = dd * (float)sc;
        float off = dm * (float)mq;
        for (int i = 0; i < 32; i++) {
            int e = 32 * j + i;
            float num = x[e] + off;
            int q = (den == 0.0f) ? 0 : (int)clampf(nearbyintf(num / den), 0.0f, 31.0f);
            blk[16 + e / 8] |= (uint8_t)(((q >> 4) & 1) << (e & 7));
            blk[48 + e / 2] |= (uint8_t)((q & 15) << (4 * (e & 1)));
        }
    }
}

static void enc_q6_k_block(const float* x, uint8_t* blk) {
    float s[16], smax = 0.0f;
    for (int j = 0; j < 16; j++) {
        float amax = 0.0f;
        for (int i = 0; i < 16; i++) { float a = fabsf(x[16 * j + i]); if (a > amax) amax = a; }
        s[j] = amax / 32.0f;
        if (s[j] > smax) smax = s[j];
    }
    uint16_t d = or_f32_to_fp16(smax / 127.0f);
    float dd = or_fp16_to_f32(d);
    memset(blk, 0, 210);
    for (int j = 0; j < 16; j++) {
        int sc = (dd == 0.0f) ? 0 : (int)clampf(nearbyintf(s[j] / dd), -128.0f, 127.0f);
        blk[192 + j] = (uint8_t)(int8_t)sc;
        float den = dd * (float)sc;
        for (int i = 0; i < 16; i++) {
            int e = 16 * j + i;
            int q = (den == 0.0f) ? 0 : (int)clampf(nearbyintf(x[e] / den), -32.0f, 31.0f);
            int u = q + 32;                               /* 0..63 */
            blk[e / 2] |= (uint8_t)((u & 15) << (4 * (e & 1)));
            blk[128 + e / 4] |= (uint8_t)(((u >> 4) & 3) << (2 * (e & 3)));
        }
    }
    wr16(blk + 208, d);
}

/* IQ4_XS: sub-block j gets the signed scale s_j that maps its element of largest
 * magnitude onto the codebook entry of largest magnitude (the first such entry);
 * d = max_j |s_j| / 31 rounded to fp16; ls_j = clamp(rint(s_j / d) + 32, 0, 63); each
 * element takes the entry c nearest to it, |w - a_j C[c]| with a_j = d (ls_j - 32)
 * (fp32), ties to the lower index. */
static void enc_iq4_xs_block(const float* x, const int8_t* cb, uint8_t* blk) {
    int cm = 0;
    for (int c = 1; c < 16; c++)
        if (abs(cb[c]) > abs(cb[cm])) cm = c;
    float s[8], smax = 0.0f;
    for (int j = 0; j < 8; j++) {
        int em = 0;
        for (int i = 1; i < 32; i++)
            if (fabsf(x[32 * j + i]) > fabsf(x[32 * j + em])) em = i;
        s[j] = (cb[cm] != 0) ? x[32 * j + em] / (float)cb[cm] : 0.0f;
        if (fabsf(s[j]) > smax) smax = fabsf(s[j]);
    }
    memset(blk, 0, 136);
    uint16_t dh = or_f32_to_fp16(smax / 31.0f);
    float d = or_fp16_to_f32(dh);
    wr16(blk, dh);
    uint16_t sh = 0;
    for (int j = 0; j < 8; j++) {
        int ls = 32;
        if (d > 0.0f) ls = (int)clampf(rintf(s[j] / d) + 32.0f, 0.0f, 63.0f);
        sh |= (uint16_t)(((ls >> 4) & 3) << (2 * j));
        blk[4 + j / 2] |= (uint8_t)((ls & 15) << (4 * (j & 1)));
        float a = d * (float)(ls - 32);
        for (int i = 0; i < 32; i++) {
            int best = 0;
            float be = fabsf(x[32 * j + i] - a * (float)cb[0]);
            for (int c = 1; c < 16; c++) {
                float e = fabsf(x[32 * j + i] - a * (float)cb[c]);
                if (e < be) { be = e; best = c; }
            }
            int e = 32 * j + i;
            blk[8 + e / 2] |= (uint8_t)(best << (4 * (e & 1)));
        }
    }
    wr16(blk + 2, sh);
}

/* IQ3_S / IQ2_S: per sub-block (32 / 16 values) s = amax / gmax, gmax = the largest
 * magnitude in the grid; d = max s / 31 in fp16; sc = clamp(rint((s / d - 1) / 2), 0, 15),
 * a = d (2 sc + 1); per group (4 / 8 weights) the signs of its weights and the grid
 * entry nearest to their magnitudes: sum_i (|w_i| - a G[c][i])^2 in fp32, i in order,
 * ties to the lower index. */
static void enc_grid_block(int fmt, const float* x, const uint8_t* G, uint8_t* blk) {
    const int iq3 = (fmt == OR_IQ3_S);
    const int gw = iq3 ? 4 : 8, ne = iq3 ? 512 : 1024, sbs = iq3 ? 32 : 16, bb = iq3 ? 110 : 82;
    int gmax = 0;
    for (int i = 0; i < ne * gw; i++)
        if (G[i] > gmax) gmax = G[i];
    float s[16], smax = 0.0f;
    for (int k = 0; k < 256 / sbs; k++) {
        float amax = 0.0f;
        for (int i = 0; i < sbs; i++)
            if (fabsf(x[k * sbs + i]) > amax) amax = fabsf(x[k * sbs + i]);
        s[k] = (gmax > 0) ? amax / (float)gmax : 0.0f;
        if (s[k] > smax) smax = s[k];
    }
    memset(blk, 0, (size_t)bb);
    uint16_t dh = or_f32_to_fp16(smax / 31.0f);
    float d = or_fp16_to_f32(dh);
    wr16(blk, dh);
    for (int k = 0; k < 256 / sbs; k++) {
        int sc = 0;
        if (d > 0.0f) sc = (int)clampf(rintf((s[k] / d - 1.0f) / 2.0f), 0.0f, 15.0f);
        blk[(iq3 ? 106 : 74) + k / 2] |= (uint8_t)(sc << (4 * (k & 1)));
        float a = d * (float)(2 * sc + 1);
        for (int g = k * sbs / gw; g < (k + 1) * sbs / gw; g++) {
            const float* xg = x + g * gw;
            int best = 0;
            float be = 0.0f;
            for (int c = 0; c < ne; c++) {
                float e = 0.0f;
                for (int i = 0; i < gw; i++) {
                    float t = fabsf(xg[i]) - a * (float)G[c * gw + i];
                    e = e + t * t;
                }
                if (c == 0 || e < be) { be = e; best = c; }
            }
            blk[2 + g] = (uint8_t)(best & 255);
            if (iq3) blk[66 + g / 8] |= (uint8_t)(((best >> 8) & 1) << (g & 7));
            else blk[66 + g / 4] |= (uint8_t)(((best >> 8) & 3) << (2 * (g & 3)));
            for (int i = 0; i < gw; i++)
                if (xg[i] < 0.0f) {
                    if (iq3) blk[74 + (g * 4 + i) / 8] |= (uint8_t)(1 << ((g * 4 + i) & 7));
                    else blk[34 + g] |= (uint8_t)(1 << i);
                }
        }
    }
}

int or_encode_cb(int fmt, const float* W, int64_t rows, int64_t K, const void* codebook,
                 uint8_t* canon) {
    if (K % 256 != 0 || codebook == NULL) return 1;
    if (fmt == OR_IQ4_XS) {
        for (int64_t r = 0; r < rows; r++)
            for (int64_t b = 0; b < K / 256; b++)
                enc_iq4_xs_block(W + r * K + b * 256, (const int8_t*)codebook, canon + (r * (K / 256) + b) * 136);
        memcpy(canon + rows * (K / 256) * 136, codebook, 16);
        return 0;
    }
    if (fmt == OR_IQ3_S || fmt == OR_IQ2_S) {
        const int64_t gb = or_grid_bytes(fmt), bb = (fmt == OR_IQ3_S) ? 110 : 82;
        memcpy(canon, codebook, (size_t)gb);
        for (int64_t r = 0; r < rows; r++)
            for (int64_t b = 0; b < K / 256; b++)
                enc_grid_block(fmt, W + r * K + b * 256, (const uint8_t*)codebook,
                               canon + gb + (r * (K / 256) + b) * bb);
        return 0;
    }
    return 1;
}

int or_encode(int fmt, const float* W, int64_t rows, int64_t K, float tensor_scale,
              uint8_t* canon) {
    int64_t bv = or_block_values(fmt);
    if (bv == 0 || K % bv != 0) return 1;
    if (fmt == OR_Q8_0 || fmt == OR_Q4_K || fmt == OR_Q5_K || fmt == OR_Q6_K) {
        int64_t bb = (fmt == OR_Q8_0) ? 34 : (fmt == OR_Q4_K ? 144 : (fmt == OR_Q5_K ? 176 : 210));
        for (int64_t r = 0; r < rows; r++)
            for (int64_t b = 0; b < K / bv; b++) {
                const float* x = W + r * K + b * bv;
                uint8_t* blk = canon + (r * (K / bv) + b) * bb;
                if (fmt == OR_Q8_0) enc_q8_0_block(x, blk);
                else if (fmt == OR_Q4_K) enc_q4_k_block(x, blk);
                else if (fmt == OR_Q5_K) enc_q5_k_block(x, blk);
                else enc_q6_k_block(x, blk);
            }
        return 0;
    }
    if (fmt == OR_NVFP4) {
        uint8_t* codes = canon;
        uint8_t* scales = canon + rows * (K / 2);
        memset(codes, 0, (size_t)(rows * (K / 2)));
        float t = 6.0f * tensor_scale;
        for (int64_t r = 0; r < rows; r++)
            for (int64_t b = 0; b < K / 16; b++) {
                const float* x = W + r * K + b * 16;
                float amax = 0.0f;
                for (int i = 0; i < 16; i++) { float a = fabsf(x[i]); if (a > amax) amax = a; }
                uint8_t sb = (t > 0.0f) ? or_f32_to_e4m3(amax / t) : 0;
                scales[r * (K / 16) + b] = sb;
                float den = or_e4m3_to_f32(sb) * tensor_scale;
                for (int i = 0; i < 16; i++) {
                    uint8_t c = (den == 0.0f) ? 0 : or_f32_to_e2m1(x[i] / den);
                    int64_t e = b * 16 + i;
                    codes[r * (K / 2) + e / 2] |= (uint8_t)(c << (4 * (e & 1)));
                }
            }
        wrf32(canon + rows * (K / 2) + rows * (K / 16), tensor_scale);
        return 0;
    }
    if (fmt == OR_FP8_ROW) {
        uint8_t* codes = canon;
        uint8_t* rs = canon + rows * K;
        for (int64_t r = 0; r < rows; r++) {
            float amax = 0.0f;
            for (int64_t k = 0; k < K; k++) { float a = fabsf(W[r * K + k]); if (a > amax) amax = a; }
            float s = amax / 448.0f;
            wrf32(rs + 4 * r, s);
            for (int64_t k = 0; k < K; k++)
                codes[r * K + k] = (s == 0.0f) ? 0 : or_f32_to_e4m3(W[r * K + k] / s);
        }
        return 0;
    }
    return 1;
}

/* ---------------------------------------------------------------------------
 * BlockToFloat. fp32, the op order written here is the canonical one:
 *   Q8_0 : w = d * q                                   (exact)
 *   Q4_K : w = (d * sc_j) * q - (dmin * m_j)           (one rounding)
 *   Q5_K : the same expression, q = lo | hi << 4 in 0..31 (one rounding)
 *   Q6_K : w = (d * sc_j) * (q - 32)                   (exact)
 *   NVFP4: w = (e2m1(c) * e4m3(s_b)) * s_T             (one rounding)
 *   FP8  : w = e4m3(c) * s_row                         (one rounding)
 *   IQ4_XS: w = (d * (ls_j - 32)) * C[q]               (one rounding)
 *   IQ3_S, IQ2_S: w = (d * (2 sc + 1)) * (+-G[idx][i])  (exact)
 * ------------------------------------------------------------------------- */
static int nvfp4_to_float(const uint8_t* canon, int64_t rows, int64_t K, float* W) {
    const uint8_t* codes = canon;
    const uint8_t* scales = canon + rows * (K / 2);
    float sT = rdf32(canon + rows * (K / 2) + rows * (K / 16));
    for (int64_t r = 0; r < rows; r++)
        for (int64_t k = 0; k < K; k++) {
            uint8_t c = (codes[r * (K / 2) + k / 2] >> (4 * (k & 1))) & 15;
            float sb = or_e4m3_to_f32(scales[r * (K / 16) + k / 16]);
            float p = or_e2m1_to_f32(c) * sb;
            W[r * K + k] = p * sT;
        }
    return 0;
}

static int fp8_row_to_float(const uint8_t* canon, int64_t rows, int64_t K, float* W) {
    for (int64_t r = 0; r < rows; r++) {
        float s = rdf32(canon + rows * K + 4 * r);
        for (int64_t k = 0; k < K; k++) W[r * K + k] = or_e4m3_to_f32(canon[r * K + k]) * s;
    }
    return 0;
}

static int iq4_xs_to_float(const uint8_t* canon, int64_t rows, int64_t K, float* W) {
    const int8_t* cb = (const int8_t*)(canon + rows * (K / 256) * 136);
    for (int64_t r = 0; r < rows; r++)
        for (int64_t b = 0; b < K / 256; b++) {
            const uint8_t* blk = canon + (r * (K / 256) + b) * 136;
            float d = or_fp16_to_f32(rd16(blk));
            int sh = rd16(blk + 2);
            for (int e = 0; e < 256; e++) {
                int j = e / 32;
                int ls = ((blk[4 + j / 2] >> (4 * (j & 1))) & 15) | (((sh >> (2 * j)) & 3) << 4);
                int q = (blk[8 + e / 2] >> (4 * (e & 1))) & 15;
                float a = d * (float)(ls - 32);
                W[r * K + b * 256 + e] = a * (float)cb[q];
            }
        }
    return 0;
}

static int grid_to_float(int fmt, const uint8_t* canon, int64_t rows, int64_t K, float* W) {
    const int iq3 = (fmt == OR_IQ3_S);
    const int gw = iq3 ? 4 : 8, sbs = iq3 ? 32 : 16, bb = iq3 ? 110 : 82;
    const uint8_t* G = canon;
    const uint8_t* blocks = canon + or_grid_bytes(fmt);
    for (int64_t r = 0; r < rows; r++)
        for (int64_t b = 0; b < K / 256; b++) {
            const uint8_t* blk = blocks + (r * (K / 256) + b) * bb;
            float d = or_fp16_to_f32(rd16(blk));
            for (int e = 0; e < 256; e++) {
                int g = e / gw, i = e % gw, k = e / sbs;
                int idx, sg, sc;
                if (iq3) {
                    idx = blk[2 + g] | (((blk[66 + g / 8] >> (g & 7)) & 1) << 8);
                    sg = (blk[74 + e / 8] >> (e & 7)) & 1;
                    sc = (blk[106 + k / 2] >> (4 * (k & 1))) & 15;
                } else {
                    idx = blk[2 + g] | (((blk[66 + g / 4] >> (2 * (g & 3))) & 3) << 8);
                    sg = (blk[34 + g] >> i) & 1;
                    sc = (blk[74 + k / 2] >> (4 * (k & 1))) & 15;
                }
                float a = d * (float)(2 * sc + 1);
                float m = (float)G[idx * gw + i];
                W[r * K + b * 256 + e] = a * (sg ? -m : m);
            }
        }
    return 0;
}

/* For NVFP4, FP8_ROW and IQ4_XS `canon` is the whole matrix stream of `rows` rows
 * (codes, scales, then the tensor scale / row scales / codebook); for IQ3_S and
 * IQ2_S it is the grid, then the blocks of the rows. */
int or_block_to_float(int fmt, const uint8_t* canon, int64_t rows, int64_t K, float* W) {
    int64_t bv = or_block_values(fmt);
    if (bv == 0 || K % bv != 0) return 1;
    if (fmt == OR_NVFP4) return nvfp4_to_float(canon, rows, K, W);
    if (fmt == OR_FP8_ROW) return fp8_row_to_float(canon, rows, K, W);
    if (fmt == OR_IQ4_XS) return iq4_xs_to_float(canon, rows, K, W);
    if (fmt == OR_IQ3_S || fmt == OR_IQ2_S) return grid_to_float(fmt, canon, rows, K, W);
    for (int64_t r = 0; r < rows; r++) {
        float* w = W + r * K;
        if (fmt == OR_Q8_0) {
            for (int64_t b = 0; b < K / 32; b++) {
                const uint8_t* blk = canon + (r * (K / 32) + b) * 34;
                float d = or_fp16_to_f32(rd16(blk));
                for (int i = 0; i < 32; i++) w[b * 32 + i] = d * (float)(int8_t)blk[2 + i];
            }
        } else if (fmt == OR_Q4_K) {
            for (int64_t b = 0; b < K / 256; b++) {
                const uint8_t* blk = canon + (r * (K / 256) + b) * 144;
                float d = or_fp16_to_f32(rd16(blk)), dmin = or_fp16_to_f32(rd16(blk + 2));
                for (int e = 0; e < 256; e++) {
                    int j = e / 32;
                    int sc = q4k_field(blk + 4, j), m = q4k_field(blk + 4, 8 + j);
                    int q = (blk[16 + e / 2] >> (4 * (e & 1))) & 15;
                    float a = d * (float)sc;
                    float c = dmin * (float)m;
                    w[b * 256 + e] = a * (float)q - c;
                }
            }
        } else if (fmt == OR_Q5_K) {
            for (int64_t b = 0; b < K / 256; b++) {
                const uint8_t* blk = canon + (r * (K / 256) + b) * 176;
                float d = or_fp16_to_f32(rd16(blk)), dmin = or_fp16_to_f32(rd16(blk + 2));
                for (int e = 0; e < 256; e++) {
                    int j = e / 32;
                    int sc = q4k_field(blk + 4, j), m = q4k_field(blk + 4, 8 + j);
                    int lo = (blk[48 + e / 2] >> (4 * (e & 1))) & 15;
                    int hi = (blk[16 + e / 8] >> (e & 7)) & 1;
                    int q = lo | (hi << 4);
                    float a = d * (float)sc;
                    float c = dmin * (float)m;
                    w[b * 256 + e] = a * (float)q - c;
                }
            }
        } else { /* OR_Q6_K */
            for (int64_t b = 0; b < K / 256; b++) {
                const uint8_t* blk = canon + (r * (K / 256) + b) * 210;
                float d = or_fp16_to_f32(rd16(blk + 208));
                for (int e = 0; e < 256; e++) {
                    int lo = (blk[e / 2] >> (4 * (e & 1))) & 15;
                    int hi = (blk[128 + e / 4] >> (2 * (e & 3))) & 3;
                    int q = lo | (hi << 4);
                    int sc = (int8_t)blk[192 + e / 16];
                    float a = d * (float)sc;
                    w[b * 256 + e] = a * (float)(q - 32);
                }
            }
        }
    }
    return 0;
}

/* ---------------------------------------------------------------------------
 * y = x . W^T in fp64, plain k-order sums; den = sum |w x| (the error scale).
 * ------------------------------------------------------------------------- */
void or_gemv_f64(const float* W, int64_t N, int64_t K, const uint16_t* x_bf16, int64_t M,
                 double* y, double* den) {
    for (int64_t m = 0; m < M; m++)
        for (int64_t n = 0; n < N; n++) {
            double acc = 0.0, ab = 0.0;
            for (int64_t k = 0; k < K; k++) {
                double p = (double)W[n * K + k] * (double)or_bf16_to_f32(x_bf16[m * K + k]);
                acc += p;
                ab += fabs(p);
            }
            y[m * N + n] = acc;
            if (den) den[m * N + n] = ab;
        }
}

/* Distinct routed experts, ascending: each expert's rows are read once per step
 * ("A 320B MoE on a free Kaggle TPU", "The decode kernel's cost is not 'distinct
 * experts'": unique routed experts first, ascending). */
int64_t or_unique_experts(const int32_t* ids, int64_t n, int32_t* out) {
    int64_t u = 0;
    for (int64_t i = 0; i < n; i++) {
        int seen = 0;
        for (int64_t j = 0; j < u; j++) if (out[j] == ids[i]) { seen = 1; break; }
        if (!seen) out[u++] = ids[i];
    }
    for (int64_t i = 1; i < u; i++) {               /* insertion sort */
        int32_t v = out[i];
        int64_t j = i - 1;
        while (j >= 0 && out[j] > v) { out[j + 1] = out[j]; j--; }
        out[j + 1] = v;
    }
    return u;
}

/* NVFP4 activation quantizer for the W4A4 route: 16-value blocks, E4M3 block
 * scale s_b = e4m3(amax_b / (6 x_scale)); codes c = e2m1(x / (s_b x_scale)),
 * all zero when s_b is zero. x_scale is a given per-site constant. */
void or_quant_act_nvfp4(const uint16_t* x_bf16, int64_t M, int64_t K, float x_scale,
                        uint8_t* codes, uint8_t* scales) {
    memset(codes, 0, (size_t)(M * (K / 2)));
    float t = 6.0f * x_scale;
    for (int64_t m = 0; m < M; m++)
        for (int64_t b = 0; b < K / 16; b++) {
            float xv[16], amax = 0.0f;
            for (int i = 0; i < 16; i++) {
                xv[i] = or_bf16_to_f32(x_bf16[m * K + b * 16 + i]);
                float a = fabsf(xv[i]);
                if (a > amax) amax = a;
            }
            uint8_t sb = (t > 0.0f) ? or_f32_to_e4m3(amax / t) : 0;
            scales[m * (K / 16) + b] = sb;
            if (sb == 0) continue;
            float den = or_e4m3_to_f32(sb) * x_scale;
            for (int i = 0; i < 16; i++) {
                uint8_t c = or_f32_to_e2m1(xv[i] / den);
                int64_t e = b * 16 + i;
                codes[m * (K / 2) + e / 2] |= (uint8_t)(c << (4 * (e & 1)));
            }
        }
}

/* W4A4 prefill ("I Built a Custom Blackwell Kernel for Qwen3.8-27B", "What the
 * custom path actually does": W4A4 kernels after the activation is quantised to
 * NVFP4). The activation goes through the quantizer above with the given static
 * x_scale, each value is dequantized as e2m1(code) * e4m3(s_b) * x_scale, and
 * y[m][n] = sum_k a[m][k] * W[n][k] in fp64 over the BlockToFloat weights W (which
 * carry the tensor scale); den[m][n] = sum_k |a[m][k] * W[n][k]|. */
void or_w4a4_f64(const uint16_t* x_bf16, int64_t M, int64_t K, float x_scale, const float* W, int64_t N,
                 double* y, double* den) {
    uint8_t* codes = (uint8_t*)malloc((size_t)(M * (K / 2)));
    uint8_t* scales = (uint8_t*)malloc((size_t)(M * (K / 16)));
    double* a = (double*)malloc(sizeof(double) * (size_t)K);
    or_quant_act_nvfp4(x_bf16, M, K, x_scale, codes, scales);
    for (int64_t m = 0; m < M; m++) {
        for (int64_t k = 0; k < K; k++) {
            uint8_t c = (uint8_t)((codes[m * (K / 2) + k / 2] >> (4 * (k & 1))) & 15);
            a[k] = (double)or_e2m1_to_f32(c) * (double)or_e4m3_to_f32(scales[m * (K / 16) + k / 16]) *
                   (double)x_scale;
        }
        for (int64_t n = 0; n < N; n++) {
            double acc = 0.0, ab = 0.0;
            for (int64_t k = 0; k < K; k++) {
                double t = a[k] * (double)W[n * K + k];
                acc += t;
                ab += fabs(t);
            }
            y[m * N + n] = acc;
            if (den) den[m * N + n] = ab;
        }
    }
    free(codes);
    free(scales);
    free(a);
}

/* The int8-dot lever ("feat(BACKEND-TENSTORRENT-KEEPQUANT) ...", "Scope", its "Out of
 * scope" line and the decode-cost note that books the lever as the repayment): the
 * activation quantized to int8 per 32-value block, d = amax / 127 (fp32) and
 * q = clamp(rint(x / d), -127, 127) (all zero when d = 0), and the product taken
 * against those integers. */
void or_quant_act_q8(const uint16_t* x_bf16, int64_t M, int64_t K, int8_t* codes, float* scales) {
    for (int64_t m = 0; m < M; m++)
        for (int64_t b = 0; b < K / 32; b++) {
            float xv[32], amax = 0.0f;
            for (int i = 0; i < 32; i++) {
                xv[i] = or_bf16_to_f32(x_bf16[m * K + b * 32 + i]);
                if (fabsf(xv[i]) > amax) amax = fabsf(xv[i]);
            }
            float d = amax / 127.0f;
            scales[m * (K / 32) + b] = d;
            for (int i = 0; i < 32; i++)
                codes[m * K + b * 32 + i] = (int8_t)((d == 0.0f) ? 0 : (int)clampf(rintf(xv[i] / d), -127.0f, 127.0f));
        }
}

/* y = sum_k W[n][k] (d_b q_k) in fp64 with W = BlockToFloat of the weights [N][K] and
 * the activation's int8 codes and block scales from or_quant_act_q8; den = sum |terms| */
void or_int8dot_f64(const uint16_t* x_bf16, int64_t M, int64_t K, const float* W, int64_t N, double* y,
                    double* den) {
    int8_t* codes = (int8_t*)malloc((size_t)(M * K));
    float* scales = (float*)malloc(sizeof(float) * (size_t)(M * (K / 32)));
    double* a = (double*)malloc(sizeof(double) * (size_t)K);
    or_quant_act_q8(x_bf16, M, K, codes, scales);
    for (int64_t m = 0; m < M; m++) {
        for (int64_t k = 0; k < K; k++) a[k] = (double)scales[m * (K / 32) + k / 32] * (double)codes[m * K + k];
        for (int64_t n = 0; n < N; n++) {
            double acc = 0.0, ab = 0.0;
            for (int64_t k = 0; k < K; k++) {
                double term = a[k] * (double)W[n * K + k];
                acc += term;
                ab += fabs(term);
            }
            y[m * N + n] = acc;
            if (den) den[m * N + n] = ab;
        }
    }
    free(codes);
    free(scales);
    free(a);
}

/* SwiGLU of the gate/up projection read as one ("Qwen3.8-27B on one Tenstorrent
 * P150", "4. Measuring the ceiling, and lots of dead ends": the MLP gate/up
 * projection and its fused SwiGLU; "A 320B MoE on a free Kaggle TPU": the gate
 * matrix inside a SwiGLU): h = silu(g) * u with silu(g) = g / (1 + exp(-g)), in
 * fp64, elementwise over n values. */
void or_swiglu_f64(const double* g, const double* u, int64_t n, double* h) {
    for (int64_t i = 0; i < n; i++) h[i] = (g[i] / (1.0 + exp(-g[i]))) * u[i];
}
