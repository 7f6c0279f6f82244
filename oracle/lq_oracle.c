/*
 * Plain CPU oracle for the low-bit linear layer: dequantization and reference
 * matrix products.  TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the
 * benchmark's CPU-baseline leg load this; the product path never does.
 *
 * Everything here is written for a reader checking it against the definitions,
 * not for speed: one loop per definition, no blocking, no vector intrinsics.
 * Compiled with -ffp-contract=off so that the only fused multiply-add is the
 * explicit fmaf() of the 2-bit dequantization.
 *
 * Definitions followed (the otf-llm 4.0.1 README, "Theoretical & Mathematical
 * Foundations"):
 *   - section 2 "The Lloyd-Max Non-Uniform Solution": codebook
 *     C = {-1.52, -0.45, +0.45, +1.52}; a code q in 0..3 indexes C in listed order;
 *   - section 3 "Closed-Form Group Linear Regression": a weight of group g is
 *     reconstructed as S_g * C[q] + Z_g;
 *   - section 4 "Profile-Guided Activation Outliers": anchor columns are kept
 *     exactly in FP16 and replace the 2-bit reconstruction there.
 * NF4 (AirQuant README, "Fundamentacao Teorica", item 2; QLoRA data type):
 *   w = T[q] * absmax of the 64-weight block.
 * INT4 (the same otf-llm README's v3.2 engine): w = S * q on a uniform symmetric grid,
 *   columns in a static permutation (oracle_dequant_int4 below).
 *
 * Rounding (fixed here because the pages leave it open): the 2-bit value is one
 * fp32 fused multiply-add fmaf(S, C[q], Z) of the binary16 scale and offset; the
 * NF4 value is one fp32 product.  fp16/bf16 outputs take one round-to-nearest-even
 * conversion of that fp32 value.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define ORACLE_API __attribute__((visibility("default")))

/* The page's four centroids, in listed (ascending) order, as fp32. */
static const float CODEBOOK[4] = {-1.52f, -0.45f, 0.45f, 1.52f};

/* IEEE binary16 bit pattern -> exact float (all finite values, incl. subnormals). */
static float half_to_float(uint16_t h) {
    int sign = (h >> 15) & 1;
    int exp = (h >> 10) & 0x1f;
    int man = h & 0x3ff;
    double v;
    if (exp == 0) {
        v = ldexp((double)man, -24);              /* subnormal: man * 2^-24 */
    } else if (exp == 31) {
        v = man ? NAN : INFINITY;
    } else {
        v = ldexp((double)(man + 1024), exp - 25); /* (1 + man/1024) * 2^(exp-15) */
    }
    return (float)(sign ? -v : v);                 /* exact: at most 11 significant bits */
}

/* bfloat16 bit pattern -> exact float (the top 16 bits of an fp32). */
static float bf16_to_float(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* float -> bfloat16 bits, round to nearest, ties to even. */
static uint16_t float_to_bf16_rne(float f) {
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7fffffffu) > 0x7f800000u) return (uint16_t)((u >> 16) | 0x40); /* quiet NaN */
    uint32_t lsb = (u >> 16) & 1u;
    u += 0x7fffu + lsb;
    return (uint16_t)(u >> 16);
}

/* float -> binary16 bits, round to nearest, ties to even (subnormals and overflow included). */
static uint16_t float_to_half_rne(float f) {
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    uint16_t sign = (uint16_t)((u >> 16) & 0x8000u);
    uint32_t a = u & 0x7fffffffu;
    if (a > 0x7f800000u) return sign | 0x7e00u;                 /* NaN */
    if (a >= 0x477ff000u) return sign | 0x7c00u;                /* >= 65520 rounds to inf */
    if (a < 0x33000000u) return sign;                           /* < 2^-25 rounds to 0 (tie at 2^-25 -> 0, even) */
    int e = (int)(a >> 23) - 127;                               /* unbiased exponent */
    uint32_t m = (a & 0x7fffffu) | 0x800000u;                   /* 24-bit significand */
    int shift;                                                  /* bits to drop */
    uint32_t base;
    if (e < -14) {                                              /* binary16 subnormal: value = k * 2^-24 */
        shift = 13 + (-14 - e);
        base = 0;
    } else {
        shift = 13;
        base = (uint32_t)(e + 15) << 10;
        m &= 0x7fffffu;                                         /* drop the implicit bit; carry fixes exponent */
    }
    uint32_t q = m >> shift;
    uint32_t rem = m & ((1u << shift) - 1u);
    uint32_t half = 1u << (shift - 1);
    if (rem > half || (rem == half && (q & 1u))) q += 1u;
    return (uint16_t)(sign | (uint16_t)(base + q));             /* mantissa overflow carries into exponent */
}

ORACLE_API float oracle_half_to_float(uint16_t h) { return half_to_float(h); }
ORACLE_API float oracle_bf16_to_float(uint16_t b) { return bf16_to_float(b); }
ORACLE_API uint16_t oracle_float_to_half(float f) { return float_to_half_rne(f); }
ORACLE_API uint16_t oracle_float_to_bf16(float f) { return float_to_bf16_rne(f); }

/* One 2-bit weight: fmaf(S, C[q], Z) in fp32, one rounding. */
ORACLE_API float oracle_dequant_2bit_one(uint16_t s_bits, int q, uint16_t z_bits) {
    return fmaf(half_to_float(s_bits), CODEBOOK[q & 3], half_to_float(z_bits));
}

/*
 * Dequantize one 2-bit matrix to fp32 [N][K].
 *   codes     [N][K/4]   byte j of a row holds columns 4j..4j+3, column 4j+i in bits 2i..2i+1
 *   scales    [N][K/32]  binary16 S_g
 *   offsets   [N][K/32]  binary16 Z_g
 *   anchor_idx[A]        sorted input columns kept in FP16
 *   anchor_w  [N][lda]   binary16 value of W[n][anchor_idx[a]] at column a
 */
ORACLE_API void oracle_dequant_2bit(const uint8_t* codes, const uint16_t* scales, const uint16_t* offsets,
                                    const int32_t* anchor_idx, const uint16_t* anchor_w, int A, int lda,
                                    int N, int K, float* out) {
    for (int n = 0; n < N; ++n) {
        for (int k = 0; k < K; ++k) {
            int byte = codes[(size_t)n * (K / 4) + k / 4];
            int q = (byte >> (2 * (k % 4))) & 3;
            size_t g = (size_t)n * (K / 32) + k / 32;
            out[(size_t)n * K + k] = fmaf(half_to_float(scales[g]), CODEBOOK[q], half_to_float(offsets[g]));
        }
        for (int a = 0; a < A; ++a) {
            out[(size_t)n * K + anchor_idx[a]] = half_to_float(anchor_w[(size_t)n * lda + a]);
        }
    }
}

/*
 * Dequantize one NF4 matrix to fp32 [N][K].
 *   codes  [N][K/2]   byte j of a row: column 2j in the low nibble, 2j+1 in the high nibble
 *   absmax [N][K/64]  fp32 block maxima
 *   table  [16]       the NF4 levels as fp32
 */
ORACLE_API void oracle_dequant_nf4(const uint8_t* codes, const float* absmax, const float* table,
                                   int N, int K, float* out) {
    for (int n = 0; n < N; ++n) {
        for (int k = 0; k < K; ++k) {
            int byte = codes[(size_t)n * (K / 2) + k / 2];
            int q = (k % 2 == 0) ? (byte & 15) : (byte >> 4);
            out[(size_t)n * K + k] = table[q] * absmax[(size_t)n * (K / 64) + k / 64];
        }
    }
}

/*
 * The otf-llm README's v3.2 INT4 format ("Comparative Analysis: INT4 (v3.2) vs INT2
 * Non-Uniform (v4.0)"): 2 weights per byte on a uniform grid with zero-point 0, input
 * columns stored in a global static permutation, the top-1% columns kept in FP16.
 * Dequantize one matrix to fp32 [N][K] in ORIGINAL column order:
 *   codes     [N][K/2]   byte j holds permuted positions 2j (low nibble) and 2j+1 (high),
 *                        each a 4-bit two's complement integer q
 *   scales    [N][K/32]  binary16 S of the 32 consecutive permuted positions of a group
 *   perm      [K]        perm[j] = the input column stored at permuted position j
 *   anchor_idx[A], anchor_w [N][lda]   as for the 2-bit format (replace the grid value)
 * w = S * q is one fp32 product (exact: 11 by 4 significant bits).
 */
ORACLE_API void oracle_dequant_int4(const uint8_t* codes, const uint16_t* scales, const int32_t* perm,
                                    const int32_t* anchor_idx, const uint16_t* anchor_w, int A, int lda,
                                    int N, int K, float* out) {
    for (int n = 0; n < N; ++n) {
        for (int j = 0; j < K; ++j) {
            int byte = codes[(size_t)n * (K / 2) + j / 2];
            int nib = (j % 2 == 0) ? (byte & 15) : (byte >> 4);
            int q = nib >= 8 ? nib - 16 : nib;
            out[(size_t)n * K + perm[j]] = half_to_float(scales[(size_t)n * (K / 32) + j / 32]) * (float)q;
        }
        for (int a = 0; a < A; ++a)
            out[(size_t)n * K + anchor_idx[a]] = half_to_float(anchor_w[(size_t)n * lda + a]);
    }
}

/*
 * NF4 with double quantization (QLoRA, the method the AirQuant README cites for NF4, item 2
 * and the reference list): the fp32 block maxima are themselves stored as 8-bit floats.
 * 8-bit float = E4M3: sign, 4 exponent bits (bias 7), 3 mantissa bits; exponent 0 holds
 * the subnormals m/8 * 2^-6; 0x7F and 0xFF are NaN; no infinities; largest finite 448.
 */
ORACLE_API double oracle_e4m3_to_double(uint8_t c) {
    int sign = (c >> 7) & 1, e = (c >> 3) & 15, m = c & 7;
    double v;
    if (e == 15 && m == 7) return NAN;
    if (e == 0)
        v = ldexp((double)m, -9);               /* m/8 * 2^-6 */
    else
        v = ldexp((double)(8 + m), e - 10);     /* (1 + m/8) * 2^(e-7) */
    return sign ? -v : v;
}

/* Nearest E4M3 value to v (ties to the even mantissa), saturating at +-448; v finite. */
ORACLE_API uint8_t oracle_double_to_e4m3(double v) {
    uint8_t sign = v < 0 ? 0x80 : 0;
    double a = fabs(v);
    if (a >= 448.0) return sign | 0x7E;
    /* candidates: every finite magnitude code 0x00..0x7E; pick the nearest, ties to even m */
    int best = 0;
    double bd = a;                               /* distance to code 0 (value 0) */
    for (int c = 1; c <= 0x7E; ++c) {
        double d = fabs(oracle_e4m3_to_double((uint8_t)c) - a);
        if (d < bd || (d == bd && (c & 1) == 0 && (best & 1) == 1)) {
            bd = d;
            best = c;
        }
    }
    return (uint8_t)(sign | best);
}

/*
 * The double-quantized block maximum of first-level block i (row-major index into the
 * [N][K/64] array): c'_i = fmaf(e4m3(acodes[i]), s2[i / 256], mean), one fp32 rounding.
 *   second [1 + ceil(N*K/64 / 256)]: second[0] = mean, second[1 + j] = s2 of 256-block j.
 * The weights: w = T[q] * c' (one fp32 rounding), as for plain NF4.
 */
ORACLE_API float oracle_nf4_dq_absmax(const uint8_t* acodes, const float* second, size_t i) {
    return fmaf((float)oracle_e4m3_to_double(acodes[i]), second[1 + i / 256], second[0]);
}

ORACLE_API void oracle_dequant_nf4_dq(const uint8_t* codes, const uint8_t* acodes, const float* second,
                                      const float* table, int N, int K, float* out) {
    for (int n = 0; n < N; ++n) {
        for (int k = 0; k < K; ++k) {
            int byte = codes[(size_t)n * (K / 2) + k / 2];
            int q = (k % 2 == 0) ? (byte & 15) : (byte >> 4);
            float am = oracle_nf4_dq_absmax(acodes, second, (size_t)n * (K / 64) + k / 64);
            out[(size_t)n * K + k] = table[q] * am;
        }
    }
}

/* fp32 values -> binary16 or bfloat16 bit patterns (kind 1 = f16, 2 = bf16), RNE. */
ORACLE_API void oracle_round_f32(const float* in, size_t count, int kind, uint16_t* out) {
    for (size_t i = 0; i < count; ++i)
        out[i] = (kind == 1) ? float_to_half_rne(in[i]) : float_to_bf16_rne(in[i]);
}

/* x bits (kind 1 = f16, 2 = bf16) -> float. */
static float x_value(uint16_t bits, int kind) { return kind == 1 ? half_to_float(bits) : bf16_to_float(bits); }

/*
 * Reference product y[m][n] = sum_k W[n][k] * x[m][k] in fp64, and the error scale
 * E[m][n] = sum_k |W[n][k]| * |x[m][k]|, for W given as fp32 [N][K] and x as
 * 16-bit bits [M][K].
 */
ORACLE_API void oracle_matmul_f64(const float* W, const uint16_t* x, int x_kind, int M, int N, int K,
                                  double* y, double* E) {
    for (int m = 0; m < M; ++m) {
        for (int n = 0; n < N; ++n) {
            double acc = 0.0, mag = 0.0;
            for (int k = 0; k < K; ++k) {
                double w = (double)W[(size_t)n * K + k];
                double v = (double)x_value(x[(size_t)m * K + k], x_kind);
                acc += w * v;
                mag += fabs(w) * fabs(v);
            }
            y[(size_t)m * N + n] = acc;
            E[(size_t)m * N + n] = mag;
        }
    }
}

/*
 * The whole 2-bit layer product as the oracle states it, row by row: dequantize
 * row n (fmaf, anchors substituted) into a scratch row, then the fp64 dot product
 * with every token.  Used for the timed CPU baseline and for sampled checks of
 * large problems (rows [n0, n1) only).
 */
ORACLE_API void oracle_gemv_2bit_rows(const uint8_t* codes, const uint16_t* scales, const uint16_t* offsets,
                                      const int32_t* anchor_idx, const uint16_t* anchor_w, int A, int lda,
                                      const uint16_t* x, int x_kind, int M, int N, int K, int n0, int n1,
                                      float* row_scratch, double* y /* [M][n1-n0] */) {
    for (int n = n0; n < n1; ++n) {
        oracle_dequant_2bit(codes + (size_t)n * (K / 4), scales + (size_t)n * (K / 32),
                            offsets + (size_t)n * (K / 32), anchor_idx, anchor_w + (size_t)n * lda, A, lda,
                            1, K, row_scratch);
        for (int m = 0; m < M; ++m) {
            double acc = 0.0;
            for (int k = 0; k < K; ++k)
                acc += (double)row_scratch[k] * (double)x_value(x[(size_t)m * K + k], x_kind);
            y[(size_t)m * (n1 - n0) + (n - n0)] = acc;
        }
    }
}

/* Same for NF4. */
ORACLE_API void oracle_gemv_nf4_rows(const uint8_t* codes, const float* absmax, const float* table,
                                     const uint16_t* x, int x_kind, int M, int N, int K, int n0, int n1,
                                     float* row_scratch, double* y) {
    for (int n = n0; n < n1; ++n) {
        oracle_dequant_nf4(codes + (size_t)n * (K / 2), absmax + (size_t)n * (K / 64), table, 1, K, row_scratch);
        for (int m = 0; m < M; ++m) {
            double acc = 0.0;
            for (int k = 0; k < K; ++k)
                acc += (double)row_scratch[k] * (double)x_value(x[(size_t)m * K + k], x_kind);
            y[(size_t)m * (n1 - n0) + (n - n0)] = acc;
        }
    }
}
