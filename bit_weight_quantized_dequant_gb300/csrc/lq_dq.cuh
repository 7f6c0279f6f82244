// Register-level dequantization building blocks for the decode kernels.
//
// 2-bit (otf-llm 4.0.1 README, sections 2-3): the four binary16 values
// fmaf(S, C[q], Z) of one 32-column group sit in two half2 registers.  A PRMT
// whose selector nibbles are (2q, 2q+1) for two codes yields two binary16
// weights at once.
// NF4 (AirQuant README, NF4): the sixteen binary16 levels sit in eight
// byte-split registers; PRMT looks up the low three index bits in both halves
// of the table and a byte mask from the fourth bit picks the half.
#pragma once

#include "lq_common.cuh"

namespace lq {

// Table of binary16 fmaf(s, C[q], z) for q = 0..3 as two half2 registers:
// P01 = (L0, L1), P23 = (L2, L3).  Byte 2q of the pair {P01, P23} is the low byte of L[q].
__device__ __forceinline__ void lut2_bits(uint16_t s_bits, uint16_t z_bits, uint32_t& P01, uint32_t& P23) {
    const float s = half_bits_to_float(s_bits), z = half_bits_to_float(z_bits);
    P01 = pack_half2_rn(__fmaf_rn(s, -1.52f, z), __fmaf_rn(s, -0.45f, z));
    P23 = pack_half2_rn(__fmaf_rn(s, 0.45f, z), __fmaf_rn(s, 1.52f, z));
}

// The same table, also raising `peak` to the group's largest |fmaf(S, C[q], Z)|, which is
// fmaf(1.52, |S|, |Z|) exactly; a peak >= kHalfOverflow means a table value overflowed.
__device__ __forceinline__ void lut2_bits_peak(uint16_t s_bits, uint16_t z_bits, uint32_t& P01, uint32_t& P23,
                                               float& peak) {
    const float s = half_bits_to_float(s_bits), z = half_bits_to_float(z_bits);
    P01 = pack_half2_rn(__fmaf_rn(s, -1.52f, z), __fmaf_rn(s, -0.45f, z));
    P23 = pack_half2_rn(__fmaf_rn(s, 0.45f, z), __fmaf_rn(s, 1.52f, z));
    peak = fmaxf(peak, __fmaf_rn(1.52f, fabsf(s), fabsf(z)));
}

// The tables of two groups at once (packed fp32 fma: one instruction per table entry for
// both; each entry still one fmaf rounding, then one RNE to binary16), raising `peak` to the
// largest |fmaf(S, C[q], Z)| of both, which is max(|L0|, |L3|) (C is symmetric, so one of the
// two is fmaf(1.52, |S|, |Z|) exactly).
__device__ __forceinline__ float2 fma_f32x2(float2 a, float c, float2 b) {
    float2 d;
    asm("{\n\t.reg .b64 a, c, b, d;\n\tmov.b64 a, {%2, %3};\n\tmov.b64 c, {%4, %4};\n\tmov.b64 b, {%5, %6};\n\t"
        "fma.rn.f32x2 d, a, c, b;\n\tmov.b64 {%0, %1}, d;\n\t}"
        : "=f"(d.x), "=f"(d.y) : "f"(a.x), "f"(a.y), "f"(c), "f"(b.x), "f"(b.y));
    return d;
}

__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

__device__ __forceinline__ void lut2_bits_x2(float2 S, float2 Z, uint32_t& A0, uint32_t& B0, uint32_t& A1,
                                             uint32_t& B1, float& peak) {
    const float2 L0 = fma_f32x2(S, -1.52f, Z), L1 = fma_f32x2(S, -0.45f, Z);
    const float2 L2 = fma_f32x2(S, 0.45f, Z), L3 = fma_f32x2(S, 1.52f, Z);
    A0 = pack_half2_rn(L0.x, L1.x);
    B0 = pack_half2_rn(L2.x, L3.x);
    A1 = pack_half2_rn(L0.y, L1.y);
    B1 = pack_half2_rn(L2.y, L3.y);
    peak = fmax3(peak, fabsf(L0.x), fabsf(L3.x));
    peak = fmax3(peak, fabsf(L0.y), fabsf(L3.y));
}

// Codes at bit offset 2j of the four bytes of w -> binary16 pairs (byte0, byte1) in `lo`
// and (byte2, byte3) in `hi`.  One multiply turns each 2-bit code q into the selector
// nibbles (2q, 2q+1) of its byte lane; the upper half of that word serves bytes 2 and 3.
__device__ __forceinline__ void expand2_fast(uint32_t w, int j, uint32_t P01, uint32_t P23, uint32_t& lo, uint32_t& hi) {
    const uint32_t t = (j == 0 ? w : (w >> (2 * j))) & 0x03030303u;
    const uint32_t sel = t * 0x22u + 0x10101010u;
    lo = prmt(P01, P23, sel);
    hi = prmt(P01, P23, sel >> 16);
}

// NF4 table in byte-split registers: TL[i] = low bytes of levels 4i..4i+3, TH[i] = high bytes.
__device__ __forceinline__ void nf4_tables(uint32_t (&TL)[4], uint32_t (&TH)[4]) {
#pragma unroll
    for (int q4 = 0; q4 < 4; ++q4) {
        const uint32_t p01 = pack_half2_rn(kNF4[4 * q4 + 0], kNF4[4 * q4 + 1]);
        const uint32_t p23 = pack_half2_rn(kNF4[4 * q4 + 2], kNF4[4 * q4 + 3]);
        TL[q4] = prmt(p01, p23, 0x6420);
        TH[q4] = prmt(p01, p23, 0x7531);
    }
}

// Four NF4 codes (16-bit chunk c of w) -> half2(T[c0],T[c1]) and half2(T[c2],T[c3]).
__device__ __forceinline__ void expand_nf4_fast(uint32_t w, int c, const uint32_t (&TL)[4], const uint32_t (&TH)[4],
                                                uint32_t& r01, uint32_t& r23) {
    const uint32_t sel = c == 0 ? (w & 0x7777u) : ((w >> 16) & 0x7777u);
    const uint32_t mask = prmt(w << 4, w, c == 0 ? 0xD9C8u : 0xFBEAu);  // 0xFF where index bit 3 is set
    const uint32_t lo = (prmt(TL[0], TL[1], sel) & ~mask) | (prmt(TL[2], TL[3], sel) & mask);
    const uint32_t hi = (prmt(TH[0], TH[1], sel) & ~mask) | (prmt(TH[2], TH[3], sel) & mask);
    r01 = prmt(lo, hi, 0x5140);
    r23 = prmt(lo, hi, 0x7362);
}

}  // namespace lq
