// Register-level dequantization building blocks for the decode kernels.
//
// 2-bit (otf-llm 4.0.1 README, sections 2-3): the four binary16 values
// fmaf(S, C[q], Z) of one 32-column group sit in two byte-split registers
// (RA = low bytes, RB = high bytes).  A PRMT whose selector nibbles are
// (q, q+4) for two codes yields two binary16 weights at once.
// NF4 (AirQuant README, NF4): the sixteen binary16 levels sit in eight
// byte-split registers; PRMT looks up the low three index bits in both halves
// of the table and a byte mask from the fourth bit picks the half.
#pragma once

#include "lq_common.cuh"

namespace lq {

__device__ __forceinline__ uint32_t mulhi_add(uint32_t a, uint32_t b, uint32_t c) {
    uint32_t d;
    asm("mad.hi.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

// Byte-split table of binary16 fmaf(s, C[q], z) for q = 0..3.
__device__ __forceinline__ void lut2_bits(uint16_t s_bits, uint16_t z_bits, uint32_t& RA, uint32_t& RB) {
    const float s = half_bits_to_float(s_bits), z = half_bits_to_float(z_bits);
    const uint32_t p01 = pack_half2_rn(__fmaf_rn(s, -1.52f, z), __fmaf_rn(s, -0.45f, z));
    const uint32_t p23 = pack_half2_rn(__fmaf_rn(s, 0.45f, z), __fmaf_rn(s, 1.52f, z));
    RA = prmt(p01, p23, 0x6420);
    RB = prmt(p01, p23, 0x7531);
}

// Codes at bit offset 2j of the four bytes of w -> binary16 pairs (byte0, byte1) in `lo`
// and (byte2, byte3) in `hi`.  Both selectors come from one masked word through the
// multiplier (IMAD / IMAD.HI), which keeps the integer pipe to three operations.
__device__ __forceinline__ void expand2_fast(uint32_t w, int j, uint32_t RA, uint32_t RB, uint32_t& lo, uint32_t& hi) {
    const uint32_t t = (j == 0 ? w : (w >> (2 * j))) & 0x03030303u;
    const uint32_t sel_lo = t * 0x11u + 0x40404040u;          // nibbles (q, q+4) for bytes 0 and 1
    const uint32_t sel_hi = mulhi_add(t, 0x00110000u, 0x4040u);  // the same for bytes 2 and 3
    lo = prmt(RA, RB, sel_lo);
    hi = prmt(RA, RB, sel_hi);
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
    const uint32_t sel = c == 0 ? (w & 0x7777u) : mulhi_add(w & 0x77770000u, 0x10000u, 0u);
    const uint32_t mask = prmt(w << 4, w, c == 0 ? 0xD9C8u : 0xFBEAu);  // 0xFF where index bit 3 is set
    const uint32_t lo = (prmt(TL[0], TL[1], sel) & ~mask) | (prmt(TL[2], TL[3], sel) & mask);
    const uint32_t hi = (prmt(TH[0], TH[1], sel) & ~mask) | (prmt(TH[2], TH[3], sel) & mask);
    r01 = prmt(lo, hi, 0x5140);
    r23 = prmt(lo, hi, 0x7362);
}

}  // namespace lq
