// Device helpers shared by the liblq kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/lq.h"

namespace lq {

// The otf-llm README's Lloyd-Max codebook (section 2), listed order, as fp32.
__device__ __forceinline__ float codebook(int q) {
    return q == 0 ? -1.52f : (q == 1 ? -0.45f : (q == 2 ? 0.45f : 1.52f));
}

// The 16 NF4 levels of the QLoRA NormalFloat data type (the AirQuant README's
// NF4 reference), ascending, exactly the published float32 values.
__device__ __constant__ static const float kNF4[16] = {
    -1.0f, -0.6961928009986877f, -0.5250730514526367f, -0.39491748809814453f,
    -0.28444138169288635f, -0.18477343022823334f, -0.09105003625154495f, 0.0f,
    0.07958029955625534f, 0.16093020141124725f, 0.24611230194568634f, 0.33791524171829224f,
    0.44070982933044434f, 0.5626170039176941f, 0.7229568362236023f, 1.0f};

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}

// Two fp32 -> packed binary16x2 (lo = a, hi = b), round to nearest even.
__device__ __forceinline__ uint32_t pack_half2_rn(float lo, float hi) {
    uint32_t d;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
    return d;
}

__device__ __forceinline__ float half_bits_to_float(uint16_t h) {
    return __half2float(__ushort_as_half(h));
}

__device__ __forceinline__ float bf16_bits_to_float(uint16_t b) {
    return __uint_as_float(((uint32_t)b) << 16);
}

// Read-only 128/64/32-bit global loads through the non-coherent path.
__device__ __forceinline__ uint4 ldg128(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
    return v;
}
__device__ __forceinline__ uint2 ldg64(const void* p) {
    uint2 v;
    asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p));
    return v;
}
__device__ __forceinline__ uint32_t ldg32(const void* p) {
    uint32_t v;
    asm volatile("ld.global.nc.u32 %0, [%1];" : "=r"(v) : "l"(p));
    return v;
}

// D += A * B, m16n8k16, binary16 inputs, fp32 accumulators.
__device__ __forceinline__ void mma_f16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                              uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// ---- x in the decode kernels' binary16 operand range ---------------------------------
//
// bf16 x reaches the decode tensor cores as binary16.  Each token's x is first scaled by
// the power of two 2^e that brings its largest |x| into [2^14, 2^15) (e clamped to
// [-125, 125]; e = 0 when x is all zero); the fp32 result is multiplied by 2^-e.  Both
// factors are exact, so the only rounding is the one to binary16, relative 2^-11 for every
// value within 2^28 of the token's largest.  maxbits is the fp32 bit pattern of max |x|.
__device__ __forceinline__ int x_scale_exp(uint32_t maxbits) {
    if (maxbits == 0u) return 0;
    const int e = 14 - ((int)(maxbits >> 23) - 127);
    return e < -125 ? -125 : (e > 125 ? 125 : e);
}
__device__ __forceinline__ float x_scale(uint32_t maxbits) { return __int_as_float((x_scale_exp(maxbits) + 127) << 23); }
__device__ __forceinline__ float x_unscale(uint32_t maxbits) { return __int_as_float((127 - x_scale_exp(maxbits)) << 23); }

// bf16 bits -> binary16 bits of (value * scale), round to nearest even.
__device__ __forceinline__ uint16_t bf16_to_half_scaled(uint16_t raw, float scale) {
    return __half_as_ushort(__float2half_rn(__uint_as_float(((uint32_t)raw) << 16) * scale));
}

// Largest value the weight lookup tables may hold: binary16 rounds |v| >= 65520 to infinity.
constexpr float kHalfOverflow = 65520.0f;

// An 8-bit float (E4M3: sign, 4 exponent bits with bias 7, 3 mantissa bits; exponent 0
// holds the subnormals m/8 * 2^-6; 0x7F / 0xFF are NaN) as fp32, exactly.
__device__ __forceinline__ float e4m3_to_float(uint32_t c) {
    const uint32_t e = (c >> 3) & 15u, m = c & 7u;
    float v = e ? __uint_as_float(((e + 120u) << 23) | (m << 20)) : (float)m * 0.001953125f;   // (2^-9)
    if (e == 15u && m == 7u) v = __uint_as_float(0x7fc00000u);
    return (c & 0x80u) ? -v : v;
}

// NF4 with double quantization: the block maximum of first-level block i (row-major in
// [N][K/64]) is fmaf(E4M3(acodes[i]), second[1 + i / 256], second[0]), one fp32 rounding.
__device__ __forceinline__ float nf4_dq_absmax(const uint8_t* acodes, const float* second, int64_t i) {
    return __fmaf_rn(e4m3_to_float(__ldg(acodes + i)), __ldg(second + 1 + (i >> 8)), __ldg(second));
}

// Store one fp32 result in the requested output dtype.
__device__ __forceinline__ void store_out(void* y, size_t idx, int dtype, float v) {
    if (dtype == LQ_F32) {
        static_cast<float*>(y)[idx] = v;
    } else if (dtype == LQ_F16) {
        static_cast<__half*>(y)[idx] = __float2half_rn(v);
    } else {
        static_cast<__nv_bfloat16*>(y)[idx] = __float2bfloat16_rn(v);
    }
}

}  // namespace lq
