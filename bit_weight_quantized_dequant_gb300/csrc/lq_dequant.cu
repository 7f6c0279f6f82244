// lq_dequant: dense W_eff from the packed formats, bit-exact to the definitions.
//
// 2-bit (otf-llm 4.0.1 README, sections 2-4): W_eff = fmaf(S_g, C[q], Z_g) in
// fp32 with one rounding; anchor columns then take their binary16 value.
// NF4 (AirQuant README, NF4 block-wise): W_eff = T[q] * absmax, one fp32 rounding; with
// double quantization (QLoRA) the maxima are decoded from their 8-bit float codes first.
// INT4 (otf-llm 4.0.1 README, the v3.2 engine): W_eff[n][perm[j]] = S * q, an exact
// fp32 product; anchor columns then take their binary16 value.
// fp16/bf16 outputs are one round-to-nearest-even conversion of the fp32 value.
//
// One thread expands one 32-bit word of codes (16 two-bit or 8 four-bit codes);
// the kernel is bound by the dense output writes.

#include "lq_common.cuh"
#include "lq_internal.h"

namespace lq {
namespace {

template <int OUT>
__device__ __forceinline__ void store16(void* out, size_t idx, const float (&v)[16]) {
    if (OUT == LQ_F32) {
        float4* p = reinterpret_cast<float4*>(static_cast<float*>(out) + idx);
        p[0] = make_float4(v[0], v[1], v[2], v[3]);
        p[1] = make_float4(v[4], v[5], v[6], v[7]);
        p[2] = make_float4(v[8], v[9], v[10], v[11]);
        p[3] = make_float4(v[12], v[13], v[14], v[15]);
    } else {
        uint32_t w[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            uint16_t lo, hi;
            if (OUT == LQ_F16) {
                lo = __half_as_ushort(__float2half_rn(v[2 * i]));
                hi = __half_as_ushort(__float2half_rn(v[2 * i + 1]));
            } else {
                lo = __bfloat16_as_ushort(__float2bfloat16_rn(v[2 * i]));
                hi = __bfloat16_as_ushort(__float2bfloat16_rn(v[2 * i + 1]));
            }
            w[i] = (uint32_t)lo | ((uint32_t)hi << 16);
        }
        uint4* p = reinterpret_cast<uint4*>(static_cast<uint16_t*>(out) + idx);
        p[0] = make_uint4(w[0], w[1], w[2], w[3]);
        p[1] = make_uint4(w[4], w[5], w[6], w[7]);
    }
}

template <int OUT>
__device__ __forceinline__ void store8(void* out, size_t idx, const float (&v)[8]) {
    if (OUT == LQ_F32) {
        float4* p = reinterpret_cast<float4*>(static_cast<float*>(out) + idx);
        p[0] = make_float4(v[0], v[1], v[2], v[3]);
        p[1] = make_float4(v[4], v[5], v[6], v[7]);
    } else {
        uint32_t w[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            uint16_t lo, hi;
            if (OUT == LQ_F16) {
                lo = __half_as_ushort(__float2half_rn(v[2 * i]));
                hi = __half_as_ushort(__float2half_rn(v[2 * i + 1]));
            } else {
                lo = __bfloat16_as_ushort(__float2bfloat16_rn(v[2 * i]));
                hi = __bfloat16_as_ushort(__float2bfloat16_rn(v[2 * i + 1]));
            }
            w[i] = (uint32_t)lo | ((uint32_t)hi << 16);
        }
        *reinterpret_cast<uint4*>(static_cast<uint16_t*>(out) + idx) = make_uint4(w[0], w[1], w[2], w[3]);
    }
}

template <int OUT>
__global__ void __launch_bounds__(256) dequant_2bit_kernel(const uint8_t* __restrict__ codes,
                                                           const uint16_t* __restrict__ scales,
                                                           const uint16_t* __restrict__ offsets, void* out,
                                                           int N, int K) {
    const int64_t words_per_row = K / 16;
    const int64_t total = (int64_t)N * words_per_row;
    for (int64_t w = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; w < total; w += (int64_t)gridDim.x * blockDim.x) {
        const int64_t n = w / words_per_row;
        const int64_t wk = w - n * words_per_row;
        const uint32_t word = ldg32(codes + n * (K / 4) + wk * 4);
        const int64_t g = n * (K / 32) + wk / 2;
        const float s = half_bits_to_float(scales[g]);
        const float z = half_bits_to_float(offsets[g]);
        const float L0 = __fmaf_rn(s, -1.52f, z);
        const float L1 = __fmaf_rn(s, -0.45f, z);
        const float L2 = __fmaf_rn(s, 0.45f, z);
        const float L3 = __fmaf_rn(s, 1.52f, z);
        float v[16];
#pragma unroll
        for (int c = 0; c < 16; ++c) {
            const uint32_t q = (word >> (2 * c)) & 3u;
            v[c] = (q & 2u) ? ((q & 1u) ? L3 : L2) : ((q & 1u) ? L1 : L0);
        }
        store16<OUT>(out, (size_t)(n * K + wk * 16), v);
    }
}

template <int OUT>
__global__ void __launch_bounds__(256) anchor_scatter_kernel(const int32_t* __restrict__ anchor_idx,
                                                             const uint16_t* __restrict__ anchor_w, int A,
                                                             int ld_anchor, void* out, int N, int K) {
    const int64_t total = (int64_t)N * A;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t n = i / A;
        const int a = (int)(i - n * A);
        const float v = half_bits_to_float(anchor_w[n * ld_anchor + a]);
        store_out(out, (size_t)(n * K + anchor_idx[a]), OUT, v);
    }
}

// NF4; with `second` set (double quantization), `absmax` holds the E4M3 codes of the
// block maxima and each maximum is decoded as fmaf(E4M3(code), s2, mean).
template <int OUT>
__global__ void __launch_bounds__(256) dequant_nf4_kernel(const uint8_t* __restrict__ codes,
                                                          const void* __restrict__ absmax,
                                                          const float* __restrict__ second, void* out, int N,
                                                          int K) {
    __shared__ float table[16];
    if (threadIdx.x < 16) table[threadIdx.x] = kNF4[threadIdx.x];
    __syncthreads();
    const int64_t words_per_row = K / 8;
    const int64_t total = (int64_t)N * words_per_row;
    for (int64_t w = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; w < total; w += (int64_t)gridDim.x * blockDim.x) {
        const int64_t n = w / words_per_row;
        const int64_t wk = w - n * words_per_row;
        const uint32_t word = ldg32(codes + n * (K / 2) + wk * 4);
        const int64_t blk = n * (K / 64) + wk / 8;
        const float am = second ? nf4_dq_absmax(static_cast<const uint8_t*>(absmax), second, blk)
                                : static_cast<const float*>(absmax)[blk];
        float v[8];
#pragma unroll
        for (int c = 0; c < 8; ++c) v[c] = __fmul_rn(table[(word >> (4 * c)) & 15u], am);
        store8<OUT>(out, (size_t)(n * K + wk * 8), v);
    }
}

// INT4: one thread per 32-bit word (8 permuted positions of one group), each value
// written at its input column perm[j].
template <int OUT>
__global__ void __launch_bounds__(256) dequant_int4_kernel(const uint8_t* __restrict__ codes,
                                                           const uint16_t* __restrict__ scales,
                                                           const int32_t* __restrict__ perm, void* out, int N, int K) {
    const int64_t words_per_row = K / 8;
    const int64_t total = (int64_t)N * words_per_row;
    for (int64_t w = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; w < total; w += (int64_t)gridDim.x * blockDim.x) {
        const int64_t n = w / words_per_row;
        const int64_t wk = w - n * words_per_row;
        const uint32_t word = ldg32(codes + n * (K / 2) + wk * 4);
        const float s = half_bits_to_float(scales[n * (K / 32) + wk / 4]);
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            const int q = ((int)(word << (28 - 4 * c))) >> 28;   // 4-bit two's complement
            const int col = __ldg(perm + wk * 8 + c);
            if ((unsigned)col < (unsigned)K) store_out(out, (size_t)(n * K + col), OUT, __fmul_rn(s, (float)q));
        }
    }
}

int grid_for(int64_t work, int num_sms) {
    int64_t blocks = (work + 255) / 256;
    int64_t cap = (int64_t)num_sms * 16;
    return (int)(blocks < cap ? (blocks > 0 ? blocks : 1) : cap);
}

template <int OUT>
lq_status dequant_typed(lq_handle h, int format, const uint8_t* codes, const void* scales, const void* offsets,
                        const int32_t* anchor_idx, const uint16_t* anchor_w, int A, int ld_anchor, void* w_out,
                        int N, int K, cudaStream_t stream) {
    if (format == LQ_FMT_2BIT_LM_G32 || format == LQ_FMT_INT4_G32) {
        if (format == LQ_FMT_2BIT_LM_G32)
            dequant_2bit_kernel<OUT><<<grid_for((int64_t)N * (K / 16), h->num_sms), 256, 0, stream>>>(
                codes, static_cast<const uint16_t*>(scales), static_cast<const uint16_t*>(offsets), w_out, N, K);
        else
            dequant_int4_kernel<OUT><<<grid_for((int64_t)N * (K / 8), h->num_sms), 256, 0, stream>>>(
                codes, static_cast<const uint16_t*>(scales), static_cast<const int32_t*>(offsets), w_out, N, K);
        if (A > 0) {
            anchor_scatter_kernel<OUT><<<grid_for((int64_t)N * A, h->num_sms), 256, 0, stream>>>(
                anchor_idx, anchor_w, A, ld_anchor, w_out, N, K);
        }
    } else {
        dequant_nf4_kernel<OUT><<<grid_for((int64_t)N * (K / 8), h->num_sms), 256, 0, stream>>>(
            codes, scales, format == LQ_FMT_NF4_DQ ? static_cast<const float*>(offsets) : nullptr, w_out, N, K);
    }
    return cudaPeekAtLastError() == cudaSuccess ? LQ_OK : LQ_ERR_CUDA;
}

}  // namespace

lq_status launch_dequant(lq_handle h, int format, const uint8_t* codes, const void* scales, const void* offsets,
                         const int32_t* anchor_idx, const uint16_t* anchor_w, int A, int ld_anchor, void* w_out,
                         int out_dtype, int N, int K, cudaStream_t stream) {
    switch (out_dtype) {
        case LQ_F32:
            return dequant_typed<LQ_F32>(h, format, codes, scales, offsets, anchor_idx, anchor_w, A, ld_anchor, w_out,
                                         N, K, stream);
        case LQ_F16:
            return dequant_typed<LQ_F16>(h, format, codes, scales, offsets, anchor_idx, anchor_w, A, ld_anchor, w_out,
                                         N, K, stream);
        default:
            return dequant_typed<LQ_BF16>(h, format, codes, scales, offsets, anchor_idx, anchor_w, A, ld_anchor,
                                          w_out, N, K, stream);
    }
}

}  // namespace lq
