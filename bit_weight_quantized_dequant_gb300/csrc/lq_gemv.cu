// lq_gemv / lq_gemv_grouped: decode-sized y = x * W_eff^T for 1 <= M <= 32.
//
// Decode is bound by streaming the packed weights once per token (otf-llm 4.0.1
// README, section 1 "The Memory-Bound Bottleneck": every parameter crosses the
// memory bus once per token), so this kernel is built to keep HBM busy while
// spending as few instructions per weight as it can:
//
//  * Work unit = 64 output rows x one K-split.  Each of the 4 warps owns 16 rows
//    and walks K in steps of 256 columns.  A unit's x slice is staged once in
//    shared memory as binary16, with the anchor columns zeroed (the anchors
//    replace those weights, section 4) and laid out in mma-fragment order.
//  * Per step a thread issues one 16-byte load of codes for each of its two rows
//    (64 codes per row).  The 4-entry codebook of each 32-column group,
//    fmaf(S, C[q], Z) rounded to binary16 (section 3 reconstruction), is held
//    as two byte-split registers, and one PRMT turns a byte-lane selector into
//    two binary16 weights.  The k order inside each 16-wide mma block is
//    permuted the same way for weights and x, so the codes need no shuffling.
//  * The multiply-accumulate runs on tensor cores (mma.sync m16n8k16, binary16
//    in, fp32 accumulate); tokens are the n dimension (up to 4 tiles of 8).
//  * Anchors (section 4) are extra k-blocks of the same accumulator: binary16
//    anchor weights feed the A fragment directly against x gathered at the
//    anchor columns.
//  * Split-K partials go to the handle's workspace; the last unit of a strip to
//    arrive (atomic counter) sums them in a fixed order and writes y, so results
//    do not depend on scheduling.
//  * NF4 (AirQuant README, NF4 block-wise): the 16 binary16 levels live in eight
//    byte-split registers; PRMT looks up 3 index bits in each half of the table
//    and a byte mask built from the 4th bit picks the half.  Each mma block stays
//    inside one 64-column block so the fp32 absmax scales the partial product.

#include <algorithm>
#include <cstdlib>
#include <cstring>

#include "lq_common.cuh"
#include "lq_internal.h"

namespace lq {
namespace {

constexpr int kStep = 256;  // K columns per warp step

struct Frag2 {
    uint4 cg, cg8;           // codes of rows g and g+8 (64 columns each)
    uint32_t sg, zg, sg8, zg8;  // binary16 pairs: scale/offset of the thread's two groups
};

struct FragNF4 {
    uint2 cg[4], cg8[4];     // 16 codes per row in each of the 4 NF4 blocks of a step
    float ag[4], ag8[4];     // absmax per block
};

__device__ __forceinline__ int tile_tokens(int M, int nt) { return min(8, M - 8 * nt); }

// Offset (in halves) of column kk of token m inside the staged code region.
template <int FMT>
__device__ __forceinline__ int xs_offset(int m, int kk, int klen_pad, int M) {
    int bi, tt, hh;
    if (FMT == LQ_FMT_2BIT_LM_G32) {
        const int step = kk >> 8, r = kk & 255;
        tt = r >> 6;
        const int i = (r >> 4) & 3, e = r & 15;
        bi = step * 16 + i * 4 + (e & 3);
        hh = e >> 2;
    } else {
        const int nb = kk >> 6, r = kk & 63;
        tt = r >> 4;
        const int e = r & 15;
        bi = nb * 4 + (e >> 2);
        hh = e & 3;
    }
    const int nt = m >> 3, gg = m & 7;
    return 8 * nt * klen_pad + (bi * tile_tokens(M, nt) + gg) * 16 + tt * 4 + hh;
}

// Offset (in halves) of anchor a of token m inside the staged anchor region.
__device__ __forceinline__ int xa_offset(int m, int a, int a_pad, int M, int base) {
    const int s = a & 15;
    const int tt = (s & 7) >> 1, hh = (s & 1) + 2 * (s >> 3);
    const int nt = m >> 3, gg = m & 7;
    return base + 8 * nt * a_pad + ((a >> 4) * tile_tokens(M, nt) + gg) * 16 + tt * 4 + hh;
}


// Byte-split 4-entry table of binary16 fmaf(s, C[q], z): RA holds the low bytes, RB the high bytes.
__device__ __forceinline__ void lut2(uint16_t s_bits, uint16_t z_bits, uint32_t& RA, uint32_t& RB, float& peak) {
    const float s = half_bits_to_float(s_bits), z = half_bits_to_float(z_bits);
    peak = fmaxf(peak, __fmaf_rn(1.52f, fabsf(s), fabsf(z)));   // the table's largest |value| (binary16 range check)
    const uint32_t p01 = pack_half2_rn(__fmaf_rn(s, -1.52f, z), __fmaf_rn(s, -0.45f, z));
    const uint32_t p23 = pack_half2_rn(__fmaf_rn(s, 0.45f, z), __fmaf_rn(s, 1.52f, z));
    RA = prmt(p01, p23, 0x6420);
    RB = prmt(p01, p23, 0x7531);
}

// Codes at bit offset 2j of each byte of w -> two binary16 pairs (bytes 0,1) and (bytes 2,3).
__device__ __forceinline__ void expand2(uint32_t w, int j, uint32_t RA, uint32_t RB, uint32_t& lo, uint32_t& hi) {
    const uint32_t t = (w >> (2 * j)) & 0x03030303u;
    const uint32_t sel = t * 0x11u + 0x40404040u;  // per byte: nibble0 = q (low byte), nibble1 = q+4 (high byte)
    lo = prmt(RA, RB, sel);
    hi = prmt(RA, RB, sel >> 16);
}

// NF4: four codes (16-bit chunk c of w) -> half2(T[c0],T[c1]) and half2(T[c2],T[c3]).
__device__ __forceinline__ void expand_nf4(uint32_t w, int c, const uint32_t (&TL)[4], const uint32_t (&TH)[4],
                                           uint32_t& r01, uint32_t& r23) {
    const uint32_t sel = (c == 0 ? w : (w >> 16)) & 0x7777u;
    const uint32_t mask = prmt(w << 4, w, c == 0 ? 0xD9C8u : 0xFBEAu);  // 0xFF where index bit 3 is set
    const uint32_t lo = (prmt(TL[0], TL[1], sel) & ~mask) | (prmt(TL[2], TL[3], sel) & mask);
    const uint32_t hi = (prmt(TH[0], TH[1], sel) & ~mask) | (prmt(TH[2], TH[3], sel) & mask);
    r01 = prmt(lo, hi, 0x5140);
    r23 = prmt(lo, hi, 0x7362);
}

__device__ __forceinline__ uint2 lds64(const uint16_t* p) { return *reinterpret_cast<const uint2*>(p); }

template <int NT>
__device__ __forceinline__ void mma_block(float (&acc)[NT][4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                          const uint16_t* xs, int bi, int klen_pad, int M, int g, int t) {
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        const int Mt = tile_tokens(M, nt);
        uint2 b = make_uint2(0u, 0u);
        if (g < Mt) b = lds64(xs + 8 * nt * klen_pad + (bi * Mt + g) * 16 + t * 4);
        mma_f16_16816(acc[nt], a0, a1, a2, a3, b.x, b.y);
    }
}

// ---- loads ---------------------------------------------------------------------

__device__ __forceinline__ Frag2 load2(const uint8_t* cg, const uint8_t* cg8, const uint16_t* sg, const uint16_t* zg,
                                       const uint16_t* sg8, const uint16_t* zg8, int valid_cols, bool vg, bool vg8,
                                       bool wide) {
    // valid_cols: columns of this thread's 64-column chunk inside K (>= 64 full, 32 half, <= 0 none)
    Frag2 f;
    f.cg = make_uint4(0, 0, 0, 0);
    f.cg8 = make_uint4(0, 0, 0, 0);
    f.sg = f.zg = f.sg8 = f.zg8 = 0;
    if (valid_cols >= 64 && wide) {
        if (vg) {
            f.cg = ldg128(cg);
            f.sg = ldg32(sg);
            f.zg = ldg32(zg);
        }
        if (vg8) {
            f.cg8 = ldg128(cg8);
            f.sg8 = ldg32(sg8);
            f.zg8 = ldg32(zg8);
        }
    } else if (valid_cols > 0) {
        const bool two = valid_cols >= 64;
        if (vg) {
            const uint2 a = ldg64(cg);
            const uint2 b = two ? ldg64(cg + 8) : make_uint2(0, 0);
            f.cg = make_uint4(a.x, a.y, b.x, b.y);
            f.sg = (uint32_t)sg[0] | (two ? ((uint32_t)sg[1] << 16) : 0u);
            f.zg = (uint32_t)zg[0] | (two ? ((uint32_t)zg[1] << 16) : 0u);
        }
        if (vg8) {
            const uint2 a = ldg64(cg8);
            const uint2 b = two ? ldg64(cg8 + 8) : make_uint2(0, 0);
            f.cg8 = make_uint4(a.x, a.y, b.x, b.y);
            f.sg8 = (uint32_t)sg8[0] | (two ? ((uint32_t)sg8[1] << 16) : 0u);
            f.zg8 = (uint32_t)zg8[0] | (two ? ((uint32_t)zg8[1] << 16) : 0u);
        }
    }
    return f;
}

template <int NT>
__device__ __forceinline__ void compute2(const Frag2& f, float (&acc)[NT][4], const uint16_t* xs, int step,
                                         int klen_pad, int M, int g, int t, float& peak) {
    uint32_t RA[4], RB[4];
    lut2((uint16_t)f.sg, (uint16_t)f.zg, RA[0], RB[0], peak);
    lut2((uint16_t)(f.sg >> 16), (uint16_t)(f.zg >> 16), RA[1], RB[1], peak);
    lut2((uint16_t)f.sg8, (uint16_t)f.zg8, RA[2], RB[2], peak);
    lut2((uint16_t)(f.sg8 >> 16), (uint16_t)(f.zg8 >> 16), RA[3], RB[3], peak);
    const uint32_t wg[4] = {f.cg.x, f.cg.y, f.cg.z, f.cg.w};
    const uint32_t wg8[4] = {f.cg8.x, f.cg8.y, f.cg8.z, f.cg8.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int lg = i >> 1;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            uint32_t a0, a1, a2, a3;
            expand2(wg[i], j, RA[lg], RB[lg], a0, a2);
            expand2(wg8[i], j, RA[2 + lg], RB[2 + lg], a1, a3);
            mma_block<NT>(acc, a0, a1, a2, a3, xs, step * 16 + i * 4 + j, klen_pad, M, g, t);
        }
    }
}

// ig, ig8: index of the first block maximum (row-major in [N][K/64]); with `second` set
// (double quantization) `am` holds the maxima's E4M3 codes, else the fp32 maxima.
__device__ __forceinline__ FragNF4 load_nf4(const uint8_t* cg, const uint8_t* cg8, const void* am, const float* second,
                                            int64_t ig, int64_t ig8, int valid_blocks, bool vg, bool vg8) {
    FragNF4 f;
#pragma unroll
    for (int nb = 0; nb < 4; ++nb) {
        const bool v = nb < valid_blocks;
        f.cg[nb] = (v && vg) ? ldg64(cg + 32 * nb) : make_uint2(0, 0);
        f.cg8[nb] = (v && vg8) ? ldg64(cg8 + 32 * nb) : make_uint2(0, 0);
        if (second) {
            f.ag[nb] = (v && vg) ? nf4_dq_absmax(static_cast<const uint8_t*>(am), second, ig + nb) : 0.f;
            f.ag8[nb] = (v && vg8) ? nf4_dq_absmax(static_cast<const uint8_t*>(am), second, ig8 + nb) : 0.f;
        } else {
            f.ag[nb] = (v && vg) ? __ldg(static_cast<const float*>(am) + ig + nb) : 0.f;
            f.ag8[nb] = (v && vg8) ? __ldg(static_cast<const float*>(am) + ig8 + nb) : 0.f;
        }
    }
    return f;
}

template <int NT>
__device__ __forceinline__ void compute_nf4(const FragNF4& f, float (&acc)[NT][4], const uint32_t (&TL)[4],
                                            const uint32_t (&TH)[4], const uint16_t* xs, int step, int klen_pad,
                                            int M, int g, int t) {
#pragma unroll
    for (int nb = 0; nb < 4; ++nb) {
        float part[NT][4];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) part[nt][0] = part[nt][1] = part[nt][2] = part[nt][3] = 0.f;
#pragma unroll
        for (int b = 0; b < 4; ++b) {
            const uint32_t w = (b < 2) ? f.cg[nb].x : f.cg[nb].y;
            const uint32_t w8 = (b < 2) ? f.cg8[nb].x : f.cg8[nb].y;
            uint32_t a0, a1, a2, a3;
            expand_nf4(w, b & 1, TL, TH, a0, a2);
            expand_nf4(w8, b & 1, TL, TH, a1, a3);
            mma_block<NT>(part, a0, a1, a2, a3, xs, (step * 4 + nb) * 4 + b, klen_pad, M, g, t);
        }
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            acc[nt][0] = __fmaf_rn(f.ag[nb], part[nt][0], acc[nt][0]);
            acc[nt][1] = __fmaf_rn(f.ag[nb], part[nt][1], acc[nt][1]);
            acc[nt][2] = __fmaf_rn(f.ag8[nb], part[nt][2], acc[nt][2]);
            acc[nt][3] = __fmaf_rn(f.ag8[nb], part[nt][3], acc[nt][3]);
        }
    }
}

// ---- the kernel ----------------------------------------------------------------

template <int NT, int FMT>
__global__ void __launch_bounds__(kGemvThreads) gemv_kernel(const __grid_constant__ GemvParams P) {
    extern __shared__ uint4 smem_u4[];
    uint16_t* xs = reinterpret_cast<uint16_t*>(smem_u4);
    __shared__ int s_last;

    // ---- locate the unit
    const int64_t u = blockIdx.x;
    int p = 0;
    while (p + 1 < P.count && u >= P.d[p + 1].unit_begin) ++p;
    const GemvDesc& D = P.d[p];
    const int64_t local = u - D.unit_begin;
    const int64_t per_member = (int64_t)D.strips * D.parts;
    const int64_t l = local / per_member;
    const int rem = (int)(local - l * per_member);
    const int strip = rem / D.parts;
    const int part = rem - strip * D.parts;

    const int M = P.M, N = D.N, K = D.K, A = D.A;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, t = lane & 3;
    const int rg = strip * kGemvStripRows + warp * 16 + g, rg8 = rg + 8;
    const bool vg = rg < N, vg8 = rg8 < N;

    const uint8_t* codes = D.codes + l * D.stride_codes;
    const char* scales = static_cast<const char*>(D.scales) + l * D.stride_scales;
    const uint16_t* x = reinterpret_cast<const uint16_t*>(static_cast<const char*>(D.x) + l * D.stride_x);
    void* y = static_cast<char*>(D.y) + l * D.stride_y;

    const bool anchor_part = (D.S > 1) && (part == D.S);
    const bool has_codes = !anchor_part;
    const bool do_anchors = (FMT == LQ_FMT_2BIT_LM_G32) && A > 0 && (anchor_part || D.S == 1);
    const int k0 = has_codes ? part * D.KC : 0;
    const int klen = has_codes ? min(D.KC, K - k0) : 0;
    const int klen_pad = (klen + kStep - 1) / kStep * kStep;
    const int a_pad = do_anchors ? (A + 15) / 16 * 16 : 0;
    const int a_base = M * klen_pad;
    const int32_t* anchor_idx = (FMT == LQ_FMT_2BIT_LM_G32 && A > 0)
        ? reinterpret_cast<const int32_t*>(reinterpret_cast<const char*>(D.anchor_idx) + l * D.stride_anchor_idx)
        : nullptr;

    // ---- issue the first weight loads before staging x, so their latency overlaps it
    const bool wide = (K % 64) == 0;
    Frag2 f2;
    FragNF4 f4;
    const uint8_t *cg = nullptr, *cg8 = nullptr;
    const uint16_t *sg = nullptr, *zg = nullptr, *sg8 = nullptr, *zg8 = nullptr;
    int64_t ig = 0, ig8 = 0;   // NF4: first block-maximum index of rows rg, rg + 8
    const float* second = P.format == LQ_FMT_NF4_DQ
                              ? reinterpret_cast<const float*>(reinterpret_cast<const char*>(D.offsets) + l * D.stride_offsets)
                              : nullptr;
    const int nsteps = klen_pad / kStep;
    if (has_codes) {
        if (FMT == LQ_FMT_2BIT_LM_G32) {
            const uint16_t* sc = reinterpret_cast<const uint16_t*>(scales);
            const uint16_t* of = reinterpret_cast<const uint16_t*>(reinterpret_cast<const char*>(D.offsets) + l * D.stride_offsets);
            const int64_t rgc = vg ? rg : 0, rg8c = vg8 ? rg8 : 0;
            cg = codes + rgc * (K / 4) + k0 / 4 + 16 * t;
            cg8 = codes + rg8c * (K / 4) + k0 / 4 + 16 * t;
            sg = sc + rgc * (K / 32) + k0 / 32 + 2 * t;
            zg = of + rgc * (K / 32) + k0 / 32 + 2 * t;
            sg8 = sc + rg8c * (K / 32) + k0 / 32 + 2 * t;
            zg8 = of + rg8c * (K / 32) + k0 / 32 + 2 * t;
            f2 = load2(cg, cg8, sg, zg, sg8, zg8, klen - 64 * t, vg, vg8, wide);
        } else {
            const int64_t rgc = vg ? rg : 0, rg8c = vg8 ? rg8 : 0;
            cg = codes + rgc * (K / 2) + k0 / 2 + 8 * t;
            cg8 = codes + rg8c * (K / 2) + k0 / 2 + 8 * t;
            ig = rgc * (K / 64) + k0 / 64;
            ig8 = rg8c * (K / 64) + k0 / 64;
            f4 = load_nf4(cg, cg8, scales, second, ig, ig8, klen / 64, vg, vg8);
        }
    }

    // ---- stage x (binary16, fragment order; bf16 x scaled per token, see x_scale) and the
    // gathered anchor columns
    const uint32_t* xmaxw = P.x_bf16 ? D.xmax + l * M : nullptr;
    if (has_codes) {
        const int chunks = klen_pad / 8;
        for (int idx = tid; idx < M * chunks; idx += kGemvThreads) {
            const int m = idx / chunks;
            const int kk = (idx - m * chunks) * 8;
            uint4 v = make_uint4(0, 0, 0, 0);
            if (kk < klen) v = *reinterpret_cast<const uint4*>(x + (int64_t)m * K + k0 + kk);
            const uint16_t h[8] = {(uint16_t)v.x, (uint16_t)(v.x >> 16), (uint16_t)v.y, (uint16_t)(v.y >> 16),
                                   (uint16_t)v.z, (uint16_t)(v.z >> 16), (uint16_t)v.w, (uint16_t)(v.w >> 16)};
            const float sc = P.x_bf16 ? x_scale(xmaxw[m]) : 1.f;
#pragma unroll
            for (int e = 0; e < 8; ++e)
                xs[xs_offset<FMT>(m, kk + e, klen_pad, M)] = P.x_bf16 ? bf16_to_half_scaled(h[e], sc) : h[e];
        }
    }
    if (FMT == LQ_FMT_2BIT_LM_G32 && do_anchors) {
        for (int idx = tid; idx < M * a_pad; idx += kGemvThreads) {
            const int ap = a_pad > 0 ? a_pad : 16;
            const int m = idx / ap;
            const int a = idx - m * ap;
            uint16_t v = 0;
            const int k = a < A ? anchor_idx[a] : -1;
            if ((unsigned)k < (unsigned)K)
                v = P.x_bf16 ? bf16_to_half_scaled(x[(int64_t)m * K + k], x_scale(xmaxw[m])) : x[(int64_t)m * K + k];
            xs[xa_offset(m, a, a_pad, M, a_base)] = v;
        }
    }
    __syncthreads();
    if (FMT == LQ_FMT_2BIT_LM_G32 && has_codes && A > 0) {
        // anchors replace the 2-bit weights in their columns: zero x there
        for (int a = tid; a < A; a += kGemvThreads) {
            const int k = anchor_idx[a];
            if (k >= k0 && k < k0 + klen)
                for (int m = 0; m < M; ++m) xs[xs_offset<FMT>(m, k - k0, klen_pad, M)] = 0;
        }
        __syncthreads();
    }

    float acc[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;
    float peak = 0.f;

    // ---- main loop over K
    if (has_codes) {
        if (FMT == LQ_FMT_2BIT_LM_G32) {
            for (int s = 0; s < nsteps; ++s) {
                Frag2 nxt;
                if (s + 1 < nsteps)
                    nxt = load2(cg + 64 * (s + 1), cg8 + 64 * (s + 1), sg + 8 * (s + 1), zg + 8 * (s + 1),
                                sg8 + 8 * (s + 1), zg8 + 8 * (s + 1), klen - kStep * (s + 1) - 64 * t, vg, vg8, wide);
                compute2<NT>(f2, acc, xs, s, klen_pad, M, g, t, peak);
                f2 = nxt;
            }
        } else {
            uint32_t TL[4], TH[4];
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
                const uint32_t p01 = pack_half2_rn(kNF4[4 * q4 + 0], kNF4[4 * q4 + 1]);
                const uint32_t p23 = pack_half2_rn(kNF4[4 * q4 + 2], kNF4[4 * q4 + 3]);
                TL[q4] = prmt(p01, p23, 0x6420);
                TH[q4] = prmt(p01, p23, 0x7531);
            }
            for (int s = 0; s < nsteps; ++s) {
                FragNF4 nxt;
                if (s + 1 < nsteps)
                    nxt = load_nf4(cg + 128 * (s + 1), cg8 + 128 * (s + 1), scales, second, ig + 4 * (s + 1),
                                   ig8 + 4 * (s + 1), klen / 64 - 4 * (s + 1), vg, vg8);
                compute_nf4<NT>(f4, acc, TL, TH, xs, s, klen_pad, M, g, t);
                f4 = nxt;
            }
        }
    }

    // ---- anchors: binary16 weights straight into the A fragment
    if (do_anchors) {
        const uint16_t* aw = reinterpret_cast<const uint16_t*>(reinterpret_cast<const char*>(D.anchor_w) + l * D.stride_anchor_w);
        const uint16_t* awg = aw + (int64_t)(vg ? rg : 0) * D.ld_anchor;
        const uint16_t* awg8 = aw + (int64_t)(vg8 ? rg8 : 0) * D.ld_anchor;
        for (int ab = 0; ab < a_pad / 16; ++ab) {
            const int a = 16 * ab + 2 * t;
            auto pair = [&](const uint16_t* row, int aa, bool v) -> uint32_t {
                if (!v || aa >= A) return 0u;
                uint32_t w = ldg32(row + aa);
                return (aa + 1 < A) ? w : (w & 0xFFFFu);
            };
            const uint32_t a0 = pair(awg, a, vg), a2 = pair(awg, a + 8, vg);
            const uint32_t a1 = pair(awg8, a, vg8), a3 = pair(awg8, a + 8, vg8);
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                const int Mt = tile_tokens(M, nt);
                uint2 b = make_uint2(0u, 0u);
                if (g < Mt) b = lds64(xs + a_base + 8 * nt * a_pad + (ab * Mt + g) * 16 + t * 4);
                mma_f16_16816(acc[nt], a0, a1, a2, a3, b.x, b.y);
            }
        }
    }

    // ---- epilogue
    if (FMT == LQ_FMT_2BIT_LM_G32 && peak >= kHalfOverflow && P.status) atomicOr(P.status, 2);
    auto unscale = [&](int m) -> float { return P.x_bf16 ? x_unscale(xmaxw[m]) : 1.f; };
    if (D.parts == 1) {
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            const int m0 = 8 * nt + 2 * t, m1 = m0 + 1;
            if (vg) {
                if (m0 < M) store_out(y, (size_t)m0 * N + rg, P.y_dtype, acc[nt][0] * unscale(m0));
                if (m1 < M) store_out(y, (size_t)m1 * N + rg, P.y_dtype, acc[nt][1] * unscale(m1));
            }
            if (vg8) {
                if (m0 < M) store_out(y, (size_t)m0 * N + rg8, P.y_dtype, acc[nt][2] * unscale(m0));
                if (m1 < M) store_out(y, (size_t)m1 * N + rg8, P.y_dtype, acc[nt][3] * unscale(m1));
            }
        }
        return;
    }
    const int64_t strip_id = D.strip_begin + l * D.strips + strip;
    float* strip_base = P.partials + D.partial_begin + (l * D.strips + strip) * (int64_t)D.parts * M * kGemvStripRows;
    float* mine = strip_base + (int64_t)part * M * kGemvStripRows;
    const int r = warp * 16 + g;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        const int m0 = 8 * nt + 2 * t, m1 = m0 + 1;
        if (m0 < M) {
            mine[m0 * kGemvStripRows + r] = acc[nt][0];
            mine[m0 * kGemvStripRows + r + 8] = acc[nt][2];
        }
        if (m1 < M) {
            mine[m1 * kGemvStripRows + r] = acc[nt][1];
            mine[m1 * kGemvStripRows + r + 8] = acc[nt][3];
        }
    }
    __threadfence();
    __syncthreads();
    if (tid == 0) {
        const unsigned old = atomicAdd(P.counters + strip_id, 1u);
        s_last = (old == (unsigned)(D.parts - 1));
    }
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    for (int idx = tid; idx < M * kGemvStripRows; idx += kGemvThreads) {
        const int m = idx / kGemvStripRows, rr = idx - m * kGemvStripRows;
        const int n = strip * kGemvStripRows + rr;
        if (n >= N) continue;
        float sum = 0.f;
        for (int p0 = 0; p0 < D.parts; p0 += 8) {   // eight loads in flight, then the adds in part order
            float v[8];
#pragma unroll
            for (int k = 0; k < 8; ++k)
                v[k] = p0 + k < D.parts ? __ldcg(strip_base + ((int64_t)(p0 + k) * M + m) * kGemvStripRows + rr) : 0.f;
#pragma unroll
            for (int k = 0; k < 8; ++k)
                if (p0 + k < D.parts) sum += v[k];
        }
        store_out(y, (size_t)m * N + n, P.y_dtype, sum * unscale(m));
    }
    if (tid == 0) P.counters[strip_id] = 0u;
}

// ---- host side -----------------------------------------------------------------

template <int NT, int FMT>
lq_status run(const GemvParams& P, size_t smem, cudaStream_t stream) {
    auto kern = gemv_kernel<NT, FMT>;
    if (smem > 48 * 1024) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
            return LQ_ERR_CUDA;
    }
    kern<<<(unsigned)P.total_units, kGemvThreads, smem, stream>>>(P);
    return cudaPeekAtLastError() == cudaSuccess ? LQ_OK : LQ_ERR_CUDA;
}

template <int FMT>
lq_status run_fmt(const GemvParams& P, size_t smem, cudaStream_t stream) {
    const int nt = (P.M + 7) / 8;
    if (nt == 1) return run<1, FMT>(P, smem, stream);
    if (nt == 2) return run<2, FMT>(P, smem, stream);
    return run<4, FMT>(P, smem, stream);
}

int round_up(int a, int b) { return (a + b - 1) / b * b; }

}  // namespace

lq_status launch_gemv(lq_handle h, const lq_problem* probs, int count, cudaStream_t stream) {
    GemvWorkspace ws;
    ws.num_sms = h->num_sms;
    ws.max_smem_optin = h->max_smem_optin;
    ws.partials = h->partials;
    ws.partial_floats = h->partial_floats;
    ws.counters = h->counters;
    ws.num_counters = h->num_counters;
    ws.clear_counters = false;
    ws.status = h->status_flag;
    return launch_gemv_ws(ws, probs, count, stream);
}

lq_status launch_gemv_layers(lq_handle h, const lq_problem* probs, const int* counts, int layers, cudaStream_t stream) {
    // One grouped launch per layer, in stream order: each ring-kernel launch lets the next one
    // start its CTAs' first weight copies while its own last CTAs finish (programmatic
    // dependent launch), and the next launch waits for it before reading its x.
    for (int l = 0, off = 0; l < layers; off += counts[l], ++l) {
        const lq_status st = launch_gemv(h, probs + off, counts[l], stream);
        if (st != LQ_OK) return st;
    }
    return LQ_OK;
}

// The streaming kernel takes every launch whose K are multiples of 256; the
// split-K kernel below covers the rest (any K % 32 == 0).
// LQ_GEMV_KERNEL=regs forces the register-fed kernel (for comparisons and tests).
lq_status launch_gemv_ws(const GemvWorkspace& ws, const lq_problem* probs, int count, cudaStream_t stream) {
    if (probs[0].format == LQ_FMT_INT4_G32)   // INT4 decodes on the ring kernel only (K % 256 == 0)
        return gemv_stream_eligible(probs, count) ? launch_gemv_stream(ws, probs, count, stream) : LQ_ERR_UNSUPPORTED;
    const char* force = getenv("LQ_GEMV_KERNEL");
    const bool regs_only = force && strcmp(force, "regs") == 0;
    if (!regs_only && gemv_stream_eligible(probs, count)) {
        // (a launch whose copies of x or row-block slots do not fit falls back to split-K)
        const lq_status s = launch_gemv_stream(ws, probs, count, stream);
        if (s != LQ_ERR_UNSUPPORTED && s != LQ_ERR_WORKSPACE) return s;
    }
    return launch_gemv_regs(ws, probs, count, stream);
}

lq_status launch_gemv_regs(const GemvWorkspace& ws, const lq_problem* probs, int count, cudaStream_t stream) {
    GemvParams P;
    memset(&P, 0, sizeof(P));
    const int M = probs[0].M;
    P.count = count;
    P.M = M;
    P.format = probs[0].format;
    P.x_bf16 = probs[0].x_dtype == LQ_BF16;
    P.y_dtype = probs[0].y_dtype;

    // K columns per split: bounded by the staged x slice (M x KC binary16 <= 32 KiB)
    const int kc_target = M <= 8 ? 2048 : (M <= 16 ? 1024 : 512);
    int64_t strips_total = 0;
    int S[kMaxGroup];
    for (int i = 0; i < count; ++i) {
        const lq_problem& q = probs[i];
        const int K = q.K;
        S[i] = (K <= kc_target + kc_target / 4) ? 1 : (K + kc_target - 1) / kc_target;
        strips_total += (int64_t)q.batch * ((q.N + kGemvStripRows - 1) / kGemvStripRows);
    }
    // small launches: split K further so every SM gets a few units
    int64_t units = 0;
    for (int i = 0; i < count; ++i) {
        const int64_t st = (int64_t)probs[i].batch * ((probs[i].N + kGemvStripRows - 1) / kGemvStripRows);
        units += st * S[i];
    }
    const int64_t want = 3LL * ws.num_sms;
    if (units < want) {
        for (int i = 0; i < count; ++i) {
            const int max_s = std::max(1, probs[i].K / kStep);
            const int64_t mult = (want + units - 1) / units;
            S[i] = (int)std::min<int64_t>(max_s, (int64_t)S[i] * mult);
        }
    }

    int kc_pad = 0, a_pad = 0;
    int64_t unit = 0, strip = 0, partial_floats = 0;
    for (int i = 0; i < count; ++i) {
        const lq_problem& q = probs[i];
        GemvDesc& d = P.d[i];
        d.codes = q.codes;
        d.scales = q.scales;
        d.offsets = static_cast<const uint16_t*>(q.offsets);
        d.anchor_idx = q.anchor_idx;
        d.anchor_w = q.anchor_w;
        d.x = q.x;
        d.y = q.y;
        d.stride_codes = q.stride_codes;
        d.stride_scales = q.stride_scales;
        d.stride_offsets = q.stride_offsets;
        d.stride_anchor_idx = q.stride_anchor_idx;
        d.stride_anchor_w = q.stride_anchor_w;
        d.stride_x = q.stride_x;
        d.stride_y = q.stride_y;
        d.N = q.N;
        d.K = q.K;
        d.A = (q.format == LQ_FMT_2BIT_LM_G32) ? q.A : 0;
        d.ld_anchor = q.ld_anchor;
        d.batch = q.batch;
        if (S[i] == 1) {
            d.S = 1;
            d.KC = q.K;
        } else {
            d.KC = round_up((q.K + S[i] - 1) / S[i], kStep);
            d.S = (q.K + d.KC - 1) / d.KC;
        }
        d.parts = d.S + ((d.S > 1 && d.A > 0) ? 1 : 0);
        d.strips = (q.N + kGemvStripRows - 1) / kGemvStripRows;
        d.unit_begin = unit;
        unit += (int64_t)q.batch * d.strips * d.parts;
        if (d.parts > 1) {
            d.strip_begin = strip;
            d.partial_begin = partial_floats;
            strip += (int64_t)q.batch * d.strips;
            partial_floats += (int64_t)q.batch * d.strips * d.parts * M * kGemvStripRows;
        } else {
            d.strip_begin = 0;
            d.partial_begin = 0;
        }
        kc_pad = std::max(kc_pad, round_up(d.KC, kStep));
        if (d.A > 0 && (d.S == 1 || d.parts > d.S)) a_pad = std::max(a_pad, round_up(d.A, 16));
    }
    // bf16 x: one max |x| word per (member, token) row after the partial sums
    int64_t xrows = 0;
    for (int i = 0; i < count; ++i) {
        P.d[i].xmax = reinterpret_cast<const uint32_t*>(ws.partials + partial_floats) + xrows;
        xrows += (int64_t)probs[i].batch * M;
    }
    if (!P.x_bf16) xrows = 0;
    if ((size_t)strip > ws.num_counters || (size_t)(partial_floats + xrows) > ws.partial_floats) return LQ_ERR_WORKSPACE;
    P.kc_pad = kc_pad;
    P.a_pad = a_pad;
    P.partials = ws.partials;
    P.counters = ws.counters;
    P.status = ws.status;
    P.total_units = unit;
    if (unit == 0) return LQ_OK;
    if (unit > 0x7fffffffLL) return LQ_ERR_UNSUPPORTED;
    const size_t smem = (size_t)M * (kc_pad + a_pad) * sizeof(uint16_t);
    if (smem > (size_t)ws.max_smem_optin) return LQ_ERR_UNSUPPORTED;
    if (ws.clear_counters && strip > 0 &&
        cudaMemsetAsync(ws.counters, 0, sizeof(unsigned) * (size_t)strip, stream) != cudaSuccess)
        return LQ_ERR_CUDA;
    if (P.x_bf16) {
        const lq_status st = launch_xmax_rows(probs, count, reinterpret_cast<uint32_t*>(ws.partials + partial_floats), stream);
        if (st != LQ_OK) return st;
    }
    if (P.format == LQ_FMT_2BIT_LM_G32) return run_fmt<LQ_FMT_2BIT_LM_G32>(P, smem, stream);
    return run_fmt<LQ_FMT_NF4_B64>(P, smem, stream);
}

}  // namespace lq
