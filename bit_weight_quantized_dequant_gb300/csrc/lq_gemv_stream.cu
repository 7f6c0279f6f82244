// Streaming decode GEMV (the fast path of lq_gemv / lq_gemv_grouped for K % 256 == 0).
//
// Decode reads every weight once per token (otf-llm 4.0.1 README, section 1, "The
// Memory-Bound Bottleneck"), so the kernel is a bandwidth streamer with the
// section 3/4 reconstruction done in registers:
//
//  * Two small pre-pass kernels write x once per call as binary16 in mma-fragment
//    order with the anchor columns zeroed (anchors replace those weights), and x
//    gathered at the anchor columns.  They chain to the main kernel by programmatic
//    dependent launch; each main CTA issues its first weight loads before it waits.
//  * One CTA = 8 warps over one tile of 16 x (8 / ks) rows and the full K: the ks
//    warps of a row tile split K into contiguous slices, so no partial sums leave
//    the CTA (shared-memory reduction at the end, no atomics, no workspace).
//  * Each thread streams its two rows with 16-byte loads (64 codes per row per
//    256-column step) and 4-byte scale/offset loads, two steps ahead of use.
//  * x fragments come straight from the pre-permuted copy (L1-resident, one 8-byte
//    load per mma).  Lanes whose token does not exist load harmless neighbouring
//    values: they only feed output columns that are never stored.
//  * Dequantization is a PRMT lookup in byte-split binary16 tables of
//    fmaf(S, C[q], Z); the multiply-accumulate is mma.sync m16n8k16 (binary16 in,
//    fp32 accumulate) with tokens as the n dimension.  Anchors are extra k-blocks
//    of the same accumulator, shared round-robin by the warps of a row tile.
//  * NF4: eight byte-split registers hold the 16 binary16 levels; each mma block
//    stays inside one 64-column block so its fp32 absmax scales the partial sums.

#include <algorithm>
#include <cstdlib>
#include <cstring>

#include "lq_common.cuh"
#include "lq_dq.cuh"
#include "lq_internal.h"
#include "lq_tma.cuh"

namespace lq {
namespace {

constexpr int kWarps = 8;
#ifndef LQ_STREAM_MIN_BLOCKS
#define LQ_STREAM_MIN_BLOCKS 2   // resident CTAs per SM the register allocation aims for
#endif
constexpr int kThreadsS = kWarps * 32;

// ---- pre-pass: x -> binary16, anchors zeroed, fragment order ------------------------

struct PrepDesc {
    const uint16_t* x;
    int64_t stride_x;          // bytes
    const int32_t* anchor_idx;
    int64_t stride_anchor_idx; // bytes
    uint16_t* xperm;           // [batch][K/16][M][16]
    uint16_t* xaperm;          // [batch][a_pad/16][M][16]
    int64_t xperm_stride, xaperm_stride;   // halves per batch member
    int K, A, a_pad, batch;
    int ctas;                  // CTAs per batch member
    int64_t cta_begin;         // first CTA of this problem
};

struct PrepParams {
    PrepDesc d[kMaxGroup];
    int count, M, x_bf16, format;
    int64_t total_ctas;
};

constexpr int kPrepItems = 256;    // 8-half output items per pre-pass CTA (one per thread)

__device__ __forceinline__ uint16_t to_half_bits(uint16_t raw, int x_bf16) {
    return x_bf16 ? __half_as_ushort(__float2half_rn(bf16_bits_to_float(raw))) : raw;
}

// One CTA covers kPrepItems consecutive 16-byte items of one batch member: first the
// fragment-ordered copy of x with the anchor columns zeroed (a bitmap of the anchor
// columns in shared memory marks them), then x gathered at the anchor columns.
__global__ void __launch_bounds__(256) xprep_kernel(const __grid_constant__ PrepParams P) {
    extern __shared__ uint32_t anchor_bits[];
    pdl_launch_dependents();
    const int64_t cta = blockIdx.x;
    int p = 0;
    while (p + 1 < P.count && cta >= P.d[p + 1].cta_begin) ++p;
    const PrepDesc& D = P.d[p];
    const int64_t local = cta - D.cta_begin;
    const int64_t l = local / D.ctas;
    const int part = (int)(local - l * D.ctas);
    const int M = P.M, K = D.K, A = D.A;
    const uint16_t* x = reinterpret_cast<const uint16_t*>(reinterpret_cast<const char*>(D.x) + l * D.stride_x);
    const int32_t* aidx = A > 0 ? reinterpret_cast<const int32_t*>(reinterpret_cast<const char*>(D.anchor_idx) + l * D.stride_anchor_idx)
                                : nullptr;
    for (int i = threadIdx.x; i < K / 32; i += blockDim.x) anchor_bits[i] = 0u;
    __syncthreads();
    for (int a = threadIdx.x; a < A; a += blockDim.x) {
        const int k = __ldg(aidx + a);
        atomicOr(&anchor_bits[k >> 5], 1u << (k & 31));
    }
    __syncthreads();
    const int64_t code_items = (int64_t)M * K / 8, all_items = code_items + (int64_t)M * D.a_pad / 8;
    const int64_t i0 = (int64_t)part * kPrepItems, i1 = min(all_items, i0 + kPrepItems);
    for (int64_t it = i0 + threadIdx.x; it < i1; it += blockDim.x) {
        const bool code = it < code_items;
        const int64_t d0 = 8 * (code ? it : it - code_items);
        const int line = (int)(d0 >> 4), pos0 = (int)(d0 & 15);
        const int bi = line / M, m = line - bi * M;
        uint16_t v[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const int pos = pos0 + e, tt = pos >> 2, hh = pos & 3;
            int k = -1;
            if (code) {
                k = P.format == LQ_FMT_2BIT_LM_G32 ? (bi >> 4) * 256 + tt * 64 + ((bi >> 2) & 3) * 16 + hh * 4 + (bi & 3)
                                                   : (bi >> 2) * 64 + tt * 16 + (bi & 3) * 4 + hh;
                if ((anchor_bits[k >> 5] >> (k & 31)) & 1u) k = -1;
            } else {
                const int a = 16 * bi + 2 * tt + (hh & 1) + 8 * (hh >> 1);
                if (a < A) k = __ldg(aidx + a);
            }
            v[e] = k >= 0 ? to_half_bits(x[(int64_t)m * K + k], P.x_bf16) : (uint16_t)0;
        }
        uint16_t* dst = (code ? D.xperm + l * D.xperm_stride : D.xaperm + l * D.xaperm_stride) + d0;
        *reinterpret_cast<uint4*>(dst) = make_uint4((uint32_t)v[0] | ((uint32_t)v[1] << 16), (uint32_t)v[2] | ((uint32_t)v[3] << 16),
                                                    (uint32_t)v[4] | ((uint32_t)v[5] << 16), (uint32_t)v[6] | ((uint32_t)v[7] << 16));
    }
}

struct SDesc {
    const uint8_t* codes;
    const void* scales;
    const uint16_t* offsets;
    const uint16_t* anchor_w;
    const uint16_t* xperm;      // [batch][K/16][M][16] (+ padding)
    const uint16_t* xaperm;     // [batch][a_pad/16][M][16] (+ padding)
    void* y;
    int64_t stride_codes, stride_scales, stride_offsets, stride_anchor_w, stride_y;
    int64_t xperm_stride, xaperm_stride;   // halves
    int N, K, A, ld_anchor, batch, ks, tiles;   // ks: warps per row tile (K slices); tiles: tiles per member
    int64_t tile_begin;   // first global tile of this problem
};

struct SParams {
    SDesc d[kMaxGroup];
    int count, M, y_dtype;
    int64_t total_tiles;
};

template <int NT, int MT>
__device__ __forceinline__ void mma_xg(float (&acc)[NT][4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                       const uint2 (&b)[NT]) {
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) mma_f16_16816(acc[nt], a0, a1, a2, a3, b[nt].x, b[nt].y);
}

// x fragment of mma block bi (n-tile nt) for this thread: 8 bytes of the permuted copy.
// `xp` already points at this thread's token and lane; for more than 8 tokens the
// n-tile offsets come from `tok` (absent tokens read the last real token: their
// products only reach output columns that are never stored).
template <int MT>
__device__ __forceinline__ uint2 xfrag(const uint16_t* xp, int bi, int M, int tok_nt) {
    const int MM = MT > 0 ? MT : M;
    return __ldg(reinterpret_cast<const uint2*>(xp + bi * MM * 16 + tok_nt));
}

// One warp's view of a tile: rows, K slice and pointers at the first step of its slice.
struct TileView {
    bool valid;
    int p, tile, rtiles, ks, rt, slice, steps;
    int64_t l;
};

__device__ __forceinline__ TileView view_tile(const SParams& P, int64_t T, int warp) {
    TileView v;
    v.valid = T < P.total_tiles;
    if (!v.valid) return v;
    int p = 0;
    while (p + 1 < P.count && T >= P.d[p + 1].tile_begin) ++p;
    const SDesc& D = P.d[p];
    const int64_t local = T - D.tile_begin;
    v.p = p;
    v.l = local / D.tiles;
    v.tile = (int)(local - v.l * D.tiles);
    v.ks = D.ks;
    v.rtiles = kWarps / D.ks;
    v.rt = warp / D.ks;
    v.slice = warp - v.rt * D.ks;
    const int nsteps = D.K / 256;
    const int s_begin = (int)((int64_t)nsteps * v.slice / D.ks);
    v.steps = (int)((int64_t)nsteps * (v.slice + 1) / D.ks) - s_begin;
    v.tile = v.tile;
    return v;
}

// Streams one thread's two rows, step after step, across the tiles of its CTA.
template <int FMT, int MT>
struct Loader {
    const uint8_t *cg, *cg8;
    const uint16_t *sg, *sg8, *zg, *zg8;   // 2-bit scales/offsets (NF4: sg/sg8 hold the absmax rows)
    const uint16_t* xsrc;                  // this step's x slice in the permuted copy (+ 8 halves per lane)
    int step, steps;
    int64_t T;
    bool valid;

    __device__ __forceinline__ void open(const SParams& P, int64_t T_, int warp, int g, int t) {
        T = T_;
        const TileView v = view_tile(P, T, warp);
        valid = v.valid;
        if (!valid) return;
        const SDesc& D = P.d[v.p];
        const int M = MT > 0 ? MT : P.M;
        const int N = D.N, K = D.K;
        const int rg = (v.tile * v.rtiles + v.rt) * 16 + g, rg8 = rg + 8;
        const int64_t r0 = rg < N ? rg : 0, r1 = rg8 < N ? rg8 : 0;   // rows past N read row 0, never stored
        const int s_begin = (int)((int64_t)(K / 256) * v.slice / v.ks);
        const uint8_t* codes = D.codes + v.l * D.stride_codes;
        const char* sc = static_cast<const char*>(D.scales) + v.l * D.stride_scales;
        if (FMT == LQ_FMT_2BIT_LM_G32) {
            const uint16_t* s16 = reinterpret_cast<const uint16_t*>(sc);
            const uint16_t* o16 = reinterpret_cast<const uint16_t*>(reinterpret_cast<const char*>(D.offsets) + v.l * D.stride_offsets);
            cg = codes + r0 * (K / 4) + 16 * t + 64 * s_begin;
            cg8 = codes + r1 * (K / 4) + 16 * t + 64 * s_begin;
            sg = s16 + r0 * (K / 32) + 2 * t + 8 * s_begin;
            sg8 = s16 + r1 * (K / 32) + 2 * t + 8 * s_begin;
            zg = o16 + r0 * (K / 32) + 2 * t + 8 * s_begin;
            zg8 = o16 + r1 * (K / 32) + 2 * t + 8 * s_begin;
        } else {
            const float* am = reinterpret_cast<const float*>(sc);
            cg = codes + r0 * (K / 2) + 8 * t + 128 * s_begin;
            cg8 = codes + r1 * (K / 2) + 8 * t + 128 * s_begin;
            sg = reinterpret_cast<const uint16_t*>(am + r0 * (K / 64) + 4 * s_begin);
            sg8 = reinterpret_cast<const uint16_t*>(am + r1 * (K / 64) + 4 * s_begin);
        }
        const int MM = MT > 0 ? MT : M;
        xsrc = D.xperm + v.l * D.xperm_stride + (int64_t)s_begin * 256 * MM + (threadIdx.x & 31) * 8;
        step = 0;
        steps = v.steps;
    }
    __device__ __forceinline__ void advance(const SParams& P, int warp, int g, int t) {
        if (++step < steps) {
            if (FMT == LQ_FMT_2BIT_LM_G32) {
                cg += 64; cg8 += 64; sg += 8; sg8 += 8; zg += 8; zg8 += 8;
            } else {
                cg += 128; cg8 += 128; sg += 8; sg8 += 8;   // 4 floats
            }
            xsrc += 256 * (MT > 0 ? MT : P.M);
        } else {
            open(P, T + gridDim.x, warp, g, t);
        }
    }
};

struct Step2 {
    uint4 c0, c1;
    uint32_t s0, z0, s1, z1;
};

struct StepNF4 {
    uint2 c0[4], c1[4];
    float a0[4], a1[4];
};

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(smem)), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

template <int FMT, int MT, int NT>
__global__ void __launch_bounds__(kThreadsS, LQ_STREAM_MIN_BLOCKS) gemv_stream_kernel(const __grid_constant__ SParams P) {
    __shared__ float red[kWarps][16][(NT * 8) + 1];
    // per warp, three x slices of one 256-column step each (binary16, fragment order)
    extern __shared__ __align__(16) uint16_t xring[];
    const int M = MT > 0 ? MT : P.M;
    const int MM = MT > 0 ? MT : M;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
    uint16_t* xw = xring + warp * 3 * 256 * MM;             // this warp's ring
    const int xlane = min(g, M - 1) * 16 + t * 4;            // this lane's fragment inside a block
    int tok[NT];   // x-fragment offset of each n-tile's token (clamped to the last real token)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) tok[nt] = (min(8 * nt + g, M - 1) - min(g, M - 1)) * 16;

    float acc[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;

    // The finished tile: anchors of this warp, then the K-slice reduction and the store of y.
    int64_t T = blockIdx.x;
    TileView CV = view_tile(P, T, warp);
    int cstep = 0;
    auto finish_tile = [&]() {
        const TileView v = CV;
        const SDesc& D = P.d[v.p];
        const int N = D.N;
        const int rg = (v.tile * v.rtiles + v.rt) * 16 + g, rg8 = rg + 8;
        if (FMT == LQ_FMT_2BIT_LM_G32 && D.A > 0) {
            const int64_t r0 = rg < N ? rg : 0, r1 = rg8 < N ? rg8 : 0;
            const uint16_t* aw = reinterpret_cast<const uint16_t*>(reinterpret_cast<const char*>(D.anchor_w) + v.l * D.stride_anchor_w);
            const uint16_t* awg = aw + r0 * D.ld_anchor;
            const uint16_t* awg8 = aw + r1 * D.ld_anchor;
            const uint16_t* xa = D.xaperm + v.l * D.xaperm_stride + xlane;
            const int A = D.A;
            auto pair = [&](const uint16_t* row, int a) -> uint32_t {
                if (a >= A) return 0u;
                const uint32_t w = ldg32(row + a);
                return (a + 1 < A) ? w : (w & 0xFFFFu);
            };
            for (int ab = v.slice; ab < (A + 15) / 16; ab += v.ks) {
                const int a = 16 * ab + 2 * t;
                const uint32_t a0 = pair(awg, a), a2 = pair(awg, a + 8);
                const uint32_t a1 = pair(awg8, a), a3 = pair(awg8, a + 8);
                uint2 xb[NT];
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) xb[nt] = __ldg(reinterpret_cast<const uint2*>(xa + ab * MM * 16 + tok[nt]));
                mma_xg<NT, MT>(acc, a0, a1, a2, a3, xb);
            }
        }
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            const int m0 = 8 * nt + 2 * t, m1 = m0 + 1;
            if (m0 < M) {
                red[warp][g][m0] = acc[nt][0];
                red[warp][g + 8][m0] = acc[nt][2];
            }
            if (m1 < M) {
                red[warp][g][m1] = acc[nt][1];
                red[warp][g + 8][m1] = acc[nt][3];
            }
            acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;
        }
        __syncthreads();
        void* y = static_cast<char*>(D.y) + v.l * D.stride_y;
        const int ks = v.ks;
        for (int idx = threadIdx.x; idx < v.rtiles * 16 * M; idx += kThreadsS) {
            const int rtile = idx / (16 * M), rem = idx - rtile * 16 * M;
            const int m = rem / 16, r = rem - m * 16;
            const int n = (v.tile * v.rtiles + rtile) * 16 + r;
            if (n >= N) continue;
            float sum = 0.f;
            for (int sl = 0; sl < ks; ++sl) sum += red[rtile * ks + sl][r][m];
            store_out(y, (size_t)m * N + n, P.y_dtype, sum);
        }
        __syncthreads();
        T += gridDim.x;
        CV = view_tile(P, T, warp);
        cstep = 0;
    };
    auto step_done = [&]() {
        if (++cstep == CV.steps) finish_tile();
    };

    Loader<FMT, MT> L;
    L.open(P, blockIdx.x, warp, g, t);
    // the x slice of a step (source `src`) goes to ring slot `slot`, one commit group per step
    auto issue_x = [&](int slot, const uint16_t* src, bool valid) {
        if (valid) {
            uint16_t* dst = xw + slot * 256 * MM + lane * 8;
#pragma unroll
            for (int c = 0; c < MM; ++c) cp_async16(dst + c * 256, src + c * 256);
        }
        cp_async_commit();
    };

    if (FMT == LQ_FMT_2BIT_LM_G32) {
        auto issue_w = [&](Step2& f) {
            if (!L.valid) return;
            f.c0 = ldg128(L.cg);
            f.c1 = ldg128(L.cg8);
            f.s0 = ldg32(L.sg);
            f.z0 = ldg32(L.zg);
            f.s1 = ldg32(L.sg8);
            f.z1 = ldg32(L.zg8);
            L.advance(P, warp, g, t);
        };
        auto issue = [&](Step2& f, int slot) {
            issue_x(slot, L.xsrc, L.valid);
            issue_w(f);
        };
        auto compute = [&](const Step2& f, int slot) {
            cp_async_wait<2>();   // this step's x slice has landed (the two later ones may be in flight)
            __syncwarp();
            const uint16_t* xs = xw + slot * 256 * MM + xlane;
            uint32_t RA[4], RB[4];
            lut2_bits((uint16_t)f.s0, (uint16_t)f.z0, RA[0], RB[0]);
            lut2_bits((uint16_t)(f.s0 >> 16), (uint16_t)(f.z0 >> 16), RA[1], RB[1]);
            lut2_bits((uint16_t)f.s1, (uint16_t)f.z1, RA[2], RB[2]);
            lut2_bits((uint16_t)(f.s1 >> 16), (uint16_t)(f.z1 >> 16), RA[3], RB[3]);
            const uint32_t w0[4] = {f.c0.x, f.c0.y, f.c0.z, f.c0.w};
            const uint32_t w1[4] = {f.c1.x, f.c1.y, f.c1.z, f.c1.w};
#pragma unroll
            for (int ii = 0; ii < 4; ++ii) {
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    uint32_t a0, a1, a2, a3;
                    expand2_fast(w0[ii], j, RA[ii >> 1], RB[ii >> 1], a0, a2);
                    expand2_fast(w1[ii], j, RA[2 + (ii >> 1)], RB[2 + (ii >> 1)], a1, a3);
                    uint2 xb[NT];
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt)
                        xb[nt] = *reinterpret_cast<const uint2*>(xs + (ii * 4 + j) * MM * 16 + tok[nt]);
                    mma_xg<NT, MT>(acc, a0, a1, a2, a3, xb);
                }
            }
            __syncwarp();   // every lane has read this slot before it is refilled
            step_done();
        };
        // three register buffers (and x slots), two steps in flight across tile boundaries,
        // unrolled so the buffers never move
        Step2 fa, fb, fc;
        // weights of the first two steps before waiting for the x pre-pass, then their x slices
        const uint16_t* xs0 = L.xsrc;
        const bool v0 = L.valid;
        issue_w(fa);
        const uint16_t* xs1 = L.xsrc;
        const bool v1 = L.valid;
        issue_w(fb);
        pdl_wait();
        issue_x(0, xs0, v0);
        issue_x(1, xs1, v1);
        for (;;) {
            if (!CV.valid) break;
            issue(fc, 2);
            compute(fa, 0);
            if (!CV.valid) break;
            issue(fa, 0);
            compute(fb, 1);
            if (!CV.valid) break;
            issue(fb, 1);
            compute(fc, 2);
        }
    } else {
        uint32_t TL[4], TH[4];
        nf4_tables(TL, TH);
        auto issue_w = [&](StepNF4& f) {
            if (!L.valid) return;
            const float* ag = reinterpret_cast<const float*>(L.sg);
            const float* ag8 = reinterpret_cast<const float*>(L.sg8);
#pragma unroll
            for (int nb = 0; nb < 4; ++nb) {
                f.c0[nb] = ldg64(L.cg + 32 * nb);
                f.c1[nb] = ldg64(L.cg8 + 32 * nb);
                f.a0[nb] = __ldg(ag + nb);
                f.a1[nb] = __ldg(ag8 + nb);
            }
            L.advance(P, warp, g, t);
        };
        auto issue = [&](StepNF4& f, int slot) {
            issue_x(slot, L.xsrc, L.valid);
            issue_w(f);
        };
        auto compute = [&](const StepNF4& f, int slot) {
            cp_async_wait<1>();
            __syncwarp();
            const uint16_t* xs = xw + slot * 256 * MM + xlane;
#pragma unroll
            for (int nb = 0; nb < 4; ++nb) {
                uint2 xb[4][NT];
#pragma unroll
                for (int b = 0; b < 4; ++b)
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) xb[b][nt] = *reinterpret_cast<const uint2*>(xs + (nb * 4 + b) * MM * 16 + tok[nt]);
                float part[NT][4];
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) part[nt][0] = part[nt][1] = part[nt][2] = part[nt][3] = 0.f;
#pragma unroll
                for (int b = 0; b < 4; ++b) {
                    uint32_t a0, a1, a2, a3;
                    expand_nf4_fast(b < 2 ? f.c0[nb].x : f.c0[nb].y, b & 1, TL, TH, a0, a2);
                    expand_nf4_fast(b < 2 ? f.c1[nb].x : f.c1[nb].y, b & 1, TL, TH, a1, a3);
                    mma_xg<NT, MT>(part, a0, a1, a2, a3, xb[b]);
                }
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    acc[nt][0] = __fmaf_rn(f.a0[nb], part[nt][0], acc[nt][0]);
                    acc[nt][1] = __fmaf_rn(f.a0[nb], part[nt][1], acc[nt][1]);
                    acc[nt][2] = __fmaf_rn(f.a1[nb], part[nt][2], acc[nt][2]);
                    acc[nt][3] = __fmaf_rn(f.a1[nb], part[nt][3], acc[nt][3]);
                }
            }
            __syncwarp();
            step_done();
        };
        StepNF4 fa, fb;
        const uint16_t* xs0 = L.xsrc;
        const bool v0 = L.valid;
        issue_w(fa);
        pdl_wait();
        issue_x(0, xs0, v0);
        for (;;) {
            if (!CV.valid) break;
            issue(fb, 1);
            compute(fa, 0);
            if (!CV.valid) break;
            issue(fa, 0);
            compute(fb, 1);
        }
    }
}

template <int FMT, int MT, int NT>
lq_status launch_s(const SParams& P, int64_t tiles, int num_sms, cudaStream_t stream) {
    const size_t smem = (size_t)kWarps * 3 * 256 * P.M * sizeof(uint16_t);   // x rings
    static int per_sm = 0;   // resident CTAs per SM for this instantiation (same smem for a given M)
    static size_t per_sm_smem = 0;
    if (per_sm == 0 || per_sm_smem != smem) {
        // static reduction buffer + dynamic x rings may pass the 48 KiB default: always opt in
        if (cudaFuncSetAttribute(gemv_stream_kernel<FMT, MT, NT>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
            return LQ_ERR_CUDA;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, gemv_stream_kernel<FMT, MT, NT>, kThreadsS, smem) != cudaSuccess)
            return LQ_ERR_CUDA;
        per_sm_smem = smem;
    }
    const int64_t grid = std::min<int64_t>(tiles, (int64_t)num_sms * std::max(1, per_sm));
    cudaLaunchConfig_t cfg;
    memset(&cfg, 0, sizeof(cfg));
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(kThreadsS);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, gemv_stream_kernel<FMT, MT, NT>, P) != cudaSuccess) return LQ_ERR_CUDA;
    return cudaPeekAtLastError() == cudaSuccess ? LQ_OK : LQ_ERR_CUDA;
}

template <int FMT>
lq_status launch_s_fmt(const SParams& P, int64_t tiles, int num_sms, cudaStream_t stream) {
    switch (P.M) {
        case 1: return launch_s<FMT, 1, 1>(P, tiles, num_sms, stream);
        case 2: return launch_s<FMT, 2, 1>(P, tiles, num_sms, stream);
        case 3: return launch_s<FMT, 3, 1>(P, tiles, num_sms, stream);
        case 4: return launch_s<FMT, 4, 1>(P, tiles, num_sms, stream);
        case 5: return launch_s<FMT, 5, 1>(P, tiles, num_sms, stream);
        case 6: return launch_s<FMT, 6, 1>(P, tiles, num_sms, stream);
        case 7: return launch_s<FMT, 7, 1>(P, tiles, num_sms, stream);
        case 8: return launch_s<FMT, 8, 1>(P, tiles, num_sms, stream);
        default: return LQ_ERR_UNSUPPORTED;   // more than 8 tokens: the split-K kernel
    }
}

int round_up(int a, int b) { return (a + b - 1) / b * b; }

}  // namespace

bool gemv_stream_eligible(const lq_problem* probs, int count) {
    if (probs[0].M > 8) return false;   // the x rings (3 steps x M tokens per warp) must stay small
    for (int i = 0; i < count; ++i)
        if (probs[i].K % 256 != 0) return false;
    return true;
}

lq_status launch_gemv_stream(const GemvWorkspace& ws, const lq_problem* probs, int count, cudaStream_t stream) {
    SParams P;
    PrepParams Q;
    memset(&P, 0, sizeof(P));
    memset(&Q, 0, sizeof(Q));
    const int M = probs[0].M;
    const int fmt = probs[0].format;
    P.count = Q.count = count;
    P.M = Q.M = M;
    P.y_dtype = probs[0].y_dtype;
    Q.format = fmt;
    Q.x_bf16 = probs[0].x_dtype == LQ_BF16;

    int64_t blocks = 0, prep = 0, xhalves = 0;
    int max_k = 0;
    // minimum K steps per warp (LQ_GEMV_STEPS_PER_WARP overrides, for tuning experiments)
    int spw = 8;
    if (const char* e = getenv("LQ_GEMV_STEPS_PER_WARP")) spw = std::max(1, atoi(e));
    for (int i = 0; i < count; ++i) {
        const lq_problem& q = probs[i];
        const int A = fmt == LQ_FMT_2BIT_LM_G32 ? q.A : 0;
        SDesc& d = P.d[i];
        PrepDesc& e = Q.d[i];
        d.codes = q.codes;
        d.scales = q.scales;
        d.offsets = q.offsets;
        d.anchor_w = q.anchor_w;
        d.y = q.y;
        d.stride_codes = q.stride_codes;
        d.stride_scales = q.stride_scales;
        d.stride_offsets = q.stride_offsets;
        d.stride_anchor_w = q.stride_anchor_w;
        d.stride_y = q.stride_y;
        d.N = q.N;
        d.K = q.K;
        d.A = A;
        d.ld_anchor = q.ld_anchor;
        d.batch = q.batch;
        // warps per row tile (K slices): as many as keep >= spw steps of 256 columns per warp
        const int steps = q.K / 256;
        d.ks = 8;
        while (d.ks > 1 && steps < spw * d.ks) d.ks /= 2;
        const int rows_per_cta = 16 * (kWarps / d.ks);
        d.tiles = (q.N + rows_per_cta - 1) / rows_per_cta;
        d.tile_begin = blocks;
        blocks += (int64_t)q.batch * d.tiles;
        const int a_pad = A > 0 ? round_up(A, 64) : 0;
        d.xperm_stride = (int64_t)M * q.K;
        d.xaperm_stride = (int64_t)M * a_pad;
        xhalves += (int64_t)q.batch * (d.xperm_stride + d.xaperm_stride) + 2 * 128;
        e.x = static_cast<const uint16_t*>(q.x);
        e.stride_x = q.stride_x;
        e.anchor_idx = A > 0 ? q.anchor_idx : nullptr;
        e.stride_anchor_idx = q.stride_anchor_idx;
        e.K = q.K;
        e.A = A;
        e.a_pad = a_pad;
        e.batch = q.batch;
        e.xperm_stride = d.xperm_stride;
        e.xaperm_stride = d.xaperm_stride;
        const int64_t items = ((int64_t)M * q.K + (int64_t)M * a_pad) / 8;
        e.ctas = (int)((items + kPrepItems - 1) / kPrepItems);
        e.cta_begin = prep;
        prep += (int64_t)q.batch * e.ctas;
        max_k = std::max(max_k, q.K);
    }
    if (blocks > 0x7fffffffLL) return LQ_ERR_UNSUPPORTED;
    if ((size_t)((xhalves + 1) / 2 + 64) > ws.partial_floats) return LQ_ERR_WORKSPACE;
    uint16_t* xp = reinterpret_cast<uint16_t*>((reinterpret_cast<uintptr_t>(ws.partials) + 255) & ~uintptr_t(255));
    for (int i = 0; i < count; ++i) {
        P.d[i].xperm = Q.d[i].xperm = xp;
        xp += (int64_t)probs[i].batch * P.d[i].xperm_stride;
        xp = reinterpret_cast<uint16_t*>((reinterpret_cast<uintptr_t>(xp) + 255) & ~uintptr_t(255));
        P.d[i].xaperm = Q.d[i].xaperm = xp;
        xp += (int64_t)probs[i].batch * P.d[i].xaperm_stride;
        xp = reinterpret_cast<uint16_t*>((reinterpret_cast<uintptr_t>(xp) + 255) & ~uintptr_t(255));
    }
    Q.total_ctas = prep;
    if (blocks == 0) return LQ_OK;

    // x pre-pass, then the main kernel, chained by programmatic dependent launch
    if (Q.total_ctas > 0x7fffffffLL) return LQ_ERR_UNSUPPORTED;
    const size_t prep_smem = sizeof(uint32_t) * (size_t)std::max(1, max_k / 32);
    if (prep_smem > 48 * 1024) return LQ_ERR_UNSUPPORTED;
    xprep_kernel<<<(unsigned)Q.total_ctas, 256, prep_smem, stream>>>(Q);
    if (cudaPeekAtLastError() != cudaSuccess) return LQ_ERR_CUDA;
    P.total_tiles = blocks;
    if (fmt == LQ_FMT_2BIT_LM_G32) return launch_s_fmt<LQ_FMT_2BIT_LM_G32>(P, blocks, ws.num_sms, stream);
    return launch_s_fmt<LQ_FMT_NF4_B64>(P, blocks, ws.num_sms, stream);
}

}  // namespace lq
