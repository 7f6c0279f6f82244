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
//  * Work is cut into units of 16 rows x 256 columns (anchor columns: 16 x 64), and
//    every warp of the launch takes an equal contiguous run of the units of all
//    problems, so no warp waits on another and no tile tail is left.  Row-block sums
//    leave a warp through a slot of its own; the last warp of a block adds the slots
//    in a fixed order (an arrival count tells it), so results are reproducible.
//  * Each thread streams its two rows with 16-byte loads (64 codes per row per
//    unit) and 4-byte scale/offset loads, one unit ahead of use.
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
#include <mutex>
#include <string>
#include <vector>

#include "lq_common.cuh"
#include "lq_dq.cuh"
#include "lq_internal.h"
#include "lq_tma.cuh"

namespace lq {
namespace {

constexpr int kWarps = 8;
constexpr int kAnchorCols = 48;   // anchor columns per anchor unit
#ifndef LQ_STREAM_MIN_BLOCKS
#define LQ_STREAM_MIN_BLOCKS 2   // resident CTAs per SM the register allocation aims for
#endif
constexpr int kThreadsS = kWarps * 32;

// ---- pre-pass: x -> binary16, anchors zeroed, fragment order ------------------------
//
// One warp writes one job: a 256-column step of the fragment-ordered copy of x with
// the anchor columns zeroed (fragment order permutes columns inside a step only), or a
// slice of 256 anchor slots of x gathered at the anchor columns.  Every lane writes
// 16-byte items; no job depends on another.

struct PrepDesc {
    const uint16_t* x;
    int64_t stride_x;          // bytes
    const int32_t* anchor_idx;
    int64_t stride_anchor_idx; // bytes
    uint16_t* xperm;           // [batch][K/16][M][16]
    uint16_t* xaperm;          // [batch][a_pad/16][M][16]
    int64_t xperm_stride, xaperm_stride;   // halves per batch member
    int K, A, a_pad, batch;
    int jobs;                  // jobs per batch member: K/256 steps, then ceil(a_pad/256) anchor slices
    int64_t job_begin;         // first job of this problem
    int xsc_off;               // halves from a member's x copy to its per-token max |x| words (bf16 x)
    int64_t row_begin;         // first (member, token) row of this problem, for the max |x| pass
    const int32_t* perm;       // INT4: the column permutation, and its bytes per member
    int64_t stride_perm;
};

struct PrepParams {
    PrepDesc d[kMaxGroup];
    int count, M, x_bf16, format;
    int ring;                  // write the ring kernel's x layout (see ring_x_pos)
    int64_t total_jobs;
    int64_t total_rows;        // (member, token) rows of all problems
};

// x layout of the ring kernel, per batch member: the code columns in blocks of 16 (block
// q at q * (16 M + 8) halves; token m at m * 16 inside it; column 16q + j + 4e at position
// 4j + e, so a lane's four x values of one mma are one 8-byte load and a token's block is
// two 16-byte loads; the 8-half pad keeps blocks 16-byte aligned and spreads the blocks that
// the four lanes of a row read over two bank groups), then x at the anchor columns in the
// pre-pass's fragment order.
__host__ __device__ constexpr int ring_kstride(int M) { return 16 * M + 8; }
__device__ __forceinline__ int ring_x_pos(int k, int m, int M) {
    return (k >> 4) * ring_kstride(M) + m * 16 + 4 * (k & 3) + ((k >> 2) & 3);
}
// INT4's order inside a block of 16 (permuted) columns: an mma takes columns c, c+4, c+1,
// c+5 (c = 8h + 2kk) from one code word, so those four sit together at 4 * (2h + kk).
__device__ __forceinline__ int int4_block_pos(int r) {
    const int rr = r & 7;
    return 4 * (2 * (r >> 3) + ((rr >> 1) & 1)) + ((rr >> 2) & 1) + 2 * (rr & 1);
}

// Sixteen binary16 x values of one token (columns 16q .. 16q+15, as loaded: word i holds
// columns 2i, 2i+1) to the ring layout's order (output word 2j + u holds columns j + 8u and
// j + 8u + 4).
__device__ __forceinline__ void ring_x_transpose(const uint32_t (&w)[8], uint32_t (&o)[8]) {
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int c0 = j + 8 * u, c1 = c0 + 4;   // same parity: both low or both high halves
            o[2 * j + u] = prmt(w[c0 >> 1], w[c1 >> 1], (c0 & 1) ? 0x7632u : 0x5410u);
        }
}

constexpr int kPrepWarps = 2;   // jobs per pre-pass CTA

__device__ __forceinline__ uint16_t to_half_bits(uint16_t raw, int x_bf16) {
    return x_bf16 ? __half_as_ushort(__float2half_rn(bf16_bits_to_float(raw))) : raw;
}

// bf16 x: max |x| of each (member, token) row over its K columns, as the fp32 bit pattern,
// into the row's word after its x copy (x_scale turns it into the conversion factor).  One
// CTA per row.  (|bf16| bit patterns order like the magnitudes, so the maximum is taken
// on the 15-bit patterns.)
__global__ void __launch_bounds__(256) xmax_kernel(const __grid_constant__ PrepParams P) {
    __shared__ uint32_t red[8];
    const int64_t row = blockIdx.x;
    int p = 0;
    while (p + 1 < P.count && row >= P.d[p + 1].row_begin) ++p;
    const PrepDesc& D = P.d[p];
    const int64_t r = row - D.row_begin, l = r / P.M;
    const int m = (int)(r - l * P.M), K = D.K;
    const uint4* x = reinterpret_cast<const uint4*>(reinterpret_cast<const char*>(D.x) + l * D.stride_x) + (int64_t)m * K / 8;
    uint32_t mx = 0;
    for (int i = threadIdx.x; i < K / 8; i += 256) {
        const uint4 v = __ldg(x + i);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) mx = max(mx, max(w[j] & 0x7FFFu, (w[j] >> 16) & 0x7FFFu));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = mx;
    __syncthreads();
    if (threadIdx.x == 0) {
        for (int i = 1; i < 8; ++i) mx = max(mx, red[i]);
        *reinterpret_cast<uint32_t*>(D.xperm + l * D.xperm_stride + D.xsc_off + 2 * m) = mx << 16;
    }
}

// The conversion factor of token m of member l (1 for binary16 x).
__device__ __forceinline__ float prep_scale(const PrepParams& P, const PrepDesc& D, int64_t l, int m) {
    return P.x_bf16 ? x_scale(*reinterpret_cast<const uint32_t*>(D.xperm + l * D.xperm_stride + D.xsc_off + 2 * m)) : 1.f;
}
__device__ __forceinline__ uint16_t to_half_scaled(uint16_t raw, int x_bf16, float scale) {
    return x_bf16 ? bf16_to_half_scaled(raw, scale) : raw;
}

__global__ void __launch_bounds__(32 * kPrepWarps) xprep_kernel(const __grid_constant__ PrepParams P) {
    __shared__ uint32_t step_bits[kPrepWarps][8];
    pdl_launch_dependents();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t job = (int64_t)blockIdx.x * kPrepWarps + warp;
    if (job >= P.total_jobs) return;
    int p = 0;
    while (p + 1 < P.count && job >= P.d[p + 1].job_begin) ++p;
    const PrepDesc& D = P.d[p];
    const int64_t local = job - D.job_begin;
    const int64_t l = local / D.jobs;
    const int jb = (int)(local - l * D.jobs);
    const int M = P.M, K = D.K, A = D.A;
    const uint16_t* x = reinterpret_cast<const uint16_t*>(reinterpret_cast<const char*>(D.x) + l * D.stride_x);
    const int32_t* aidx = A > 0 ? reinterpret_cast<const int32_t*>(reinterpret_cast<const char*>(D.anchor_idx) + l * D.stride_anchor_idx)
                                : nullptr;
    const int steps = K / 256;
    if (jb < steps && P.ring && P.format == LQ_FMT_INT4_G32) {
        // INT4 in the ring layout: x through the permutation, no column zeroed (anchor positions
        // store q = 0); one item = 16 permuted positions of one token
        const int k0 = jb * 256, S = ring_kstride(M);
        const int32_t* perm = reinterpret_cast<const int32_t*>(reinterpret_cast<const char*>(D.perm) + l * D.stride_perm);
        uint16_t* dst = D.xperm + l * D.xperm_stride + (int64_t)(k0 / 16) * S;
        for (int it = lane; it < 16 * M; it += 32) {
            const int m = it >> 4, ql = it & 15;
            const float sc = prep_scale(P, D, l, m);
            const int4* pp = reinterpret_cast<const int4*>(perm + k0 + 16 * ql);
            uint16_t v[16];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int4 c4 = __ldg(pp + i);
                const int cs[4] = {c4.x, c4.y, c4.z, c4.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int c = cs[e];
                    v[int4_block_pos(4 * i + e)] =
                        (unsigned)c < (unsigned)K ? to_half_scaled(x[(int64_t)m * K + c], P.x_bf16, sc) : (uint16_t)0;
                }
            }
            uint2* d2 = reinterpret_cast<uint2*>(dst + ql * S + m * 16);
#pragma unroll
            for (int i = 0; i < 4; ++i)
                d2[i] = make_uint2((uint32_t)v[4 * i] | ((uint32_t)v[4 * i + 1] << 16), (uint32_t)v[4 * i + 2] | ((uint32_t)v[4 * i + 3] << 16));
        }
    } else if (jb < steps && P.ring) {
        // the ring layout: one item = 16 columns of one token (two 16-byte loads, one 8-word store)
        const int k0 = jb * 256, S = ring_kstride(M);
        if (lane < 8) step_bits[warp][lane] = 0u;
        __syncwarp();
        for (int a0 = 0; a0 < A; a0 += 32) {
            const int a = a0 + lane;
            const int kk = a < A ? __ldg(aidx + a) - k0 : -1;
            if (kk >= 0 && kk < 256) atomicOr(&step_bits[warp][kk >> 5], 1u << (kk & 31));
        }
        __syncwarp();
        uint16_t* dst = D.xperm + l * D.xperm_stride + (int64_t)(k0 / 16) * S;
        for (int it = lane; it < 16 * M; it += 32) {
            const int m = it >> 4, ql = it & 15;
            const float sc = prep_scale(P, D, l, m);
            const uint4* src = reinterpret_cast<const uint4*>(x + (int64_t)m * K + k0 + 16 * ql);
            const uint4 v0 = __ldg(src), v1 = __ldg(src + 1);
            uint32_t w[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w}, o[8];
            const uint32_t amask = (step_bits[warp][ql >> 1] >> (16 * (ql & 1))) & 0xFFFFu;   // anchor columns of the block
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const uint32_t lo = (amask >> (2 * i)) & 1u ? 0u : to_half_scaled((uint16_t)w[i], P.x_bf16, sc);
                const uint32_t hi = (amask >> (2 * i + 1)) & 1u ? 0u : to_half_scaled((uint16_t)(w[i] >> 16), P.x_bf16, sc);
                w[i] = lo | (hi << 16);
            }
            ring_x_transpose(w, o);
            uint2* d2 = reinterpret_cast<uint2*>(dst + ql * S + m * 16);
            d2[0] = make_uint2(o[0], o[1]);
            d2[1] = make_uint2(o[2], o[3]);
            d2[2] = make_uint2(o[4], o[5]);
            d2[3] = make_uint2(o[6], o[7]);
        }
    } else if (jb < steps) {
        const int k0 = jb * 256;
        uint16_t* dst = D.xperm + l * D.xperm_stride + (int64_t)k0 * M;
        // column of element e of item `it` inside this step (fragment order)
        auto col = [&](int it, int e) {
            const int d0 = 8 * it, line = d0 >> 4, pos = (d0 & 15) + e;
            const int bl = line / M, tt = pos >> 2, hh = pos & 3;   // mma block inside the step
            return P.format == LQ_FMT_2BIT_LM_G32 ? tt * 64 + ((bl >> 2) & 3) * 16 + hh * 4 + (bl & 3)
                                                   : (bl >> 2) * 64 + tt * 16 + (bl & 3) * 4 + hh;
        };
        auto tok = [&](int it) { const int line = (8 * it) >> 4; return line - (line / M) * M; };
        // x loads of the first items go out before the anchor bitmap is built: no dependence
        constexpr int C = 4;   // items per lane held in registers at a time
        uint16_t v[C][8];
        auto load = [&](int it0) {
#pragma unroll
            for (int c = 0; c < C; ++c) {
                const int it = it0 + 32 * c + lane;
                if (it < 32 * M) {
                    const int m = tok(it);
#pragma unroll
                    for (int e = 0; e < 8; ++e) v[c][e] = x[(int64_t)m * K + k0 + col(it, e)];
                }
            }
        };
        load(0);
        // anchor columns of this step, as 8 words of bits
        if (lane < 8) step_bits[warp][lane] = 0u;
        __syncwarp();
        for (int a0 = 0; a0 < A; a0 += 8 * 32) {
            int kk[8];   // all loads of a round issue before any of them is used
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int a = a0 + 32 * j + lane;
                kk[j] = a < A ? __ldg(aidx + a) - k0 : -1;
            }
#pragma unroll
            for (int j = 0; j < 8; ++j)
                if (kk[j] >= 0 && kk[j] < 256) atomicOr(&step_bits[warp][kk[j] >> 5], 1u << (kk[j] & 31));
        }
        __syncwarp();
        for (int it0 = 0; it0 < 32 * M; it0 += 32 * C) {
            if (it0 > 0) load(it0);
#pragma unroll
            for (int c = 0; c < C; ++c) {
                const int it = it0 + 32 * c + lane;
                if (it >= 32 * M) continue;
                const float sc = prep_scale(P, D, l, tok(it));
                uint32_t w[4];
#pragma unroll
                for (int e2 = 0; e2 < 4; ++e2) {
                    uint32_t pr = 0;
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const int e = 2 * e2 + h, kl = col(it, e);
                        const bool anchor = (step_bits[warp][kl >> 5] >> (kl & 31)) & 1u;
                        pr |= (uint32_t)(anchor ? (uint16_t)0 : to_half_scaled(v[c][e], P.x_bf16, sc)) << (16 * h);
                    }
                    w[e2] = pr;
                }
                *reinterpret_cast<uint4*>(dst + 8 * it) = make_uint4(w[0], w[1], w[2], w[3]);
            }
        }
    } else {
        // x gathered at anchor slots [256 * j, 256 * j + 256) (zero past A)
        const int a_base = (jb - steps) * 256, n_slots = min(256, D.a_pad - a_base);
        uint16_t* dst = D.xaperm + l * D.xaperm_stride + (int64_t)a_base * M;
        for (int it = lane; it < n_slots * M / 8; it += 32) {
            const int d0 = 8 * it, line = d0 >> 4, pos0 = d0 & 15;
            const int bl = line / M, m = line - bl * M;
            const float sc = prep_scale(P, D, l, m);
            uint16_t v[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const int pos = pos0 + e, tt = pos >> 2, hh = pos & 3;
                const int a = a_base + 16 * bl + 2 * tt + (hh & 1) + 8 * (hh >> 1);
                const int k = a < A ? __ldg(aidx + a) : -1;
                v[e] = (unsigned)k < (unsigned)K ? to_half_scaled(x[(int64_t)m * K + k], P.x_bf16, sc) : (uint16_t)0;
            }
            *reinterpret_cast<uint4*>(dst + d0) = make_uint4((uint32_t)v[0] | ((uint32_t)v[1] << 16), (uint32_t)v[2] | ((uint32_t)v[3] << 16),
                                                            (uint32_t)v[4] | ((uint32_t)v[5] << 16), (uint32_t)v[6] | ((uint32_t)v[7] << 16));
        }
    }
}

// ---- main kernel ---------------------------------------------------------------
//
// Work unit: 16 output rows x 256 code columns of one batch member (code unit), or
// 16 rows x 48 anchor columns (anchor unit: three mma blocks, the register size of a
// code unit's loads).  A problem's units are ordered member,
// 16-row block, then K (code units, then anchor units).  All units of the launch
// form one sequence, and warp w of W takes the contiguous range [U*w/W, U*(w+1)/W):
// every warp does the same work to within one unit, whatever the shapes.  A warp
// keeps the sums of the row block it is in and writes them to its own slot when it
// leaves the block; an arrival count per row block tells the warp that completes the
// block to add the slots in warp order and write y (the result does not depend on
// timing).

struct FDesc {
    const uint8_t* codes;
    const void* scales;
    const uint16_t* offsets;
    const uint16_t* anchor_w;
    const uint16_t* xperm;      // [batch][K/16][M][16]
    const uint16_t* xaperm;     // [batch][a_pad/16][M][16]
    float* part;                // partial sums [batch][rblocks][cmax][M][16], one slot per contributing warp
    unsigned* cnt;              // arrival counts [batch][rblocks]
    void* y;
    int64_t stride_codes, stride_scales, stride_offsets, stride_anchor_w, stride_y;   // bytes per member
    int64_t xperm_stride, xaperm_stride;                                               // halves per member
    int N, K, A, ld_anchor, batch;
    int steps, su, rblocks;     // code units per row block; units per row block (code + anchor)
    int cmax;                   // most warps that can share one row block
    int64_t unit_begin;         // first unit of this problem in the launch
    int64_t xoff;               // first half of this problem's x copies in the x buffer
    int xa_off;                 // ring layout: halves from a member's x to its x at the anchor columns
    int xsc_off;                // halves from a member's x to its per-token max |x| words (bf16 x; see x_scale)
    int a_pad;                  // anchor slots of a member's x at the anchor columns (A rounded up to 48)
    const int32_t* perm;        // INT4: the column permutation (perm[j] = input column at position j)
    int64_t stride_perm;        //   bytes per member
    int G;                      // ring kernel: anchor unit spacing inside a row block (su / anchor units)
    int fuse;                   // ring kernel: 1..16 anchors, carried in each row block's last code unit
    const uint16_t* x;          // the caller's x [batch][M][K] (16-bit) and anchor columns, for
    int64_t stride_x;           //   the in-kernel build of the fragment-ordered copy (bytes)
    const int32_t* anchor_idx;
    int64_t stride_anchor_idx;  // bytes
};

struct FParams {
    // (read first by every warp: kept together so that the first lookups share cache lines)
    int64_t total_units, total_warps;
    int count, div32;           // div32: total_units * total_warps < 2^32, warp ranges in 32-bit arithmetic
    int64_t unit_begin[kMaxGroup];   // first unit of each problem (copies of d[i].unit_begin)
    int* status;                // device status word: bit 2 is raised when a weight table value overflows binary16
    int stage;                  // ring kernel: bytes of one ring stage (a code unit, plus fused anchors if any)
    FDesc d[kMaxGroup];
    const uint16_t* xbuf;       // all x copies: per problem, per member [x in fragment order | x at the anchors]
    int M, y_dtype, x_bf16, format;
    int bitmap_words;           // STAGED: shared-memory words of the anchor bitmap (max K / 32)
};

// First unit of warp w's range, U * w / W (32-bit division when the product fits).
__device__ __forceinline__ int64_t split_at(const FParams& P, int64_t w) {
    if (P.div32) return (int64_t)((uint32_t)P.total_units * (uint32_t)w / (uint32_t)P.total_warps);
    return P.total_units * w / P.total_warps;
}

// The warp whose range [U*w/W, U*(w+1)/W) holds unit u.
__device__ __forceinline__ int64_t owner_of(const FParams& P, int64_t u) {
    if (P.div32) return (int64_t)((((uint32_t)u + 1u) * (uint32_t)P.total_warps - 1u) / (uint32_t)P.total_units);
    return ((u + 1) * P.total_warps - 1) / P.total_units;
}


// Position of a unit: problem, member, 16-row block, unit inside the row block, with
// the problem's units per row block cached.
struct Pos {
    int p, rb, s, steps, su;
    int64_t l;
};

__device__ __forceinline__ Pos locate(const FParams& P, int64_t u) {
    Pos q;
    q.p = 0;
    while (q.p + 1 < P.count && u >= P.unit_begin[q.p + 1]) ++q.p;
    const FDesc& D = P.d[q.p];
    int64_t loc = u - D.unit_begin;
    const int64_t per_member = (int64_t)D.rblocks * D.su;
    if (loc < 0x7fffffff && per_member < 0x7fffffff) {   // (32-bit divisions when the numbers fit)
        const unsigned lu = (unsigned)loc, pm = (unsigned)per_member;
        const unsigned l = lu / pm, rem = lu - l * pm, rb = rem / (unsigned)D.su;
        q.l = l;
        q.rb = (int)rb;
        q.s = (int)(rem - rb * (unsigned)D.su);
    } else {
        q.l = loc / per_member;
        loc -= q.l * per_member;
        q.rb = (int)(loc / D.su);
        q.s = (int)(loc - (int64_t)q.rb * D.su);
    }
    q.steps = D.steps;
    q.su = D.su;
    return q;
}

__device__ __forceinline__ void next_block(const FParams& P, Pos& q) {
    const FDesc& D = P.d[q.p];
    if (++q.rb == D.rblocks) {
        q.rb = 0;
        if (++q.l == D.batch) {
            q.l = 0;
            if (++q.p < P.count) {
                q.steps = P.d[q.p].steps;
                q.su = P.d[q.p].su;
            }
        }
    }
}

// Arrival count update with release and acquire semantics at GPU scope (one instruction, no
// separate membar on either side).
__device__ __forceinline__ unsigned atom_add_acq_rel_gpu(unsigned* p, unsigned v) {
    unsigned old;
    asm volatile("atom.add.acq_rel.gpu.global.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}


// The last warp of a row block adds the slots of its nc contributors in order and writes y.
// A slot holds [M][rows] fp32 sums; rows is 16 (streaming kernel) or 32 (ring kernel).
__device__ __noinline__ void finish_block(const float* slots, int nc, int M, void* y, int N, int row0, int y_dtype,
                                          int lane, int rows = 16) {
    for (int i = lane; i < rows * M; i += 32) {
        const int m = i / rows, row = row0 + (i - m * rows);
        float sum = 0.f;
        for (int c0 = 0; c0 < nc; c0 += 8) {   // eight loads in flight, then the adds in slot order
            float v[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) v[k] = c0 + k < nc ? __ldcg(slots + (c0 + k) * M * rows + i) : 0.f;
#pragma unroll
            for (int k = 0; k < 8; ++k)
                if (c0 + k < nc) sum += v[k];
        }
        if (row < N) store_out(y, (size_t)m * N + row, y_dtype, sum);
    }
}

template <int NT, int MT>
__device__ __forceinline__ void mma_xg(float (&acc)[NT][4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                       const uint2 (&b)[NT]) {
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) mma_f16_16816(acc[nt], a0, a1, a2, a3, b[nt].x, b[nt].y);
}

struct Step2 {
    uint4 c0, c1;
    uint32_t s0, z0, s1, z1;
};

struct StepNF4 {
    uint2 c0[4], c1[4];
    float a0[4], a1[4];
};

// The fragment-ordered copy of one member's x (anchor columns zeroed) and x gathered at
// its anchor columns, written by the whole CTA into shared memory at `dst` (the same
// layout the pre-pass writes to global memory).  `bits` is K/32 words of scratch.
__device__ __forceinline__ void build_member_x(const FParams& P, const FDesc& D, int64_t l, uint16_t* dst, uint32_t* bits) {
    const int M = P.M, K = D.K, A = D.A, a_pad = D.a_pad;
    const uint16_t* x = reinterpret_cast<const uint16_t*>(reinterpret_cast<const char*>(D.x) + l * D.stride_x);
    const int32_t* aidx = A > 0 ? reinterpret_cast<const int32_t*>(reinterpret_cast<const char*>(D.anchor_idx) + l * D.stride_anchor_idx)
                                : nullptr;
    for (int i = threadIdx.x; i < K / 32; i += blockDim.x) bits[i] = 0u;
    __syncthreads();
    for (int a = threadIdx.x; a < A; a += blockDim.x) {
        const int k = __ldg(aidx + a);
        if ((unsigned)k < (unsigned)K) atomicOr(&bits[k >> 5], 1u << (k & 31));   // (a column outside [0, K) is ignored)
    }
    __syncthreads();
    const int items = M * K / 8, aitems = M * a_pad / 8;
    for (int it = threadIdx.x; it < items + aitems; it += blockDim.x) {
        const bool code = it < items;
        const int d0 = 8 * (code ? it : it - items), line = d0 >> 4, pos0 = d0 & 15;
        const int bi = line / M, m = line - bi * M;   // mma block, token
        uint16_t v[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const int pos = pos0 + e, tt = pos >> 2, hh = pos & 3;
            if (code) {
                const int k = P.format == LQ_FMT_2BIT_LM_G32 ? (bi >> 4) * 256 + tt * 64 + ((bi >> 2) & 3) * 16 + hh * 4 + (bi & 3)
                                                             : (bi >> 2) * 64 + tt * 16 + (bi & 3) * 4 + hh;
                v[e] = ((bits[k >> 5] >> (k & 31)) & 1u) ? (uint16_t)0 : to_half_bits(x[(int64_t)m * K + k], P.x_bf16);
            } else {
                const int a = 16 * bi + 2 * tt + (hh & 1) + 8 * (hh >> 1);
                const int k = a < A ? __ldg(aidx + a) : -1;
                v[e] = (unsigned)k < (unsigned)K ? to_half_bits(x[(int64_t)m * K + k], P.x_bf16) : (uint16_t)0;
            }
        }
        *reinterpret_cast<uint4*>(dst + (code ? 0 : (int64_t)M * K) + d0) =
            make_uint4((uint32_t)v[0] | ((uint32_t)v[1] << 16), (uint32_t)v[2] | ((uint32_t)v[3] << 16),
                       (uint32_t)v[4] | ((uint32_t)v[5] << 16), (uint32_t)v[6] | ((uint32_t)v[7] << 16));
    }
    __syncthreads();   // the bitmap is reused by the next member
}

// A warp walks its range as segments: the units of its range inside one row block.
// Inside a segment the code units run in a tight loop (one unit of loads in flight,
// pointers only move), then the anchor units; the row block's sums leave through
// flush() at the segment's end.  x fragments are read straight from the permuted copy
// (L1-resident: every warp of an SM streams the same few tens of KiB).
// (more than two n-tiles of accumulators need the register file of a whole SM per CTA)
template <int FMT, int MT, int NT, bool STAGED>
__global__ void __launch_bounds__(kThreadsS, NT <= 2 ? LQ_STREAM_MIN_BLOCKS : 1) gemv_stream_kernel(const __grid_constant__ FParams P) {
    // STAGED: the x span this CTA's units read is copied to shared memory once
    extern __shared__ __align__(16) uint16_t xsm[];
    const int M = MT > 0 ? MT : P.M;   // MT 0: token count at run time (9..32 tokens, NT n-tiles of 8)
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
    const int64_t W = P.total_warps;
    const int wid = blockIdx.x * kWarps + warp;
    int64_t span0 = 0;
    if (STAGED) {
        const int64_t w_lo = (int64_t)blockIdx.x * kWarps, w_hi = (w_lo + kWarps < W) ? w_lo + kWarps : W;
        if (w_lo >= W) return;   // the whole CTA is idle
        const int64_t uc0 = split_at(P, w_lo), uc1 = split_at(P, w_hi);
        const Pos a = locate(P, uc0), b = locate(P, uc1 - 1);
        const FDesc& Da = P.d[a.p];
        const FDesc& Db = P.d[b.p];
        span0 = Da.xoff + a.l * Da.xperm_stride;
        const int64_t span1 = Db.xoff + (b.l + 1) * Db.xperm_stride;
        uint32_t* bits = reinterpret_cast<uint32_t*>(xsm + (span1 - span0));
        pdl_wait();   // x may come from the kernel before; the workspace is free once it is done
        for (int p = a.p; p <= b.p; ++p) {
            const FDesc& D = P.d[p];
            const int64_t l0 = p == a.p ? a.l : 0, l1 = p == b.p ? b.l : D.batch - 1;
            for (int64_t l = l0; l <= l1; ++l) build_member_x(P, D, l, xsm + (D.xoff + l * D.xperm_stride - span0), bits);
        }
        (void)Db;
    }
    if (wid >= W) return;
    const int64_t u_begin = split_at(P, wid), u_end = split_at(P, wid + 1);
    const int xlane = min(g, M - 1) * 16 + t * 4;            // this lane's fragment inside a block
    int tok[NT];   // x-fragment offset of each n-tile's token (clamped to the last real token)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) tok[nt] = (min(8 * nt + g, M - 1) - min(g, M - 1)) * 16;

    float acc[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;

    // write this warp's sums of row block `q` to its slot; the warp completing the block adds the
    // slots in warp order and writes y
    auto flush = [&](const Pos& q, int units) {
        const FDesc& D = P.d[q.p];
        if (P.x_bf16) {   // remove each token's x scale
            const uint32_t* xmaxw = reinterpret_cast<const uint32_t*>(
                (STAGED ? xsm + (D.xoff + q.l * D.xperm_stride - span0) : D.xperm + q.l * D.xperm_stride) + D.xsc_off);
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    const float u = x_unscale(xmaxw[min(8 * nt + 2 * t + c, M - 1)]);
                    acc[nt][c] *= u;
                    acc[nt][c + 2] *= u;
                }
        }
        if (units == q.su) {
            // the whole row block is this warp's: y straight from the accumulators
            void* y = static_cast<char*>(D.y) + q.l * D.stride_y;
            const int rg = q.rb * 16 + g;
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int m = 8 * nt + 2 * t + (e & 1), row = rg + (e >> 1) * 8;
                    if (m < M && row < D.N) store_out(y, (size_t)m * D.N + row, P.y_dtype, acc[nt][e]);
                    acc[nt][e] = 0.f;
                }
            }
            return;
        }
        const int64_t blk = q.l * D.rblocks + q.rb;
        const int64_t first_u = D.unit_begin + blk * q.su;
        // this warp's slot: its place among the warps that share the block
        const int64_t w0 = first_u >= u_begin ? wid : owner_of(P, first_u);
        float* slots = D.part + blk * D.cmax * M * 16;
        float* mine = slots + (int)(wid - w0) * M * 16;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int m = 8 * nt + 2 * t + (e & 1), r = g + (e >> 1) * 8;
                if (m < M) __stcg(mine + m * 16 + r, acc[nt][e]);
                acc[nt][e] = 0.f;
            }
        }
        __syncwarp();   // orders the warp's slot stores before lane 0's release below
        unsigned last = 0;
        if (lane == 0) {
            // release: this slot is visible with the count; acquire: so are the slots counted before
            const unsigned old = atom_add_acq_rel_gpu(D.cnt + blk, (unsigned)units);
            last = old + (unsigned)units == (unsigned)q.su;
        }
        if (__shfl_sync(0xffffffffu, last, 0)) {
            __syncwarp();   // lane 0's acquire orders the other lanes' slot loads too
            if (lane == 0) D.cnt[blk] = 0u;   // counts start at zero for the next launch
            const int nc = (int)(owner_of(P, first_u + q.su - 1) - w0 + 1);
            finish_block(slots, nc, M, static_cast<char*>(D.y) + q.l * D.stride_y, D.N, q.rb * 16, P.y_dtype, lane);
        }
    };

    Pos q = locate(P, u_begin);
    int64_t u = u_begin;
    float peak = 0.f;      // largest |weight table value| seen (binary16 range check)
    bool waited = false;   // x is read only after the pre-pass has finished
    while (u < u_end) {
        const FDesc& D = P.d[q.p];
        const int64_t left = u_end - u;
        const int n = left < (int64_t)(q.su - q.s) ? (int)left : q.su - q.s;
        const int s_end = q.s + n, code_end = min(s_end, q.steps);
        const int N = D.N, K = D.K;
        const int rg = q.rb * 16 + g, rg8 = rg + 8;
        const int64_t r0 = rg < N ? rg : N - 1, r1 = rg8 < N ? rg8 : N - 1;   // rows past N: never stored
        const uint16_t* xb0 = (STAGED ? xsm + (D.xoff + q.l * D.xperm_stride - span0) : D.xperm + q.l * D.xperm_stride) + xlane;
        if (FMT == LQ_FMT_2BIT_LM_G32) {
            if (q.s < code_end) {
                const uint8_t* cb = D.codes + q.l * D.stride_codes + 16 * t;
                const uint8_t* c0p = cb + r0 * (K / 4);
                const uint8_t* c1p = cb + r1 * (K / 4);
                const uint16_t* s16 = reinterpret_cast<const uint16_t*>(static_cast<const char*>(D.scales) + q.l * D.stride_scales) + 2 * t;
                const uint16_t* o16 = reinterpret_cast<const uint16_t*>(reinterpret_cast<const char*>(D.offsets) + q.l * D.stride_offsets) + 2 * t;
                const uint16_t *s0p = s16 + r0 * (K / 32), *s1p = s16 + r1 * (K / 32);
                const uint16_t *z0p = o16 + r0 * (K / 32), *z1p = o16 + r1 * (K / 32);
                auto load = [&](Step2& f, int s) {
                    f.c0 = ldg128(c0p + 64 * s);
                    f.c1 = ldg128(c1p + 64 * s);
                    f.s0 = ldg32(s0p + 8 * s);
                    f.z0 = ldg32(z0p + 8 * s);
                    f.s1 = ldg32(s1p + 8 * s);
                    f.z1 = ldg32(z1p + 8 * s);
                };
                auto compute = [&](const Step2& f, int s) {
                    const uint16_t* xs = xb0 + (int64_t)s * 256 * M;
                    uint32_t RA[4], RB[4];
                    lut2_bits_peak((uint16_t)f.s0, (uint16_t)f.z0, RA[0], RB[0], peak);
                    lut2_bits_peak((uint16_t)(f.s0 >> 16), (uint16_t)(f.z0 >> 16), RA[1], RB[1], peak);
                    lut2_bits_peak((uint16_t)f.s1, (uint16_t)f.z1, RA[2], RB[2], peak);
                    lut2_bits_peak((uint16_t)(f.s1 >> 16), (uint16_t)(f.z1 >> 16), RA[3], RB[3], peak);
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
                                xb[nt] = *reinterpret_cast<const uint2*>(xs + (ii * 4 + j) * M * 16 + tok[nt]);
                            mma_xg<NT, MT>(acc, a0, a1, a2, a3, xb);
                        }
                    }
                };
                // three buffers: two units of loads in flight
                int s = q.s;
                Step2 fa, fb, fc;
                load(fa, s);
                if (s + 1 < code_end) load(fb, s + 1);
                if (!STAGED && !waited) {
                    pdl_wait();
                    waited = true;
                }
                for (;;) {
                    if (s + 2 < code_end) load(fc, s + 2);
                    compute(fa, s);
                    if (++s >= code_end) break;
                    if (s + 2 < code_end) load(fa, s + 2);
                    compute(fb, s);
                    if (++s >= code_end) break;
                    if (s + 2 < code_end) load(fb, s + 2);
                    compute(fc, s);
                    if (++s >= code_end) break;
                }
            }
            const int anchor_begin = q.s > q.steps ? q.s : q.steps;   // this segment's first anchor unit
            if (anchor_begin < s_end) {
                // anchor units: binary16 anchor weights (zero past A) against x at the anchor columns
                if (!STAGED && !waited) {
                    pdl_wait();
                    waited = true;
                }
                const int A = D.A;
                const uint16_t* aw = reinterpret_cast<const uint16_t*>(reinterpret_cast<const char*>(D.anchor_w) + q.l * D.stride_anchor_w);
                const uint16_t* awg = aw + r0 * D.ld_anchor;
                const uint16_t* awg8 = aw + r1 * D.ld_anchor;
                const uint16_t* xab = (STAGED ? xsm + (D.xoff + q.l * D.xperm_stride - span0) + (int64_t)M * K
                                              : D.xaperm + q.l * D.xaperm_stride) + xlane;
                auto pair = [&](const uint16_t* row, int a) -> uint32_t {
                    if (a >= A) return 0u;
                    const uint32_t w = ldg32(row + a);
                    return (a + 1 < A) ? w : (w & 0xFFFFu);
                };
                auto load = [&](Step2& f, int s) {
                    const int a = (s - q.steps) * kAnchorCols + 2 * t;
                    f.c0 = make_uint4(pair(awg, a), pair(awg8, a), pair(awg, a + 8), pair(awg8, a + 8));
                    f.c1 = make_uint4(pair(awg, a + 16), pair(awg8, a + 16), pair(awg, a + 24), pair(awg8, a + 24));
                    f.s0 = pair(awg, a + 32);
                    f.z0 = pair(awg8, a + 32);
                    f.s1 = pair(awg, a + 40);
                    f.z1 = pair(awg8, a + 40);
                };
                auto compute = [&](const Step2& f, int s) {
                    const uint16_t* xs = xab + (int64_t)(s - q.steps) * kAnchorCols * M;
                    uint2 xb[3][NT];
#pragma unroll
                    for (int kb = 0; kb < 3; ++kb)
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt) xb[kb][nt] = *reinterpret_cast<const uint2*>(xs + kb * M * 16 + tok[nt]);
                    mma_xg<NT, MT>(acc, f.c0.x, f.c0.y, f.c0.z, f.c0.w, xb[0]);
                    mma_xg<NT, MT>(acc, f.c1.x, f.c1.y, f.c1.z, f.c1.w, xb[1]);
                    mma_xg<NT, MT>(acc, f.s0, f.z0, f.s1, f.z1, xb[2]);
                };
                int s = anchor_begin;
                Step2 fa, fb;
                load(fa, s);
                for (;;) {
                    if (s + 1 < s_end) load(fb, s + 1);
                    compute(fa, s);
                    if (++s >= s_end) break;
                    if (s + 1 < s_end) load(fa, s + 1);
                    compute(fb, s);
                    if (++s >= s_end) break;
                }
            }
        } else {
            const uint8_t* cb = D.codes + q.l * D.stride_codes + 8 * t;
            const uint8_t* c0p = cb + r0 * (K / 2);
            const uint8_t* c1p = cb + r1 * (K / 2);
            // the rows' block maxima: fp32, or (double quantization) E4M3 codes, four blocks (one
            // 256-column step) per 32-bit word sharing one second-level scale (256 is a multiple of 4)
            const float* second = FMT == LQ_FMT_NF4_DQ
                                      ? reinterpret_cast<const float*>(reinterpret_cast<const char*>(D.offsets) + q.l * D.stride_offsets)
                                      : nullptr;
            const int mb = FMT == LQ_FMT_NF4_DQ ? 1 : 4;   // bytes per block maximum
            const char* am = static_cast<const char*>(D.scales) + q.l * D.stride_scales;
            const char* a0p = am + r0 * (K / 64) * mb;
            const char* a1p = am + r1 * (K / 64) * mb;
            uint32_t TL[4], TH[4];
            nf4_tables(TL, TH);
            auto load = [&](StepNF4& f, int s) {
#pragma unroll
                for (int nb = 0; nb < 4; ++nb) {
                    f.c0[nb] = ldg64(c0p + 128 * s + 32 * nb);
                    f.c1[nb] = ldg64(c1p + 128 * s + 32 * nb);
                }
                if (FMT == LQ_FMT_NF4_DQ) {
                    const uint32_t w0 = ldg32(a0p + 4 * s), w1 = ldg32(a1p + 4 * s);
                    const float s0 = __ldg(second + 1 + ((r0 * (K / 64) + 4 * s) >> 8));
                    const float s1 = __ldg(second + 1 + ((r1 * (K / 64) + 4 * s) >> 8));
                    const float mean = __ldg(second);
#pragma unroll
                    for (int nb = 0; nb < 4; ++nb) {
                        f.a0[nb] = __fmaf_rn(e4m3_to_float((w0 >> (8 * nb)) & 0xFFu), s0, mean);
                        f.a1[nb] = __fmaf_rn(e4m3_to_float((w1 >> (8 * nb)) & 0xFFu), s1, mean);
                    }
                } else {
#pragma unroll
                    for (int nb = 0; nb < 4; ++nb) {
                        f.a0[nb] = __ldg(reinterpret_cast<const float*>(a0p) + 4 * s + nb);
                        f.a1[nb] = __ldg(reinterpret_cast<const float*>(a1p) + 4 * s + nb);
                    }
                }
            };
            auto compute = [&](const StepNF4& f, int s) {
                const uint16_t* xs = xb0 + (int64_t)s * 256 * M;
#pragma unroll
                for (int nb = 0; nb < 4; ++nb) {
                    uint2 xb[4][NT];
#pragma unroll
                    for (int b = 0; b < 4; ++b)
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt) xb[b][nt] = *reinterpret_cast<const uint2*>(xs + (nb * 4 + b) * M * 16 + tok[nt]);
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
            };
            int s = q.s;
            StepNF4 fa, fb;
            load(fa, s);
            if (!STAGED && !waited) {
                pdl_wait();
                waited = true;
            }
            for (;;) {
                if (s + 1 < s_end) load(fb, s + 1);
                compute(fa, s);
                if (++s >= s_end) break;
                if (s + 1 < s_end) load(fa, s + 1);
                compute(fb, s);
                if (++s >= s_end) break;
            }
        }
        flush(q, n);
        u += n;
        if (u < u_end) {
            q.s = 0;
            next_block(P, q);
        }
    }
    if (peak >= kHalfOverflow && P.status) atomicOr(P.status, 2);
}

// ---- ring kernel (2-bit) ----------------------------------------------------------
//
// The same grouped launch, unit partition, x pre-pass and slot reduction as
// gemv_stream_kernel, reorganised around what bounds decode on this part: the integer
// pipe that turns codes into binary16 weights, and the instructions spent per unit.
//  * A unit is 32 output rows x 256 code columns (or 32 rows x 48 anchor columns): two
//    mma row tiles that share every x fragment, so one shared-memory x load feeds two
//    independent accumulator chains.
//  * Weights reach the registers through shared memory: each warp keeps kRingDepth unit
//    stages that its lanes fill with 16-byte cp.async copies (the next units are in flight
//    while one is multiplied; a stage is refilled as soon as it is consumed), so loads in
//    flight hold no registers.  One CTA of 16 warps per SM.
//  * x: when the span of x that a CTA's warps read fits in shared memory (XS), the CTA
//    builds it there itself (binary16, fragment order, anchor columns zeroed) and no
//    pre-pass runs; otherwise the pre-pass writes it to global memory once per call.
//  * Each CTA lets the next kernel in the stream launch at once (programmatic dependent
//    launch), so a following call's weight copies start while this call finishes; every
//    kernel waits for its predecessor before it reads x or touches the workspace or y.
//
// Stage layouts:
//   2-bit code unit (3072 B): codes [32 rows][64 B] | scales [32][8 x binary16] | offsets [32][8]
//   INT4 code unit (4608 B):  codes [32 rows][128 B] (16-byte chunk c of row r at chunk
//                             c ^ (r & 1), so the lanes of a quarter-warp hit distinct banks)
//                             | scales [32][8 x binary16]
//   anchor unit:              anchor weights [32 rows][48 x binary16] (zero past A)

__host__ __device__ constexpr int ring_stage(int FMT) { return FMT == LQ_FMT_INT4_G32 ? 4608 : 3072; }
// A problem with 1..16 anchors carries them in the last code unit of each row block (no
// anchor units): [32 rows][16 x binary16] after the stage's code part, zero past A.
constexpr int kFuseA = 16;
constexpr int kFuseBytes = 32 * kFuseA * 2;
#ifndef LQ_RING_DEPTH
#define LQ_RING_DEPTH 2
#endif
constexpr int kRingDepth = LQ_RING_DEPTH;
constexpr int kRingRows = 32;

#ifndef LQ_RING_WARPS1
#define LQ_RING_WARPS1 16
#endif
__host__ __device__ constexpr int ring_warps(int NT) { return NT == 1 ? LQ_RING_WARPS1 : 16; }

__device__ __forceinline__ void prefetch_l1(const void* p) { asm volatile("prefetch.global.L1 [%0];" ::"l"(p)); }

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint32_t src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

__device__ __forceinline__ uint32_t lds32(const unsigned char* p) { return *reinterpret_cast<const uint32_t*>(p); }

// Issue side of a warp's ring: the lane's source pointers for the next unit to copy and
// the cursor (problem, member, row block, unit) that moves them.  Inside a row block the
// pointers only advance; entering the next row block recomputes them (out of line).
// Order of a row block's units: its na anchor units sit at positions G-1, 2G-1, ..., naG-1
// (G = su / na) among the code units, so that any run of consecutive units holds code and
// anchor units in about the block's proportion and equal runs cost about the same.
struct UnitOrder {
    int a;    // anchor units before the cursor
    int ua;   // units from the cursor to the next anchor unit (large when none is left)
    int G, na;
};

__device__ __forceinline__ UnitOrder unit_order(int s, int steps, int su, int G) {
    UnitOrder o;
    o.na = su - steps;
    o.G = G;
    o.a = s == 0 ? 0 : min(o.na, s / G);
    o.ua = o.a < o.na ? (o.a + 1) * G - 1 - s : 1 << 30;
    return o;
}

// Is the cursor's unit an anchor unit; then step the cursor past it.
__device__ __forceinline__ bool unit_step(UnitOrder& o) {
    if (o.ua == 0) {
        ++o.a;
        o.ua = o.a < o.na ? o.G - 1 : 1 << 30;
        return true;
    }
    --o.ua;
    return false;
}

struct Feed {
    const uint8_t* c0;       // codes of row g at this lane's 16-byte slice of the next code unit
    const uint8_t* meta;     // lane < 16: scales of rows 2i, 2i+1 (i = lane & 15); else offsets
    const uint8_t* arow;     // anchor weights of row `lane`
    int o8, o16, o24;        // byte offsets from c0 to the codes of rows g+8, g+16, g+24
    int om;                  // byte offset from meta to the second row's metadata
    int s, su;               // next unit inside the row block; all units of a row block
    UnitOrder ord;           // where the anchor units of the row block fall
    int left;                // units of the warp's range not yet issued
    int A;                   // anchors of the problem
    int fast;                // following row blocks of this member that are full (pointers only advance)
    int fuse;                // the problem's anchors ride in each row block's last code unit
    int dc, dm, da;          // pointer steps from the end of a full row block to the next one
    int64_t u;               // launch-wide index of the next unit
};

// The feed cursor at unit u (left units remain in the warp's range).
template <int FMT>
__device__ __forceinline__ Feed feed_at(const FParams& P, int64_t u, int left, int lane) {
    constexpr int CB = FMT == LQ_FMT_INT4_G32 ? 2 : 4;   // codes per byte
    const Pos q = locate(P, u);
    Feed f;
    f.u = u;
    f.s = q.s;
    f.left = left;
    const FDesc& D = P.d[q.p];
    const int g = lane >> 2, t = lane & 3, N = D.N, K = D.K;
    const int base = q.rb * kRingRows;
    auto row = [&](int r) -> int64_t { return base + r < N ? base + r : N - 1; };   // rows past N: never stored
    f.ord = unit_order(q.s, D.steps, D.su, D.G);
    const int sc = q.s - f.ord.a;   // code units before unit s
    const int64_t rg = row(g);
    f.c0 = D.codes + q.l * D.stride_codes + rg * (K / CB) + (256 / CB / 4) * t + (256 / CB) * sc;
    f.o8 = (int)((row(g + 8) - rg) * (K / CB));
    f.o16 = (int)((row(g + 16) - rg) * (K / CB));
    f.o24 = (int)((row(g + 24) - rg) * (K / CB));
    if (FMT == LQ_FMT_INT4_G32) {   // scales of row `lane`
        f.meta = static_cast<const uint8_t*>(D.scales) + q.l * D.stride_scales + row(lane) * (K / 16) + 16 * sc;
        f.om = 0;
    } else {                        // lane < 16: scales of rows 2i, 2i+1; else their offsets
        const int i = lane & 15;
        const uint8_t* mb = lane < 16 ? static_cast<const uint8_t*>(D.scales) + q.l * D.stride_scales
                                      : reinterpret_cast<const uint8_t*>(D.offsets) + q.l * D.stride_offsets;
        const int64_t rm = row(2 * i);
        f.meta = mb + rm * (K / 16) + 16 * sc;
        f.om = (int)((row(2 * i + 1) - rm) * (K / 16));
    }
    f.su = D.su;
    f.A = D.A;
    f.fuse = D.fuse;
    const int full = N / kRingRows;   // row blocks with all 32 rows inside N
    f.fast = q.rb < full ? full - 1 - q.rb : 0;
    f.dc = (kRingRows - 1) * (K / CB);
    f.dm = (kRingRows - 1) * (K / 16);
    f.da = kRingRows * D.ld_anchor * 2;
    f.arow = D.A > 0 ? reinterpret_cast<const uint8_t*>(D.anchor_w) + q.l * D.stride_anchor_w + row(lane) * D.ld_anchor * 2
                     : D.codes;
    return f;
}

// Row `lane`'s anchors 0..15 (zero past A) to [dst + 32 lane, +32).
__device__ __forceinline__ void feed_fused_anchors(const Feed& f, uint32_t dst, int lane) {
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const int n = f.A - 8 * i;
        const uint32_t bytes = n >= 8 ? 16u : (n > 0 ? 2u * n : 0u);
        cp_async16(dst + lane * 32 + 16 * i, bytes ? f.arow + 16 * i : f.arow, bytes);
    }
}

// Copy the next unit into the stage at `st` and step the cursor; one commit group per call
// (empty once the warp's range is exhausted).
template <int FMT>
__device__ __forceinline__ void feed_issue(const FParams& P, Feed& f, uint32_t st, int lane) {
    if (f.left > 0) {
        const int g = lane >> 2, t = lane & 3;
        const int a_unit = f.ord.a;
        if (!unit_step(f.ord)) {
            if (FMT == LQ_FMT_INT4_G32) {
                // rows g + 8r: 32 bytes each (chunks 2t, 2t+1, swizzled by the row's parity)
                const uint32_t d0 = st + g * 128 + (((2 * t) ^ (g & 1)) << 4), d1 = st + g * 128 + (((2 * t + 1) ^ (g & 1)) << 4);
                const int off[4] = {0, f.o8, f.o16, f.o24};
#pragma unroll
                for (int r = 0; r < 4; ++r) {
                    cp_async16(d0 + r * 8 * 128, f.c0 + off[r], 16);
                    cp_async16(d1 + r * 8 * 128, f.c0 + off[r] + 16, 16);
                }
                cp_async16(st + 4096 + lane * 16, f.meta, 16);
                f.c0 += 128;
                f.meta += 16;
                if (f.fuse && f.s == f.su - 1) feed_fused_anchors(f, st + ring_stage(FMT), lane);
            } else {
                const uint32_t dc = st + g * 64 + 16 * t;
                cp_async16(dc, f.c0, 16);
                cp_async16(dc + 8 * 64, f.c0 + f.o8, 16);
                cp_async16(dc + 16 * 64, f.c0 + f.o16, 16);
                cp_async16(dc + 24 * 64, f.c0 + f.o24, 16);
                const uint32_t dm = st + 2048 + (lane >> 4) * 512 + (lane & 15) * 32;
                cp_async16(dm, f.meta, 16);
                cp_async16(dm + 16, f.meta + f.om, 16);
                f.c0 += 64;
                f.meta += 16;
                if (f.fuse && f.s == f.su - 1) feed_fused_anchors(f, st + ring_stage(FMT), lane);
            }
        } else {
            const int a0 = a_unit * kAnchorCols;
            const uint32_t dst = st + lane * 96;
            const int npieces = 2 * ((f.A - a0 + 15) >> 4);   // the k-blocks that hold anchors (the rest is not read)
#pragma unroll
            for (int i = 0; i < 6; ++i) {
                if (i > 0 && i >= npieces) break;
                const int a = a0 + 8 * i;
                const int n = f.A - a;   // anchors left from column a: copy at most 8, zero the rest
                const uint32_t bytes = n >= 8 ? 16u : (n > 0 ? 2u * n : 0u);
                cp_async16(dst + 16 * i, bytes ? f.arow + 2 * a : f.arow, bytes);
            }
        }
        --f.left;
        ++f.u;
        if (++f.s == f.su && f.left > 0) {
            if (f.fast > 0) {   // the next row block of the same member, all rows inside N
                --f.fast;
                f.s = 0;
                f.c0 += f.dc;
                f.meta += f.dm;
                f.arow += f.A > 0 ? f.da : 0;
                f.ord.a = 0;
                f.ord.ua = f.ord.na > 0 ? f.ord.G - 1 : 1 << 30;
            } else {
                f = feed_at<FMT>(P, f.u, f.left, lane);
            }
        }
    }
    cp_async_commit();
}

// Write a warp's sums of the row block at q (units: how many of the block's units it did)
// to y directly when it did them all, else to its slot; the warp completing the block adds
// the slots in warp order and writes y.
template <int NT>
__device__ __forceinline__ void ring_flush(const FParams& P, const Pos& q, int units, float (&acc)[2][NT][4], int M,
                                           int lane, const uint16_t* xmember) {
    const FDesc& D = P.d[q.p];
    const int g = lane >> 2, t = lane & 3;
    if (P.x_bf16) {   // remove each token's x scale
        const uint32_t* xmaxw = reinterpret_cast<const uint32_t*>(xmember + D.xsc_off);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                const int m = min(8 * nt + 2 * t + c, M - 1);
                const float u = x_unscale(xmaxw[m]);
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    acc[h][nt][c] *= u;
                    acc[h][nt][c + 2] *= u;
                }
            }
    }
    if (units == q.su) {
        void* y = static_cast<char*>(D.y) + q.l * D.stride_y;
        const int rg = q.rb * kRingRows + g;
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int m = 8 * nt + 2 * t + (e & 1), row = rg + 16 * h + (e >> 1) * 8;
                    if (m < M && row < D.N) store_out(y, (size_t)m * D.N + row, P.y_dtype, acc[h][nt][e]);
                    acc[h][nt][e] = 0.f;
                }
        return;
    }
    const int64_t wid = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    const int64_t u_begin = split_at(P, wid);
    const int64_t blk = q.l * D.rblocks + q.rb;
    const int64_t first_u = D.unit_begin + blk * q.su;
    const int64_t w0 = first_u >= u_begin ? wid : owner_of(P, first_u);
    float* slots = D.part + blk * D.cmax * M * kRingRows;
    float* mine = slots + (int)(wid - w0) * M * kRingRows;
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int m = 8 * nt + 2 * t + (e & 1), r = 16 * h + g + (e >> 1) * 8;
                if (m < M) __stcg(mine + m * kRingRows + r, acc[h][nt][e]);
                acc[h][nt][e] = 0.f;
            }
    __syncwarp();
    unsigned last = 0;
    if (lane == 0) {
        const unsigned old = atom_add_acq_rel_gpu(D.cnt + blk, (unsigned)units);
        last = old + (unsigned)units == (unsigned)q.su;
    }
    if (__shfl_sync(0xffffffffu, last, 0)) {
        __syncwarp();
        if (lane == 0) D.cnt[blk] = 0u;
        const int nc = (int)(owner_of(P, first_u + q.su - 1) - w0 + 1);
        finish_block(slots, nc, M, static_cast<char*>(D.y) + q.l * D.stride_y, D.N, q.rb * kRingRows, P.y_dtype,
                     lane, kRingRows);
    }
}

// The x span of a CTA (members a..b of the launch, a few at most) built in shared memory
// in the ring layout, with one CTA barrier after each pass:
// (0) every code column as binary16 (two 16-byte loads per 16 columns of a token);
// (1) x at the anchor columns (zero past A) taken from (0), and those columns of (0) zeroed
//     (the anchors replace those weights).
// bf16 x first takes each token's max |x| (passes -2: clear, -1: max), for its scale.
// INT4: x is taken through the permutation (position j holds x at column perm[j]) with
// INT4's order inside each block of 16, x at the anchor columns comes from the caller's x in
// pass (0), and no column is zeroed (an anchor position stores q = 0, which is exactly 0), so
// pass (1) is not needed.
template <int FMT>
__device__ __forceinline__ void build_span_x(const FParams& P, const Pos& a, const Pos& b, int64_t span0, uint16_t* xsm) {
    const int M = P.M, tid = threadIdx.x, nth = blockDim.x, S = ring_kstride(M);
    const int last_pass = FMT == LQ_FMT_INT4_G32 ? 0 : 1;
    for (int pass = P.x_bf16 ? -2 : 0; pass <= last_pass; ++pass) {
        for (int p = a.p; p <= b.p; ++p) {
            const FDesc& D = P.d[p];
            const int K = D.K, A = D.A;
            const int64_t l0 = p == a.p ? a.l : 0, l1 = p == b.p ? b.l : D.batch - 1;
            for (int64_t l = l0; l <= l1; ++l) {
                uint16_t* dst = xsm + (D.xoff + l * D.xperm_stride - span0);
                const int32_t* aidx = A > 0 ? reinterpret_cast<const int32_t*>(reinterpret_cast<const char*>(D.anchor_idx) +
                                                                                 l * D.stride_anchor_idx)
                                            : nullptr;
                const uint16_t* x = reinterpret_cast<const uint16_t*>(reinterpret_cast<const char*>(D.x) + l * D.stride_x);
                uint32_t* xmaxw = reinterpret_cast<uint32_t*>(dst + D.xsc_off);
                if (pass == -2) {
                    for (int m = tid; m < M; m += nth) xmaxw[m] = 0u;
                } else if (pass == -1) {
                    for (int it = tid; it < M * K / 16; it += nth) {
                        const int m = it / (K / 16), q = it - m * (K / 16);
                        const uint4* src = reinterpret_cast<const uint4*>(x + (int64_t)m * K + 16 * q);
                        const uint4 v0 = __ldg(src), v1 = __ldg(src + 1);
                        const uint32_t w[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
                        uint32_t mx = 0;
#pragma unroll
                        for (int i = 0; i < 8; ++i) mx = max(mx, max(w[i] & 0x7FFFu, (w[i] >> 16) & 0x7FFFu));
                        atomicMax(&xmaxw[m], mx << 16);
                    }
                } else if (pass == 0) {
                    if (FMT == LQ_FMT_INT4_G32) {
                        // x at the anchor columns (fragment order), straight from the caller's x
                        const int a_pad = D.a_pad;
                        uint16_t* xa = dst + D.xa_off;
                        for (int it = tid; it < M * a_pad; it += nth) {
                            const int m = it / a_pad, aa = it - m * a_pad;
                            const int k = aa < A ? __ldg(aidx + aa) : -1;
                            const int bi = aa >> 4, r = aa & 15, pos = 4 * ((r & 7) >> 1) + (r & 1) + 2 * (r >> 3);
                            xa[(bi * M + m) * 16 + pos] =
                                (unsigned)k < (unsigned)K ? to_half_scaled(x[(int64_t)m * K + k], P.x_bf16, P.x_bf16 ? x_scale(xmaxw[m]) : 1.f)
                                                          : (uint16_t)0;
                        }
                    } else {
                        // the anchor columns are read in pass 1: bring them into L1 now
                        for (int i = tid * 32; i < A; i += nth * 32) prefetch_l1(aidx + i);
                    }
                    if (FMT == LQ_FMT_INT4_G32) {
                        const int32_t* perm = reinterpret_cast<const int32_t*>(reinterpret_cast<const char*>(D.perm) + l * D.stride_perm);
                        for (int it = tid; it < M * K / 16; it += nth) {
                            const int m = it / (K / 16), q = it - m * (K / 16);
                            const float sc = P.x_bf16 ? x_scale(xmaxw[m]) : 1.f;
                            const int4* pp = reinterpret_cast<const int4*>(perm + 16 * q);
                            int cols[16];
#pragma unroll
                            for (int i = 0; i < 4; ++i) {
                                const int4 c4 = __ldg(pp + i);
                                cols[4 * i] = c4.x;
                                cols[4 * i + 1] = c4.y;
                                cols[4 * i + 2] = c4.z;
                                cols[4 * i + 3] = c4.w;
                            }
                            uint16_t v[16];
#pragma unroll
                            for (int r = 0; r < 16; ++r) {
                                const int c = cols[r];
                                const uint16_t raw = (unsigned)c < (unsigned)K ? x[(int64_t)m * K + c] : (uint16_t)0;
                                v[int4_block_pos(r)] = to_half_scaled(raw, P.x_bf16, sc);
                            }
                            uint2* d2 = reinterpret_cast<uint2*>(dst + q * S + m * 16);
#pragma unroll
                            for (int i = 0; i < 4; ++i)
                                d2[i] = make_uint2((uint32_t)v[4 * i] | ((uint32_t)v[4 * i + 1] << 16),
                                                   (uint32_t)v[4 * i + 2] | ((uint32_t)v[4 * i + 3] << 16));
                        }
                    } else {
                        for (int it = tid; it < M * K / 16; it += nth) {
                            const int m = it / (K / 16), q = it - m * (K / 16);
                            const uint4* src = reinterpret_cast<const uint4*>(x + (int64_t)m * K + 16 * q);
                            const uint4 v0 = __ldg(src), v1 = __ldg(src + 1);
                            uint32_t w[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w}, o[8];
                            if (P.x_bf16) {
                                const float sc = x_scale(xmaxw[m]);
#pragma unroll
                                for (int i = 0; i < 8; ++i)
                                    w[i] = (uint32_t)bf16_to_half_scaled((uint16_t)w[i], sc) |
                                           ((uint32_t)bf16_to_half_scaled((uint16_t)(w[i] >> 16), sc) << 16);
                            }
                            ring_x_transpose(w, o);
                            uint4* d4 = reinterpret_cast<uint4*>(dst + q * S + m * 16);
                            d4[0] = make_uint4(o[0], o[1], o[2], o[3]);
                            d4[1] = make_uint4(o[4], o[5], o[6], o[7]);
                        }
                    }
                } else if (FMT != LQ_FMT_INT4_G32) {
                    // x at the anchor columns (fragment order, zero past A) taken from pass 0's copy,
                    // then those columns of the copy zeroed (the item that reads a column zeroes it)
                    const int a_pad = D.a_pad;
                    uint16_t* xa = dst + D.xa_off;
                    for (int it = tid; it < M * a_pad; it += nth) {
                        const int m = it / a_pad, aa = it - m * a_pad;
                        const int k = aa < A ? __ldg(aidx + aa) : -1;
                        const int bi = aa >> 4, r = aa & 15, pos = 4 * ((r & 7) >> 1) + (r & 1) + 2 * (r >> 3);
                        uint16_t v = 0;
                        if ((unsigned)k < (unsigned)K) {   // (a column outside [0, K) is ignored)
                            uint16_t& c = dst[ring_x_pos(k, m, M)];
                            v = c;
                            c = 0;
                        }
                        xa[(bi * M + m) * 16 + pos] = v;
                    }
                }
            }
        }
        __syncthreads();
    }
}

// binary16 half h (0: low, 1: high) of a 32-bit word, as fp32
__device__ __forceinline__ float half_of(uint32_t v, int h) {
    return half_bits_to_float(h == 0 ? (uint16_t)(v & 0xFFFFu) : (uint16_t)(v >> 16));
}

// One 16-column block of x for the n-tiles of a lane: with one n-tile, two 16-byte loads
// cover the block's four mma steps (j = 0..3, 4 halves each); with more, each step loads
// its 8 bytes when used (fewer live registers).
template <int NT>
struct XBlock {
    uint4 v[2];
    __device__ __forceinline__ void load(const uint16_t* blk, const int (&tok)[NT]) {
        if (NT == 1) {
            v[0] = *reinterpret_cast<const uint4*>(blk + tok[0]);
            v[1] = *reinterpret_cast<const uint4*>(blk + 8 + tok[0]);
        }
    }
    __device__ __forceinline__ void get(int j, const uint16_t* blk, const int (&tok)[NT], uint2 (&xb)[NT]) const {
        if (NT == 1) {
            const uint4& u = v[j >> 1];
            xb[0] = (j & 1) ? make_uint2(u.z, u.w) : make_uint2(u.x, u.y);
        } else {
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) xb[nt] = *reinterpret_cast<const uint2*>(blk + 4 * j + tok[nt]);
        }
    }
};

// INT4: two codes of a word (nibbles k and k+4, the word XORed with 0x88888888 so each
// nibble is q + 8) -> binary16 pair (S q_k, S q_{k+4}): OR into 1024's bit pattern gives
// 1032 + q exactly, subtracting 1032 gives q, and one product by the group's scale rounds
// once.  (Integer ops on the ALU pipe, half-precision ops on the FMA pipe.)
__device__ __forceinline__ uint32_t int4_pair(uint32_t wx, int k, uint32_t s2) {
    const uint32_t v = ((k == 0 ? wx : (wx >> (4 * k))) & 0x000F000Fu) | 0x64006400u;
    uint32_t d;
    asm("{\n\t.reg .b32 t;\n\tsub.rn.f16x2 t, %1, %2;\n\tmul.rn.f16x2 %0, t, %3;\n\t}"
        : "=r"(d) : "r"(v), "r"(0x64086408u), "r"(s2));
    return d;
}

template <int FMT, int MT, int NT, bool XS>
__global__ void __launch_bounds__(32 * ring_warps(NT), 16 / ring_warps(NT)) gemv_ring_kernel(const __grid_constant__ FParams P) {
    constexpr int kW = ring_warps(NT);
    const int kStage = P.stage;
    extern __shared__ __align__(128) unsigned char ring_smem[];
    const int M = MT > 0 ? MT : P.M;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
    const int64_t W = P.total_warps;
    const int64_t wid = (int64_t)blockIdx.x * kW + warp;
    const bool active = wid < W;
    if (!XS && !active) return;
    const uint32_t ring = smem_u32(ring_smem) + warp * kRingDepth * kStage;
    const unsigned char* ringp = ring_smem + warp * kRingDepth * kStage;
    const int64_t u_begin = active ? split_at(P, wid) : 0, u_end = active ? split_at(P, wid + 1) : 0;

    // Weights do not depend on the kernel before: the first unit's copies go out before
    // waiting for it, after the cheap lookups (the warp's cursor, the CTA's x span) and before
    // the x build; the second unit's copies go out after the build, so that the build's loads
    // do not queue behind both.
    Feed f;
    if (active) f = feed_at<FMT>(P, u_begin, (int)(u_end - u_begin), lane);
    int64_t span0 = 0;
    uint16_t* xsm = reinterpret_cast<uint16_t*>(ring_smem + kW * kRingDepth * kStage);
    Pos a, b;
    const int64_t w_lo = (int64_t)blockIdx.x * kW, w_hi = (w_lo + kW < W) ? w_lo + kW : W;
    if (XS) {
        if (w_lo >= W) return;   // the whole CTA is idle
        a = locate(P, split_at(P, w_lo));
        b = locate(P, split_at(P, w_hi) - 1);
        span0 = P.d[a.p].xoff + a.l * P.d[a.p].xperm_stride;
    }
    if (active) feed_issue<FMT>(P, f, ring, lane);
    pdl_launch_dependents();
    if (XS) {
        pdl_wait();   // x may come from the kernel before
        build_span_x<FMT>(P, a, b, span0, xsm);
        if (!active) return;
    } else {
        pdl_wait();
    }
#pragma unroll
    for (int i = 1; i < kRingDepth; ++i) feed_issue<FMT>(P, f, ring + i * kStage, lane);

    const int S = ring_kstride(M);
    const int xlane = min(g, M - 1) * 16 + 4 * t * S;    // code columns: block 4t of each 64-column quarter
    const int xlane_a = min(g, M - 1) * 16 + t * 4;      // anchor columns (fragment order)
    int tok[NT];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) tok[nt] = (min(8 * nt + g, M - 1) - min(g, M - 1)) * 16;
    float acc[2][NT][4];
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) acc[h][nt][0] = acc[h][nt][1] = acc[h][nt][2] = acc[h][nt][3] = 0.f;

    auto xbase = [&](const Pos& c) -> const uint16_t* {
        const FDesc& D = P.d[c.p];
        return XS ? xsm + (D.xoff + c.l * D.xperm_stride - span0) : D.xperm + c.l * D.xperm_stride;
    };
    Pos q = locate(P, u_begin);
    UnitOrder ord = unit_order(q.s, q.steps, q.su, P.d[q.p].G);
    int fuse_blk = P.d[q.p].fuse;
    const uint16_t* xb0 = xbase(q);
    int seg_units = 0;
    float peak = 0.f;   // largest |weight table value| seen (binary16 range check)
    uint32_t cst = 0;   // byte offset of the stage to compute (the others are being filled)
    for (int left = (int)(u_end - u_begin); left > 0; --left) {
        cp_async_wait<kRingDepth - 1>();
        __syncwarp();   // every lane's copies of this unit have landed (the next units may still be in flight)
        const unsigned char* st = ringp + cst;
        const int a_unit = ord.a;
        const bool anchor_unit = unit_step(ord);
        if (FMT == LQ_FMT_INT4_G32 && !anchor_unit) {
            const uint16_t* xs = xb0 + xlane + (q.s - a_unit) * 16 * S;
#pragma unroll
            for (int h = 0; h < 2; ++h) {   // group 2t + h: 32 columns = words 4h .. 4h+3 of the lane's slice
                uint32_t s2[4];
                uint4 w[4];
#pragma unroll
                for (int r = 0; r < 4; ++r) {
                    const uint16_t sb = *reinterpret_cast<const uint16_t*>(st + 4096 + (g + 8 * r) * 16 + 4 * t + 2 * h);
                    s2[r] = (uint32_t)sb | ((uint32_t)sb << 16);
                    peak = fmaxf(peak, 8.f * fabsf(half_bits_to_float(sb)));   // |S q| for the widest code
                    w[r] = *reinterpret_cast<const uint4*>(st + (g + 8 * r) * 128 + (((2 * t + h) ^ (g & 1)) << 4));
                    w[r].x ^= 0x88888888u;
                    w[r].y ^= 0x88888888u;
                    w[r].z ^= 0x88888888u;
                    w[r].w ^= 0x88888888u;
                }
                XBlock<NT> xk;
#pragma unroll
                for (int i = 0; i < 4; ++i) {   // word 4h + i: block 2h + i/2, half i & 1 of it
                    if ((i & 1) == 0) xk.load(xs + (2 * h + (i >> 1)) * S, tok);
#pragma unroll
                    for (int kk = 0; kk < 2; ++kk) {
                        uint2 xb[NT];
                        xk.get(2 * (i & 1) + kk, xs + (2 * h + (i >> 1)) * S, tok, xb);
                        uint32_t wd[4];
#pragma unroll
                        for (int r = 0; r < 4; ++r) wd[r] = i == 0 ? w[r].x : (i == 1 ? w[r].y : (i == 2 ? w[r].z : w[r].w));
                        const uint32_t a0 = int4_pair(wd[0], 2 * kk, s2[0]), a2 = int4_pair(wd[0], 2 * kk + 1, s2[0]);
                        const uint32_t a1 = int4_pair(wd[1], 2 * kk, s2[1]), a3 = int4_pair(wd[1], 2 * kk + 1, s2[1]);
                        mma_xg<NT, MT>(acc[0], a0, a1, a2, a3, xb);
                        const uint32_t b0 = int4_pair(wd[2], 2 * kk, s2[2]), b2 = int4_pair(wd[2], 2 * kk + 1, s2[2]);
                        const uint32_t b1 = int4_pair(wd[3], 2 * kk, s2[3]), b3 = int4_pair(wd[3], 2 * kk + 1, s2[3]);
                        mma_xg<NT, MT>(acc[1], b0, b1, b2, b3, xb);
                    }
                }
            }
        } else if (FMT != LQ_FMT_INT4_G32 && !anchor_unit) {
            const uint16_t* xs = xb0 + xlane + (q.s - a_unit) * 16 * S;
            uint32_t sp[4], zp[4];   // row g + 8r: binary16 S (Z) of groups 2t (low half) and 2t+1
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                sp[r] = lds32(st + 2048 + (g + 8 * r) * 16 + 4 * t);
                zp[r] = lds32(st + 2560 + (g + 8 * r) * 16 + 4 * t);
            }
#pragma unroll
            for (int hg = 0; hg < 2; ++hg) {   // group 2t + hg: code words 2hg, 2hg+1 of each row
                uint32_t RA[4], RB[4];
                uint2 w[4];
#pragma unroll
                for (int rp = 0; rp < 4; rp += 2)   // rows g + 8rp and g + 8rp + 8 share the table arithmetic
                    lut2_bits_x2(make_float2(half_of(sp[rp], hg), half_of(sp[rp + 1], hg)),
                                 make_float2(half_of(zp[rp], hg), half_of(zp[rp + 1], hg)), RA[rp], RB[rp], RA[rp + 1],
                                 RB[rp + 1], peak);
#pragma unroll
                for (int r = 0; r < 4; ++r) w[r] = *reinterpret_cast<const uint2*>(st + (g + 8 * r) * 64 + 16 * t + 8 * hg);
#pragma unroll
                for (int iw = 0; iw < 2; ++iw) {
                    const int ii = 2 * hg + iw;
                    XBlock<NT> xk;
                    xk.load(xs + ii * S, tok);
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        uint2 xb[NT];
                        xk.get(j, xs + ii * S, tok, xb);
                        uint32_t a0, a1, a2, a3, b0, b1, b2, b3;
                        const uint32_t w0 = iw ? w[0].y : w[0].x, w1 = iw ? w[1].y : w[1].x;
                        const uint32_t w2 = iw ? w[2].y : w[2].x, w3 = iw ? w[3].y : w[3].x;
                        expand2_fast(w0, j, RA[0], RB[0], a0, a2);
                        expand2_fast(w1, j, RA[1], RB[1], a1, a3);
                        mma_xg<NT, MT>(acc[0], a0, a1, a2, a3, xb);
                        expand2_fast(w2, j, RA[2], RB[2], b0, b2);
                        expand2_fast(w3, j, RA[3], RB[3], b1, b3);
                        mma_xg<NT, MT>(acc[1], b0, b1, b2, b3, xb);
                    }
                }
            }
        } else {
            const uint16_t* xs = xb0 + xlane_a + P.d[q.p].xa_off + M * a_unit * kAnchorCols;
            const int nkb = (P.d[q.p].A - a_unit * kAnchorCols + 15) >> 4;   // k-blocks of this unit that hold anchors
#pragma unroll
            for (int kb = 0; kb < 3; ++kb) {
                if (kb > 0 && kb >= nkb) break;
                uint2 xb[NT];
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) xb[nt] = *reinterpret_cast<const uint2*>(xs + kb * M * 16 + tok[nt]);
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const unsigned char* r0p = st + (16 * h + g) * 96 + 32 * kb + 4 * t;
                    mma_xg<NT, MT>(acc[h], lds32(r0p), lds32(r0p + 8 * 96), lds32(r0p + 16), lds32(r0p + 8 * 96 + 16), xb);
                }
            }
        }
        if (fuse_blk && !anchor_unit && q.s == q.su - 1) {   // the row block's anchors, in its last code unit
            const uint16_t* xs = xb0 + xlane_a + P.d[q.p].xa_off;
            uint2 xb[NT];
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) xb[nt] = *reinterpret_cast<const uint2*>(xs + tok[nt]);
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const unsigned char* r0p = st + ring_stage(FMT) + (16 * h + g) * 32 + 4 * t;
                mma_xg<NT, MT>(acc[h], lds32(r0p), lds32(r0p + 8 * 32), lds32(r0p + 16), lds32(r0p + 8 * 32 + 16), xb);
            }
        }
        __syncwarp();   // every lane is done with this stage: refill it kRingDepth units ahead
        feed_issue<FMT>(P, f, ring + cst, lane);
        cst = cst + kStage == kRingDepth * kStage ? 0 : cst + kStage;
        ++seg_units;
        if (++q.s == q.su || left == 1) {
            ring_flush<NT>(P, q, seg_units, acc, M, lane, xb0);
            seg_units = 0;
            if (left > 1) {
                q.s = 0;
                const int p0 = q.p;
                const int64_t l0 = q.l;
                next_block(P, q);
                ord = unit_order(0, q.steps, q.su, P.d[q.p].G);
                fuse_blk = P.d[q.p].fuse;
                if (q.p != p0 || q.l != l0) xb0 = xbase(q);
            }
        }
    }
    cp_async_wait<0>();
    if (peak >= kHalfOverflow && P.status) atomicOr(P.status, 2);
}

// Resident CTAs per SM of a kernel at a given dynamic shared-memory size; the answer is cached
// per kernel (the lock keeps host threads that launch different sizes from racing on the cache).
// The kernel's shared-memory attribute only ever rises, to the largest size asked for, so that a
// launch planned earlier for a larger size (and kept in the plan cache) stays valid.
std::mutex g_occ_mutex;

template <typename Kern>
int resident_ctas_of(Kern kern, size_t smem, size_t& set_smem, int& per_sm, int threads = kThreadsS) {
    std::lock_guard<std::mutex> lock(g_occ_mutex);
    if (set_smem != smem) {
        static std::vector<std::pair<const void*, size_t>> attr;   // (kernel, attribute set)
        size_t* cur = nullptr;
        for (auto& e : attr)
            if (e.first == reinterpret_cast<const void*>(kern)) cur = &e.second;
        if (!cur) {
            attr.push_back({reinterpret_cast<const void*>(kern), 0});
            cur = &attr.back().second;
        }
        if (smem > *cur) {
            if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
                return -1;
            *cur = smem;
        }
        int n = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, threads, smem) != cudaSuccess) return -1;
        per_sm = n;
        set_smem = smem;
    }
    return per_sm;
}

template <int FMT, int MT, int NT, bool STAGED>
int resident_ctas(size_t smem) {
    static size_t set_smem = (size_t)-1;
    static int per_sm = 0;
    return resident_ctas_of(gemv_stream_kernel<FMT, MT, NT, STAGED>, smem, set_smem, per_sm);
}

template <int FMT, int MT, int NT, bool XS>
int resident_ctas_ring(size_t smem) {
    static size_t set_smem = (size_t)-1;
    static int per_sm = 0;
    return resident_ctas_of(gemv_ring_kernel<FMT, MT, NT, XS>, smem, set_smem, per_sm, 32 * ring_warps(NT));
}

template <int FMT, int MT, int NT, bool STAGED>
lq_status launch_one(const FParams& P, int64_t grid, size_t smem, cudaStream_t stream) {
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
    if (cudaLaunchKernelEx(&cfg, gemv_stream_kernel<FMT, MT, NT, STAGED>, P) != cudaSuccess) return LQ_ERR_CUDA;
    return cudaPeekAtLastError() == cudaSuccess ? LQ_OK : LQ_ERR_CUDA;
}

// mode 0: occupancy query (returns CTAs per SM through *per_sm); mode 1: launch
template <int FMT, int MT, int NT>
lq_status dispatch_mt(int mode, bool staged, const FParams& P, int64_t grid, size_t smem, int* per_sm, cudaStream_t stream) {
    if (mode == 0) {
        *per_sm = staged ? resident_ctas<FMT, MT, NT, true>(smem) : resident_ctas<FMT, MT, NT, false>(smem);
        return *per_sm < 0 ? LQ_ERR_CUDA : LQ_OK;
    }
    return staged ? launch_one<FMT, MT, NT, true>(P, grid, smem, stream) : launch_one<FMT, MT, NT, false>(P, grid, smem, stream);
}

template <int FMT>
lq_status dispatch_fmt(int mode, bool staged, const FParams& P, int64_t grid, size_t smem, int* per_sm, cudaStream_t stream) {
    switch (P.M) {
        case 1: return dispatch_mt<FMT, 1, 1>(mode, staged, P, grid, smem, per_sm, stream);
        case 2: return dispatch_mt<FMT, 2, 1>(mode, staged, P, grid, smem, per_sm, stream);
        case 3: return dispatch_mt<FMT, 3, 1>(mode, staged, P, grid, smem, per_sm, stream);
        case 4: return dispatch_mt<FMT, 4, 1>(mode, staged, P, grid, smem, per_sm, stream);
        case 5: return dispatch_mt<FMT, 5, 1>(mode, staged, P, grid, smem, per_sm, stream);
        case 6: return dispatch_mt<FMT, 6, 1>(mode, staged, P, grid, smem, per_sm, stream);
        case 7: return dispatch_mt<FMT, 7, 1>(mode, staged, P, grid, smem, per_sm, stream);
        case 8: return dispatch_mt<FMT, 8, 1>(mode, staged, P, grid, smem, per_sm, stream);
        default:
            if (P.M <= 16) return dispatch_mt<FMT, 0, 2>(mode, staged, P, grid, smem, per_sm, stream);
            if (P.M <= 24) return dispatch_mt<FMT, 0, 3>(mode, staged, P, grid, smem, per_sm, stream);
            if (P.M <= 32) return dispatch_mt<FMT, 0, 4>(mode, staged, P, grid, smem, per_sm, stream);
            return LQ_ERR_UNSUPPORTED;
    }
}

template <int FMT, int MT, int NT, bool XS>
lq_status ring_launch(int mode, const FParams& P, int64_t grid, size_t smem, int* per_sm, cudaStream_t stream) {
    if (mode == 0) {
        *per_sm = resident_ctas_ring<FMT, MT, NT, XS>(smem);
        return *per_sm < 0 ? LQ_ERR_CUDA : LQ_OK;
    }
    cudaLaunchConfig_t cfg;
    memset(&cfg, 0, sizeof(cfg));
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(32 * ring_warps(NT));
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, gemv_ring_kernel<FMT, MT, NT, XS>, P) != cudaSuccess) return LQ_ERR_CUDA;
    return cudaPeekAtLastError() == cudaSuccess ? LQ_OK : LQ_ERR_CUDA;
}

template <int FMT, int MT, int NT>
lq_status ring_mt(int mode, bool xs, const FParams& P, int64_t grid, size_t smem, int* per_sm, cudaStream_t stream) {
    return xs ? ring_launch<FMT, MT, NT, true>(mode, P, grid, smem, per_sm, stream)
              : ring_launch<FMT, MT, NT, false>(mode, P, grid, smem, per_sm, stream);
}

lq_status dispatch_ring(int mode, bool xs, const FParams& P, int64_t grid, size_t smem, int* per_sm,
                        cudaStream_t stream) {
    if (P.format == LQ_FMT_INT4_G32) {   // (one token at compile time; 2..8 tokens share one instantiation)
        if (P.M == 1) return ring_mt<LQ_FMT_INT4_G32, 1, 1>(mode, xs, P, grid, smem, per_sm, stream);
        if (P.M <= 8) return ring_mt<LQ_FMT_INT4_G32, 0, 1>(mode, xs, P, grid, smem, per_sm, stream);
        if (P.M <= 16) return ring_mt<LQ_FMT_INT4_G32, 0, 2>(mode, xs, P, grid, smem, per_sm, stream);
        if (P.M <= 24) return ring_mt<LQ_FMT_INT4_G32, 0, 3>(mode, xs, P, grid, smem, per_sm, stream);
        if (P.M <= 32) return ring_mt<LQ_FMT_INT4_G32, 0, 4>(mode, xs, P, grid, smem, per_sm, stream);
        return LQ_ERR_UNSUPPORTED;
    }
    switch (P.M) {
        case 1: return ring_mt<LQ_FMT_2BIT_LM_G32, 1, 1>(mode, xs, P, grid, smem, per_sm, stream);
        case 2: return ring_mt<LQ_FMT_2BIT_LM_G32, 2, 1>(mode, xs, P, grid, smem, per_sm, stream);
        case 3: return ring_mt<LQ_FMT_2BIT_LM_G32, 3, 1>(mode, xs, P, grid, smem, per_sm, stream);
        case 4: return ring_mt<LQ_FMT_2BIT_LM_G32, 4, 1>(mode, xs, P, grid, smem, per_sm, stream);
        case 5: return ring_mt<LQ_FMT_2BIT_LM_G32, 5, 1>(mode, xs, P, grid, smem, per_sm, stream);
        case 6: return ring_mt<LQ_FMT_2BIT_LM_G32, 6, 1>(mode, xs, P, grid, smem, per_sm, stream);
        case 7: return ring_mt<LQ_FMT_2BIT_LM_G32, 7, 1>(mode, xs, P, grid, smem, per_sm, stream);
        case 8: return ring_mt<LQ_FMT_2BIT_LM_G32, 8, 1>(mode, xs, P, grid, smem, per_sm, stream);
        default:
            if (P.M <= 16) return ring_mt<LQ_FMT_2BIT_LM_G32, 0, 2>(mode, xs, P, grid, smem, per_sm, stream);
            if (P.M <= 24) return ring_mt<LQ_FMT_2BIT_LM_G32, 0, 3>(mode, xs, P, grid, smem, per_sm, stream);
            if (P.M <= 32) return ring_mt<LQ_FMT_2BIT_LM_G32, 0, 4>(mode, xs, P, grid, smem, per_sm, stream);
            return LQ_ERR_UNSUPPORTED;
    }
}

lq_status dispatch(int fmt, int mode, bool staged, const FParams& P, int64_t grid, size_t smem, int* per_sm,
                   cudaStream_t stream) {
    if (fmt == LQ_FMT_NF4_DQ) {   // (fewer instantiations: one token at compile time, the rest by n-tiles)
        if (P.M == 1) return dispatch_mt<LQ_FMT_NF4_DQ, 1, 1>(mode, staged, P, grid, smem, per_sm, stream);
        if (P.M <= 8) return dispatch_mt<LQ_FMT_NF4_DQ, 0, 1>(mode, staged, P, grid, smem, per_sm, stream);
        if (P.M <= 16) return dispatch_mt<LQ_FMT_NF4_DQ, 0, 2>(mode, staged, P, grid, smem, per_sm, stream);
        if (P.M <= 24) return dispatch_mt<LQ_FMT_NF4_DQ, 0, 3>(mode, staged, P, grid, smem, per_sm, stream);
        if (P.M <= 32) return dispatch_mt<LQ_FMT_NF4_DQ, 0, 4>(mode, staged, P, grid, smem, per_sm, stream);
        return LQ_ERR_UNSUPPORTED;
    }
    return fmt == LQ_FMT_2BIT_LM_G32 ? dispatch_fmt<LQ_FMT_2BIT_LM_G32>(mode, staged, P, grid, smem, per_sm, stream)
                                     : dispatch_fmt<LQ_FMT_NF4_B64>(mode, staged, P, grid, smem, per_sm, stream);
}

// Host copy of the kernel's unit lookup (problem and member of unit u).
void host_locate(const FParams& P, int64_t u, int& p, int64_t& l) {
    p = 0;
    while (p + 1 < P.count && u >= P.d[p + 1].unit_begin) ++p;
    const FDesc& D = P.d[p];
    l = (u - D.unit_begin) / ((int64_t)D.rblocks * D.su);
}

int round_up(int a, int b) { return (a + b - 1) / b * b; }

size_t align256(size_t b) { return (b + 255) & ~size_t(255); }

}  // namespace

lq_status launch_xmax_rows(const lq_problem* probs, int count, uint32_t* words, cudaStream_t stream) {
    PrepParams Q;
    memset(&Q, 0, sizeof(Q));
    const int M = probs[0].M;
    Q.count = count;
    Q.M = M;
    Q.x_bf16 = 1;
    int64_t rows = 0;
    for (int i = 0; i < count; ++i) {
        PrepDesc& e = Q.d[i];
        e.x = static_cast<const uint16_t*>(probs[i].x);
        e.stride_x = probs[i].stride_x;
        e.K = probs[i].K;
        e.batch = probs[i].batch;
        e.xperm = reinterpret_cast<uint16_t*>(words + rows);   // member l's words at 2 * M * l halves
        e.xperm_stride = 2 * M;
        e.xsc_off = 0;
        e.row_begin = rows;
        rows += (int64_t)probs[i].batch * M;
    }
    Q.total_rows = rows;
    if (rows == 0) return LQ_OK;
    if (rows > 0x7fffffffLL) return LQ_ERR_UNSUPPORTED;
    xmax_kernel<<<(unsigned)rows, 256, 0, stream>>>(Q);
    return cudaPeekAtLastError() == cudaSuccess ? LQ_OK : LQ_ERR_CUDA;
}

bool gemv_stream_eligible(const lq_problem* probs, int count) {
    if (probs[0].M > 32) return false;
    for (int i = 0; i < count; ++i)
        if (probs[i].K % 256 != 0) return false;
    return true;
}

// The launch description of one grouped call: descriptors, grid, kernel variant, shared memory
// and the workspace regions.  units == 0: nothing to launch.
struct GemvPlan {
    FParams P;
    PrepParams Q;
    bool use_ring = false, ring_xs = false, staged = false;
    int64_t grid = 0, jobs = 0, rows = 0, units = 0, blocks = 0;
    size_t smem = 0;   // dynamic shared memory of the kernel variant that runs
};

lq_status plan_gemv(const GemvWorkspace& ws, const lq_problem* probs, int count, GemvPlan& G, cudaStream_t stream) {
    FParams& P = G.P;
    PrepParams& Q = G.Q;
    memset(&P, 0, sizeof(P));
    memset(&Q, 0, sizeof(Q));
    const int M = probs[0].M;
    const int fmt = probs[0].format;
    P.count = Q.count = count;
    P.M = Q.M = M;
    P.y_dtype = probs[0].y_dtype;
    P.format = Q.format = fmt;
    P.x_bf16 = Q.x_bf16 = probs[0].x_dtype == LQ_BF16;
    // 2-bit launches of up to eight tokens run the ring kernel (measured faster there); NF4
    // and more tokens run the register-fed one.  LQ_GEMV_KERNEL=stream / ring forces either
    // for 2-bit (comparisons and tests).
    const char* kern_env = getenv("LQ_GEMV_KERNEL");
    const bool use_ring = fmt == LQ_FMT_INT4_G32 ||   // (INT4 decodes on the ring kernel only)
                          (fmt == LQ_FMT_2BIT_LM_G32 && (M <= 8 || (kern_env && strcmp(kern_env, "ring") == 0)) &&
                           !(kern_env && strcmp(kern_env, "stream") == 0));
    const int rows_blk = use_ring ? kRingRows : 16;            // output rows per row block
    const int cta_warps = use_ring ? ring_warps(M <= 8 ? 1 : 2) : kWarps;

    int64_t units = 0, jobs = 0, xhalves = 0, blocks = 0, rows = 0;
    int any_fuse = 0;
    int max_k = 0;
    for (int i = 0; i < count; ++i) {
        const lq_problem& q = probs[i];
        const int A = fmt == LQ_FMT_2BIT_LM_G32 || fmt == LQ_FMT_INT4_G32 ? q.A : 0;
        FDesc& d = P.d[i];
        PrepDesc& e = Q.d[i];
        d.codes = q.codes;
        d.scales = q.scales;
        d.offsets = fmt == LQ_FMT_2BIT_LM_G32 || fmt == LQ_FMT_NF4_DQ ? static_cast<const uint16_t*>(q.offsets) : nullptr;
        d.perm = e.perm = fmt == LQ_FMT_INT4_G32 ? static_cast<const int32_t*>(q.offsets) : nullptr;
        d.stride_perm = e.stride_perm = q.stride_offsets;
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
        d.x = static_cast<const uint16_t*>(q.x);
        d.stride_x = q.stride_x;
        d.anchor_idx = A > 0 ? q.anchor_idx : nullptr;
        d.stride_anchor_idx = q.stride_anchor_idx;
        const int a_pad = A > 0 ? round_up(A, kAnchorCols) : 0;
        d.steps = q.K / 256;
        d.fuse = use_ring && A > 0 && A <= kFuseA ? 1 : 0;
        any_fuse |= d.fuse;
        d.su = d.steps + (d.fuse ? 0 : a_pad / kAnchorCols);
        d.G = d.su > d.steps ? d.su / (d.su - d.steps) : d.su + 1;
        d.rblocks = (q.N + rows_blk - 1) / rows_blk;
        d.unit_begin = P.unit_begin[i] = units;
        units += (int64_t)q.batch * d.rblocks * d.su;
        blocks += (int64_t)q.batch * d.rblocks;
        // per member: [x (fragment order, or the ring layout) | x at the anchors (M*a_pad)]
        d.xa_off = use_ring ? (q.K / 16) * ring_kstride(M) : M * q.K;
        d.xsc_off = d.xa_off + M * a_pad;   // then one 32-bit max |x| word per token (16-half aligned)
        d.a_pad = a_pad;
        d.xperm_stride = d.xaperm_stride = (int64_t)d.xsc_off + round_up(2 * M, 16);
        d.xoff = xhalves;
        xhalves += (int64_t)q.batch * d.xperm_stride;
        e.x = d.x;
        e.stride_x = q.stride_x;
        e.anchor_idx = d.anchor_idx;
        e.stride_anchor_idx = q.stride_anchor_idx;
        e.K = q.K;
        e.A = A;
        e.a_pad = a_pad;
        e.batch = q.batch;
        e.xperm_stride = d.xperm_stride;
        e.xaperm_stride = d.xaperm_stride;
        e.jobs = q.K / 256 + (a_pad + 255) / 256;
        e.job_begin = jobs;
        jobs += (int64_t)q.batch * e.jobs;
        e.xsc_off = d.xsc_off;
        e.row_begin = rows;
        rows += (int64_t)q.batch * M;
        max_k = std::max(max_k, q.K);
    }
    G.units = units;
    G.blocks = blocks;
    if (units == 0) return LQ_OK;
    // arrival counts live in the counter area, which every kernel leaves at zero
    if ((size_t)blocks > ws.num_counters) return LQ_ERR_UNSUPPORTED;
    P.stage = ring_stage(fmt) + (any_fuse ? kFuseBytes : 0);
    const size_t ring_smem = (size_t)cta_warps * kRingDepth * P.stage;
    // size the grid; the warp partition then fixes the x span of each CTA
    int per_sm = 0;
    if (use_ring) {
        if (dispatch_ring(0, false, P, 0, ring_smem, &per_sm, stream) != LQ_OK) return LQ_ERR_CUDA;
    } else if (dispatch(fmt, 0, false, P, 0, 0, &per_sm, stream) != LQ_OK) {
        return LQ_ERR_CUDA;
    }
    const int64_t grid = std::max<int64_t>(1, std::min<int64_t>((units + cta_warps - 1) / cta_warps, (int64_t)ws.num_sms * std::max(1, per_sm)));
    const int64_t W = std::min<int64_t>(grid * cta_warps, units);
    P.total_units = units;
    P.div32 = (uint64_t)units * (uint64_t)W < (1ull << 32) ? 1 : 0;
    P.total_warps = W;
    // With LQ_GEMV_STAGE=1 each CTA builds the x its units read in shared memory when that
    // span is small (a few members, room for a second resident CTA), and no pre-pass runs;
    // by default the pre-pass does it once for all CTAs (measured faster on this part), and the
    // per-CTA spans are not needed.
    const char* st_env = getenv("LQ_GEMV_STAGE");
    const bool want_stage = !use_ring && st_env && atoi(st_env) == 1 && !P.x_bf16;   // (binary16 x only)
    int64_t max_span = 0, max_members = 0, max_raw = 0, max_idx = 0, max_bits = 0;
    for (int64_t b = 0; (want_stage || use_ring) && b < grid; ++b) {
        const int64_t w_lo = b * cta_warps, w_hi = std::min<int64_t>(w_lo + cta_warps, W);
        if (w_lo >= W) break;
        int pa, pb;
        int64_t la, lb;
        host_locate(P, units * w_lo / W, pa, la);
        host_locate(P, units * w_hi / W - 1, pb, lb);
        max_span = std::max<int64_t>(max_span, P.d[pb].xoff + (lb + 1) * P.d[pb].xperm_stride - (P.d[pa].xoff + la * P.d[pa].xperm_stride));
        int64_t members = 0, raw = 0, idx = 0, bw = 0;
        for (int p = pa; p <= pb; ++p) {
            const int64_t n = (p == pb ? lb : P.d[p].batch - 1) - (p == pa ? la : 0) + 1;
            members += n;
            raw += n * M * P.d[p].K;
            idx += n * P.d[p].A;
            bw += n * (P.d[p].K / 32);
        }
        max_members = std::max(max_members, members);
        max_raw = std::max(max_raw, raw);
        max_idx = std::max(max_idx, idx);
        max_bits = std::max(max_bits, bw);
    }
    P.bitmap_words = std::max(1, max_k / 32);
    const size_t smem = (size_t)max_span * 2 + (size_t)P.bitmap_words * 4;
    bool staged = want_stage && max_members <= 4 && smem <= (size_t)std::min(ws.max_smem_optin, 110 * 1024);
    if (staged) {
        int per_sm_s = 0;
        if (dispatch(fmt, 0, true, P, 0, smem, &per_sm_s, stream) != LQ_OK) return LQ_ERR_CUDA;
        staged = per_sm_s >= per_sm;   // staging must not cost occupancy
    }
    // the ring kernel reads x from shared memory when each CTA's span of the x buffer fits
    // without costing occupancy (LQ_GEMV_XS=0 keeps x in global memory)
    const char* xs_env = getenv("LQ_GEMV_XS");
    bool ring_xs = use_ring && max_members <= 4 && !(xs_env && xs_env[0] == '0');
    const size_t ring_xs_smem = ring_smem + align256((size_t)max_span * 2);
    if (ring_xs) {
        int per_sm_x = 0;
        if (ring_xs_smem > (size_t)ws.max_smem_optin ||
            dispatch_ring(0, true, P, 0, ring_xs_smem, &per_sm_x, stream) != LQ_OK || per_sm_x < per_sm)
            ring_xs = false;
    }
    const int64_t min_run = units / W;   // every warp's run has at least this many units (>= 1)
    const bool no_xbuf = staged || (use_ring && ring_xs);   // x is built in shared memory by each CTA
    size_t ws_bytes = no_xbuf ? 0 : align256((size_t)xhalves * 2);
    for (int i = 0; i < count; ++i) {
        FDesc& d = P.d[i];
        d.cmax = (int)std::min<int64_t>(d.su / min_run + 2, d.su);
        ws_bytes += align256((size_t)probs[i].batch * d.rblocks * d.cmax * M * rows_blk * 4);
    }
    if (ws_bytes + 256 > ws.partial_floats * sizeof(float)) return LQ_ERR_WORKSPACE;
    // workspace: x copies (pre-pass only), then per problem the partial-sum slots
    char* wp = reinterpret_cast<char*>((reinterpret_cast<uintptr_t>(ws.partials) + 255) & ~uintptr_t(255));
    uint16_t* xbuf = reinterpret_cast<uint16_t*>(wp);
    if (!no_xbuf) wp += align256((size_t)xhalves * 2);
    P.xbuf = xbuf;
    unsigned* cnt = ws.counters;
    for (int i = 0; i < count; ++i) {
        FDesc& d = P.d[i];
        const lq_problem& q = probs[i];
        d.xperm = Q.d[i].xperm = xbuf + d.xoff;
        d.xaperm = Q.d[i].xaperm = xbuf + d.xoff + d.xa_off;
        d.part = reinterpret_cast<float*>(wp);
        wp += align256((size_t)q.batch * d.rblocks * d.cmax * M * rows_blk * 4);
        d.cnt = cnt;
        cnt += (int64_t)q.batch * d.rblocks;
    }
    Q.total_jobs = jobs;
    Q.total_rows = rows;
    Q.ring = use_ring ? 1 : 0;
    P.status = ws.status;
    G.use_ring = use_ring;
    G.ring_xs = use_ring && ring_xs;
    G.staged = staged;
    G.grid = grid;
    G.jobs = jobs;
    G.rows = rows;
    G.smem = staged ? smem : (use_ring ? (ring_xs ? ring_xs_smem : ring_smem) : 0);
    return LQ_OK;
}

// Launch a planned call: the kernel, after the x pre-pass when the x copy is in global memory.
lq_status run_plan(const GemvPlan& G, cudaStream_t stream) {
    const FParams& P = G.P;
    const PrepParams& Q = G.Q;
    const int fmt = P.format;
    const int64_t grid = G.grid, jobs = G.jobs, rows = G.rows;
    const bool use_ring = G.use_ring, ring_xs = G.ring_xs;
    int unused = 0;
    if (G.staged) return dispatch(fmt, 1, true, P, grid, G.smem, &unused, stream);
    if (use_ring && ring_xs) return dispatch_ring(1, true, P, grid, G.smem, &unused, stream);

    // x pre-pass (bf16 x: after each token's max |x|), then the main kernel, chained by
    // programmatic dependent launch
    const int64_t prep_ctas = (jobs + kPrepWarps - 1) / kPrepWarps;
    if (prep_ctas > 0x7fffffffLL || rows > 0x7fffffffLL) return LQ_ERR_UNSUPPORTED;
    if (P.x_bf16) {
        xmax_kernel<<<(unsigned)rows, 256, 0, stream>>>(Q);
        if (cudaPeekAtLastError() != cudaSuccess) return LQ_ERR_CUDA;
    }
    xprep_kernel<<<(unsigned)prep_ctas, 32 * kPrepWarps, 0, stream>>>(Q);
    if (cudaPeekAtLastError() != cudaSuccess) return LQ_ERR_CUDA;
    if (use_ring) return dispatch_ring(1, false, P, grid, G.smem, &unused, stream);
    return dispatch(fmt, 1, false, P, grid, 0, &unused, stream);
}

// Plans of recent calls.  A decode loop makes the same calls (the same layers, buffers and
// workspace) every token; such a call launches its kept plan instead of planning again, which
// takes the per-CTA span walk and the occupancy queries off the host's path.  The key is every
// byte the plan depends on: the problems, the workspace, and the kernel-choice settings.
constexpr int kPlanCache = 16;
struct PlanEntry {
    std::vector<unsigned char> key;
    GemvPlan plan;
    uint64_t used = 0;
};
std::mutex g_plan_mutex;
std::vector<PlanEntry> g_plans;
uint64_t g_plan_clock = 0;

void plan_key(const GemvWorkspace& ws, const lq_problem* probs, int count, std::vector<unsigned char>& key) {
    auto put = [&](const void* p, size_t n) {
        const unsigned char* b = static_cast<const unsigned char*>(p);
        key.insert(key.end(), b, b + n);
    };
    key.clear();
    put(&count, sizeof(count));
    put(probs, sizeof(lq_problem) * (size_t)count);
    const void* wsp[4] = {ws.partials, ws.counters, ws.status, nullptr};
    put(wsp, sizeof(wsp));
    const size_t wsn[4] = {ws.partial_floats, ws.num_counters, (size_t)ws.num_sms, (size_t)ws.max_smem_optin};
    put(wsn, sizeof(wsn));
    for (const char* name : {"LQ_GEMV_KERNEL", "LQ_GEMV_STAGE", "LQ_GEMV_XS"}) {
        const char* v = getenv(name);
        const std::string sv = v ? std::string("=") + v : std::string("-");
        put(sv.data(), sv.size() + 1);
    }
}

lq_status launch_gemv_stream(const GemvWorkspace& ws, const lq_problem* probs, int count, cudaStream_t stream) {
    thread_local std::vector<unsigned char> key;
    plan_key(ws, probs, count, key);
    std::lock_guard<std::mutex> lock(g_plan_mutex);
    PlanEntry* hit = nullptr;
    for (auto& e : g_plans)
        if (e.key == key) hit = &e;
    if (!hit) {
        PlanEntry fresh;
        const lq_status st = plan_gemv(ws, probs, count, fresh.plan, stream);
        if (st != LQ_OK) return st;
        fresh.key = key;
        if ((int)g_plans.size() < kPlanCache) {
            g_plans.push_back(std::move(fresh));
            hit = &g_plans.back();
        } else {
            hit = &g_plans[0];
            for (auto& e : g_plans)
                if (e.used < hit->used) hit = &e;
            *hit = std::move(fresh);
        }
    }
    hit->used = ++g_plan_clock;
    const GemvPlan& G = hit->plan;
    if (G.units == 0) return LQ_OK;
    if (ws.clear_counters && cudaMemsetAsync(ws.counters, 0, sizeof(unsigned) * (size_t)G.blocks, stream) != cudaSuccess)
        return LQ_ERR_CUDA;
    return run_plan(G, stream);
}

}  // namespace lq
