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
};

struct PrepParams {
    PrepDesc d[kMaxGroup];
    int count, M, x_bf16, format;
    int64_t total_jobs;
};

constexpr int kPrepWarps = 2;   // jobs per pre-pass CTA

__device__ __forceinline__ uint16_t to_half_bits(uint16_t raw, int x_bf16) {
    return x_bf16 ? __half_as_ushort(__float2half_rn(bf16_bits_to_float(raw))) : raw;
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
    if (jb < steps) {
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
                uint32_t w[4];
#pragma unroll
                for (int e2 = 0; e2 < 4; ++e2) {
                    uint32_t pr = 0;
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const int e = 2 * e2 + h, kl = col(it, e);
                        const bool anchor = (step_bits[warp][kl >> 5] >> (kl & 31)) & 1u;
                        pr |= (uint32_t)(anchor ? (uint16_t)0 : to_half_bits(v[c][e], P.x_bf16)) << (16 * h);
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
            uint16_t v[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const int pos = pos0 + e, tt = pos >> 2, hh = pos & 3;
                const int a = a_base + 16 * bl + 2 * tt + (hh & 1) + 8 * (hh >> 1);
                v[e] = a < A ? to_half_bits(x[(int64_t)m * K + __ldg(aidx + a)], P.x_bf16) : (uint16_t)0;
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
    const uint16_t* x;          // the caller's x [batch][M][K] (16-bit) and anchor columns, for
    int64_t stride_x;           //   the in-kernel build of the fragment-ordered copy (bytes)
    const int32_t* anchor_idx;
    int64_t stride_anchor_idx;  // bytes
};

struct FParams {
    FDesc d[kMaxGroup];
    const uint16_t* xbuf;       // all x copies: per problem, per member [x in fragment order | x at the anchors]
    int count, M, y_dtype, x_bf16, format;
    int bitmap_words;           // STAGED: shared-memory words of the anchor bitmap (max K / 32)
    int64_t total_units, total_warps;
};


// Position of a unit: problem, member, 16-row block, unit inside the row block, with
// the problem's units per row block cached.
struct Pos {
    int p, rb, s, steps, su;
    int64_t l;
};

// (rare paths are kept out of line: the unrolled unit loop must stay small)
__device__ __noinline__ Pos locate(const FParams& P, int64_t u) {
    Pos q;
    q.p = 0;
    while (q.p + 1 < P.count && u >= P.d[q.p + 1].unit_begin) ++q.p;
    const FDesc& D = P.d[q.p];
    int64_t loc = u - D.unit_begin;
    const int64_t per_member = (int64_t)D.rblocks * D.su;
    q.l = loc / per_member;
    loc -= q.l * per_member;
    q.rb = (int)(loc / D.su);
    q.s = (int)(loc - (int64_t)q.rb * D.su);
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

// The warp whose range [U*w/W, U*(w+1)/W) holds unit u.
__device__ __noinline__ int64_t owner_warp(int64_t u, int64_t W, int64_t U) { return ((u + 1) * W - 1) / U; }

// The last warp of a row block adds the slots of its nc contributors in order and writes y.
__device__ __noinline__ void finish_block(const float* slots, int nc, int M, void* y, int N, int row0, int y_dtype,
                                          int lane) {
    for (int i = lane; i < 16 * M; i += 32) {
        const int m = i >> 4, row = row0 + (i & 15);
        float sum = 0.f;
        for (int c = 0; c < nc; ++c) sum += __ldcg(slots + c * M * 16 + i);
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
    const int M = P.M, K = D.K, A = D.A, a_pad = (int)(D.xperm_stride / M) - K;
    const uint16_t* x = reinterpret_cast<const uint16_t*>(reinterpret_cast<const char*>(D.x) + l * D.stride_x);
    const int32_t* aidx = A > 0 ? reinterpret_cast<const int32_t*>(reinterpret_cast<const char*>(D.anchor_idx) + l * D.stride_anchor_idx)
                                : nullptr;
    for (int i = threadIdx.x; i < K / 32; i += blockDim.x) bits[i] = 0u;
    __syncthreads();
    for (int a = threadIdx.x; a < A; a += blockDim.x) {
        const int k = __ldg(aidx + a);
        atomicOr(&bits[k >> 5], 1u << (k & 31));
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
                v[e] = a < A ? to_half_bits(x[(int64_t)m * K + __ldg(aidx + a)], P.x_bf16) : (uint16_t)0;
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
        const int64_t uc0 = P.total_units * w_lo / W, uc1 = P.total_units * w_hi / W;
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
    const int64_t u_begin = P.total_units * wid / W, u_end = P.total_units * (wid + 1) / W;
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
        const int64_t w0 = first_u >= u_begin ? wid : owner_warp(first_u, W, P.total_units);
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
            const int nc = (int)(owner_warp(first_u + q.su - 1, W, P.total_units) - w0 + 1);
            finish_block(slots, nc, M, static_cast<char*>(D.y) + q.l * D.stride_y, D.N, q.rb * 16, P.y_dtype, lane);
        }
    };

    Pos q = locate(P, u_begin);
    int64_t u = u_begin;
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
            const float* am = reinterpret_cast<const float*>(static_cast<const char*>(D.scales) + q.l * D.stride_scales);
            const float *a0p = am + r0 * (K / 64), *a1p = am + r1 * (K / 64);
            uint32_t TL[4], TH[4];
            nf4_tables(TL, TH);
            auto load = [&](StepNF4& f, int s) {
#pragma unroll
                for (int nb = 0; nb < 4; ++nb) {
                    f.c0[nb] = ldg64(c0p + 128 * s + 32 * nb);
                    f.c1[nb] = ldg64(c1p + 128 * s + 32 * nb);
                    f.a0[nb] = __ldg(a0p + 4 * s + nb);
                    f.a1[nb] = __ldg(a1p + 4 * s + nb);
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
}

// Resident CTAs per SM of one instantiation at a given dynamic shared-memory size.
template <int FMT, int MT, int NT, bool STAGED>
int resident_ctas(size_t smem) {
    static size_t set_smem = (size_t)-1;
    static int per_sm = 0;
    if (set_smem != smem) {
        if (cudaFuncSetAttribute(gemv_stream_kernel<FMT, MT, NT, STAGED>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
            return -1;
        int n = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, gemv_stream_kernel<FMT, MT, NT, STAGED>, kThreadsS, smem) != cudaSuccess)
            return -1;
        per_sm = n;
        set_smem = smem;
    }
    return per_sm;
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

lq_status dispatch(int fmt, int mode, bool staged, const FParams& P, int64_t grid, size_t smem, int* per_sm,
                   cudaStream_t stream) {
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

bool gemv_stream_eligible(const lq_problem* probs, int count) {
    if (probs[0].M > 32) return false;
    for (int i = 0; i < count; ++i)
        if (probs[i].K % 256 != 0) return false;
    return true;
}

lq_status launch_gemv_stream(const GemvWorkspace& ws, const lq_problem* probs, int count, cudaStream_t stream) {
    FParams P;
    PrepParams Q;
    memset(&P, 0, sizeof(P));
    memset(&Q, 0, sizeof(Q));
    const int M = probs[0].M;
    const int fmt = probs[0].format;
    P.count = Q.count = count;
    P.M = Q.M = M;
    P.y_dtype = probs[0].y_dtype;
    P.format = Q.format = fmt;
    P.x_bf16 = Q.x_bf16 = probs[0].x_dtype == LQ_BF16;

    int64_t units = 0, jobs = 0, xhalves = 0, blocks = 0;
    int max_k = 0;
    for (int i = 0; i < count; ++i) {
        const lq_problem& q = probs[i];
        const int A = fmt == LQ_FMT_2BIT_LM_G32 ? q.A : 0;
        FDesc& d = P.d[i];
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
        d.x = static_cast<const uint16_t*>(q.x);
        d.stride_x = q.stride_x;
        d.anchor_idx = A > 0 ? q.anchor_idx : nullptr;
        d.stride_anchor_idx = q.stride_anchor_idx;
        const int a_pad = A > 0 ? round_up(A, kAnchorCols) : 0;
        d.steps = q.K / 256;
        d.su = d.steps + a_pad / kAnchorCols;
        d.rblocks = (q.N + 15) / 16;
        d.unit_begin = units;
        units += (int64_t)q.batch * d.rblocks * d.su;
        blocks += (int64_t)q.batch * d.rblocks;
        // per member: [x in fragment order (M*K) | x at the anchors (M*a_pad)]
        d.xperm_stride = d.xaperm_stride = (int64_t)M * (q.K + a_pad);
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
        max_k = std::max(max_k, q.K);
    }
    if (units == 0) return LQ_OK;
    // arrival counts live in the counter area, which every kernel leaves at zero
    if ((size_t)blocks > ws.num_counters) return LQ_ERR_UNSUPPORTED;
    // size the grid; the warp partition then fixes the x span of each CTA
    int per_sm = 0;
    if (dispatch(fmt, 0, false, P, 0, 0, &per_sm, stream) != LQ_OK) return LQ_ERR_CUDA;
    const int64_t grid = std::max<int64_t>(1, std::min<int64_t>((units + kWarps - 1) / kWarps, (int64_t)ws.num_sms * std::max(1, per_sm)));
    const int64_t W = std::min<int64_t>(grid * kWarps, units);
    P.total_units = units;
    P.total_warps = W;
    // With LQ_GEMV_STAGE=1 each CTA builds the x its units read in shared memory when that
    // span is small (a few members, room for a second resident CTA), and no pre-pass runs;
    // by default the pre-pass does it once for all CTAs (measured faster on this part), and the
    // per-CTA spans are not needed.
    const char* st_env = getenv("LQ_GEMV_STAGE");
    const bool want_stage = st_env && atoi(st_env) == 1;
    int64_t max_span = 0, max_members = 0;
    for (int64_t b = 0; want_stage && b < grid; ++b) {
        const int64_t w_lo = b * kWarps, w_hi = std::min<int64_t>(w_lo + kWarps, W);
        if (w_lo >= W) break;
        int pa, pb;
        int64_t la, lb;
        host_locate(P, units * w_lo / W, pa, la);
        host_locate(P, units * w_hi / W - 1, pb, lb);
        max_span = std::max<int64_t>(max_span, P.d[pb].xoff + (lb + 1) * P.d[pb].xperm_stride - (P.d[pa].xoff + la * P.d[pa].xperm_stride));
        int64_t members = 0;
        for (int p = pa; p <= pb; ++p) members += (p == pb ? lb : P.d[p].batch - 1) - (p == pa ? la : 0) + 1;
        max_members = std::max(max_members, members);
    }
    P.bitmap_words = std::max(1, max_k / 32);
    const size_t smem = (size_t)max_span * 2 + (size_t)P.bitmap_words * 4;
    bool staged = want_stage && max_members <= 4 && smem <= (size_t)std::min(ws.max_smem_optin, 110 * 1024);
    if (staged) {
        int per_sm_s = 0;
        if (dispatch(fmt, 0, true, P, 0, smem, &per_sm_s, stream) != LQ_OK) return LQ_ERR_CUDA;
        staged = per_sm_s >= per_sm;   // staging must not cost occupancy
    }
    const int64_t min_run = units / W;   // every warp's run has at least this many units (>= 1)
    size_t ws_bytes = staged ? 0 : align256((size_t)xhalves * 2);
    for (int i = 0; i < count; ++i) {
        FDesc& d = P.d[i];
        d.cmax = (int)std::min<int64_t>(d.su / min_run + 2, d.su);
        ws_bytes += align256((size_t)probs[i].batch * d.rblocks * d.cmax * M * 16 * 4);
    }
    if (ws_bytes + 256 > ws.partial_floats * sizeof(float)) return LQ_ERR_WORKSPACE;
    // workspace: x copies (pre-pass only), then per problem the partial-sum slots
    char* wp = reinterpret_cast<char*>((reinterpret_cast<uintptr_t>(ws.partials) + 255) & ~uintptr_t(255));
    uint16_t* xbuf = reinterpret_cast<uint16_t*>(wp);
    if (!staged) wp += align256((size_t)xhalves * 2);
    P.xbuf = xbuf;
    unsigned* cnt = ws.counters;
    for (int i = 0; i < count; ++i) {
        FDesc& d = P.d[i];
        const lq_problem& q = probs[i];
        d.xperm = Q.d[i].xperm = xbuf + d.xoff;
        d.xaperm = Q.d[i].xaperm = xbuf + d.xoff + (int64_t)M * q.K;
        d.part = reinterpret_cast<float*>(wp);
        wp += align256((size_t)q.batch * d.rblocks * d.cmax * M * 16 * 4);
        d.cnt = cnt;
        cnt += (int64_t)q.batch * d.rblocks;
    }
    if (ws.clear_counters && cudaMemsetAsync(ws.counters, 0, sizeof(unsigned) * (size_t)blocks, stream) != cudaSuccess)
        return LQ_ERR_CUDA;
    Q.total_jobs = jobs;
    int unused = 0;
    if (staged) return dispatch(fmt, 1, true, P, grid, smem, &unused, stream);

    // x pre-pass, then the main kernel, chained by programmatic dependent launch
    const int64_t prep_ctas = (jobs + kPrepWarps - 1) / kPrepWarps;
    if (prep_ctas > 0x7fffffffLL) return LQ_ERR_UNSUPPORTED;
    xprep_kernel<<<(unsigned)prep_ctas, 32 * kPrepWarps, 0, stream>>>(Q);
    if (cudaPeekAtLastError() != cudaSuccess) return LQ_ERR_CUDA;
    return dispatch(fmt, 1, false, P, grid, 0, &unused, stream);
}

}  // namespace lq
