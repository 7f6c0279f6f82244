// lq_gemm: prefill-sized y = x * W_eff^T on tcgen05 tensor cores.
//
// A dense contraction at M = 2048 tokens, so the weights are dequantized in
// registers and multiplied on the 5th-generation tensor cores by CTA pairs:
//
//  * Clusters of two CTAs (one per SM) walk output tiles of 256 weight rows x
//    256 tokens.  The pair's MMA (tcgen05.mma.cta_group::2, M = 256, N = 256,
//    K = 16) is issued by one thread of the even CTA; each CTA holds 128 rows of
//    the fp32 accumulator in its own tensor memory.
//  * Each CTA dequantizes its own 128 weight rows (2-bit: fmaf(S, C[q], Z) per
//    group, otf-llm README sections 2-3; NF4: T[q] * absmax, AirQuant README NF4;
//    INT4: S * q): a thread turns the 64 columns of one row in a K-block into
//    16-bit values and stores them straight into its tensor-memory lane
//    (tcgen05.st), which the MMA reads as its A operand.  Anchor columns
//    (section 4) are zeroed in the weight tile, and the anchors join as extra
//    K-blocks: binary16 anchor weights against x gathered at the anchor columns.
//  * Each CTA loads its own half of every x tile (128 tokens x 64 columns,
//    16-bit, 128-byte swizzle) by TMA; the pair MMA reads both halves.  Per SM,
//    shared memory carries only that half: a quarter of what one CTA with a
//    256-token tile and a shared-memory weight operand moves per K-block.
//  * One ring of K-block stages (weights in tensor memory, x in shared memory)
//    with one "stage full" barrier per stage in the even CTA and one pair commit
//    per K-block back to both CTAs: the MMA thread waits once and commits once
//    per K-block (extra barrier work in that thread shows up as tensor-pipe idle
//    time; measured).  The odd CTA's x arrival is relayed to the even CTA's
//    barrier by its otherwise idle MMA warp.
//  * A metadata warp streams codes, scales and anchor weights by TMA; the last
//    warps read the accumulator back with tcgen05.ld and write y.
// The multiply runs in the dtype of x (bf16 or binary16) with fp32 accumulation.
// Every mbarrier wait is bounded in time.

#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstring>
#include <mutex>
#include <vector>

#include "lq_common.cuh"
#include "lq_dq.cuh"
#include "lq_internal.h"
#include "lq_tcgen05.cuh"
#include "lq_tma.cuh"

namespace lq {
namespace {

constexpr int kSmemLimit = 227 * 1024;   // dynamic shared memory per CTA (opt-in maximum)
constexpr int kBM = 128;                 // weight rows per CTA; a CTA pair's MMA covers 2 x 128
constexpr int kPairM = 2 * kBM;          // weight rows per tile
constexpr int kBN = 256;                 // tokens per tile (MMA N)
constexpr int kHalfN = kBN / 2;          // x rows each CTA of the pair holds
constexpr int kBK = 64;                  // columns per K-block (one 128-byte swizzle row of 16-bit values)
constexpr int kATile = kBM * kBK * 2;    // 16 KiB: one anchor weight tile in a metadata slot
constexpr int kBTile = kHalfN * kBK * 2; // 16 KiB: this CTA's half of one x tile
constexpr int kChunk = 4;                // K-blocks of codes and scales per metadata load
constexpr int kMetaSlots = 3;            // metadata chunks in flight
constexpr int kDqWarp0 = 3;              // warps: 0 x TMA, 1 MMA (relay in the odd CTA), 2 metadata, dequant, epilogue
// tensor memory of each CTA: the accumulator (128 lanes x kBN columns), then the weight stages
// (32 columns each: one K-block of 64 16-bit values per lane)
constexpr int kTmemCols = 512;
constexpr int kACol0 = kBN;
// One ring of K-block stages: stage s holds the weights in tensor memory columns kACol0 + 32 s
// and this CTA's half of the x tile in shared memory.
constexpr int kStages = (kTmemCols - kACol0) / 32;
static_assert(kStages >= 4 && kACol0 + 32 * kStages <= kTmemCols, "tensor memory columns");
static_assert(kTmemCols >= 32 && kTmemCols <= 512 && (kTmemCols & (kTmemCols - 1)) == 0,
              "tcgen05.alloc takes a power of two from 32 to 512 columns");
static_assert(kBN % 16 == 0 && kBN <= 256 && kBN % 64 == 0, "MMA N");

// Per-format layout of the shared memory: the x ring (this CTA's half of each x tile), two
// metadata slots, the barriers.
template <int FMT>
struct GemmLayout {
    static constexpr bool kNF4Fmt = FMT == LQ_FMT_NF4_B64;
    static constexpr bool kInt4Fmt = FMT == LQ_FMT_INT4_G32;
    static constexpr bool kNib = kNF4Fmt || kInt4Fmt;   // 4-bit codes, 32 bytes per row and K-block
    // Warp roles (measured per format on the 14B prefill layer): groups of four dequant warps
    // take the K-blocks in turn (three for the 4-bit codes, whose expansion costs more; two for
    // 2-bit), then the epilogue warps (one or two per tensor-memory lane quarter).
    static constexpr int kDqGroups = kNib ? 3 : 2;
    static constexpr int kDqWarps = 4 * kDqGroups;
    static constexpr int kEpiWarps = kNib ? 4 : 8;
    static constexpr int kEpiWarp0 = kDqWarp0 + kDqWarps;
    static constexpr int kThreads = (kEpiWarp0 + kEpiWarps) * 32;
    static_assert(kBN * 4 % (32 * kEpiWarps) == 0, "epilogue split");
    // one metadata chunk (kChunk K-blocks of 128 rows):
    //   2-bit: codes [128][64 B] (64-byte swizzle) | scales [128][8 x f16] | offsets [128][8 x f16] |
    //          anchor bits [4][u64] | keep masks [4][32 x u32] (word w clears the halves of anchor columns 2w, 2w+1)
    //   NF4:   codes [128][128 B] (128-byte swizzle) | absmax [128][4 x f32]
    //   INT4:  codes [128][128 B] (128-byte swizzle; permuted positions) | scales [128][8 x f16]
    static constexpr int kCodesBytes = kBM * kChunk * (kNib ? 32 : 16);
    static constexpr int kScaleOff = kCodesBytes;
    static constexpr int kOffsetOff = kScaleOff + kBM * 16;
    static constexpr int kBitsOff = kOffsetOff + (kNib ? 0 : kBM * 16);
    static constexpr int kMaskOff = kBitsOff + 32;
    // a 2-bit or INT4 slot also carries one anchor weight tile [128][64 x f16] (128-byte swizzle)
    static constexpr int kMetaBytes = ((kNib ? kBitsOff : kMaskOff + kChunk * 128) + 1023) / 1024 * 1024;
    static constexpr int kChunkBytes = kNF4Fmt ? kMetaBytes : (kMetaBytes > kATile ? kMetaBytes : kATile);
    static constexpr int kBOff = 0;
    static constexpr int kMetaOff = kBOff + kStages * kBTile;
    static constexpr int kBarOff = kMetaOff + kMetaSlots * kChunkBytes;
    static constexpr int kNumBars = 3 * kStages + 2 * kMetaSlots + 2;
    static constexpr int kSmemBytes = 1024 + kBarOff + kNumBars * 8;
    static_assert(kSmemBytes <= kSmemLimit, "shared memory");
};

// One problem of a (grouped) launch: tensor maps, pointers and shape.
struct GemmProb {
    CUtensorMap xmap;          // x [M][K] 16-bit, box 64 x 256, 128-byte swizzle
    CUtensorMap xamap;         // x at the anchor columns [M][a_pad], same box
    CUtensorMap awmap;         // anchor weights [N][ld_anchor] binary16, box 64 x 128, 128-byte swizzle
    CUtensorMap cmap;          // codes [N][K/4] or [N][K/2] bytes, box (chunk of K-blocks) x 128
    CUtensorMap smap;          // scales [N][K/32] f16 or absmax [N][K/64] f32, box 16 bytes x 128
    CUtensorMap omap;          // offsets [N][K/32] f16, box 16 bytes x 128
    const void* scales;
    const uint16_t* offsets;
    const uint32_t* anchor_bits;   // [K/32 + 8] anchor columns of each 32-column half block
    void* y;
    int M, N, K, A, a_pad, y_dtype, meta_tma;
    int tiles_m, tile_begin;   // token tiles per row tile (of kPairM rows); first tile of this problem in the launch
};

struct GemmParams {
    GemmProb d[kMaxGemmGroup];
    int count, bf16, total_tiles;
    const int* sched_off;      // tile list of CTA pair c: sched_tiles[sched_off[c] .. sched_off[c+1]) (null: round robin)
    const int* sched_tiles;
    int* status;
};

// Tiles of CTA pair c (of npair), the i-th of them, and the problem a tile belongs to.
__device__ __forceinline__ int pair_tiles(const GemmParams& P, int c, int npair) {
    if (P.sched_off) return P.sched_off[c + 1] - P.sched_off[c];
    return c < P.total_tiles ? (P.total_tiles - 1 - c) / npair + 1 : 0;
}
__device__ __forceinline__ int tile_id(const GemmParams& P, int i, int c, int npair) {
    return P.sched_off ? __ldg(P.sched_tiles + P.sched_off[c] + i) : c + i * npair;
}
__device__ __forceinline__ int tile_prob(const GemmParams& P, int gt) {
    int p = 0;
    while (p + 1 < P.count && gt >= P.d[p + 1].tile_begin) ++p;
    return p;
}

__device__ __forceinline__ uint32_t pack2(float lo, float hi, int bf16) {
    uint32_t d;
    if (bf16)
        asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
    else
        asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
    return d;
}

// 16 natural-order weights of one code word -> two 16-byte chunks (8 values each).
__device__ __forceinline__ void dq2_word(uint32_t w, uint32_t P01, uint32_t P23, uint32_t (&c0)[4], uint32_t (&c1)[4]) {
    const uint32_t t0 = w & 0x03030303u, t1 = (w >> 2) & 0x03030303u;
    const uint32_t t2 = (w >> 4) & 0x03030303u, t3 = (w >> 6) & 0x03030303u;
    // byte lanes of (t0,t1) / (t2,t3) interleaved: selector nibbles (2q, 2q+1) per value
    const uint32_t sa = prmt(t0, t1, 0x5140) * 0x22u + 0x10101010u;   // columns 0,1 | 4,5
    const uint32_t sb = prmt(t2, t3, 0x5140) * 0x22u + 0x10101010u;   // columns 2,3 | 6,7
    const uint32_t sc = prmt(t0, t1, 0x7362) * 0x22u + 0x10101010u;   // columns 8,9 | 12,13
    const uint32_t sd = prmt(t2, t3, 0x7362) * 0x22u + 0x10101010u;   // columns 10,11 | 14,15
    c0[0] = prmt(P01, P23, sa);
    c0[1] = prmt(P01, P23, sb);
    c0[2] = prmt(P01, P23, sa >> 16);
    c0[3] = prmt(P01, P23, sb >> 16);
    c1[0] = prmt(P01, P23, sc);
    c1[1] = prmt(P01, P23, sd);
    c1[2] = prmt(P01, P23, sc >> 16);
    c1[3] = prmt(P01, P23, sd >> 16);
}

struct Ring {
    int s = 0, ph = 0;
    __device__ __forceinline__ void next(int depth) {
        if (++s == depth) {
            s = 0;
            ph ^= 1;
        }
    }
};

template <int FMT>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(GemmLayout<FMT>::kThreads, 1)
    gemm_kernel(const __grid_constant__ GemmParams P) {
    using L = GemmLayout<FMT>;
    constexpr int kDqGroups = L::kDqGroups, kDqWarps = L::kDqWarps, kEpiWarps = L::kEpiWarps, kEpiWarp0 = L::kEpiWarp0;
    constexpr int S = kStages;
    extern __shared__ uint8_t smem_raw[];
    // (the same offsets in both CTAs of a pair: the pair's MMA reads x at one shared-memory
    // offset in each, and commits arrive at one barrier offset in each)
    uint8_t* base = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
    uint8_t* btile = base + L::kBOff;       // [S][128 rows][128 B], 128-byte swizzle
    uint8_t* meta = base + L::kMetaOff;     // [kMetaSlots][chunk]
    uint64_t* bars = reinterpret_cast<uint64_t*>(base + L::kBarOff);
    __shared__ uint32_t s_tmem;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t rank = cluster_rank();   // 0: issues the pair's MMAs; 1: its partner
    const int pair = (int)(blockIdx.x >> 1), npair = (int)(gridDim.x >> 1);
    const uint32_t full0 = smem_u32(bars), empty0 = full0 + 8 * S, xloc0 = empty0 + 8 * S;
    const uint32_t m_full0 = xloc0 + 8 * S, m_empty0 = m_full0 + 8 * kMetaSlots;
    const uint32_t acc_full0 = m_empty0 + 8 * kMetaSlots, acc_empty0 = acc_full0 + 8;

    // Barriers.  full[s] (used in rank 0) completes when the stage is whole in both CTAs: the
    // owning dequant group's four warps in each CTA, rank 0's x TMA (arrival and bytes) and the
    // relay of rank 1's x TMA.  empty[s] (both CTAs) receives the pair commit of the MMAs that
    // read the stage.  xloc[s] (rank 1) completes on rank 1's x TMA.  acc_full (both) receives
    // the pair commit of a tile; acc_empty (rank 0) the epilogue warps of both CTAs.  The
    // metadata ring is local.  The MMA thread waits on one barrier and commits to one per
    // K-block: every extra wait or commit there shows up as tensor-pipe idle time.
    if (tid == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(full0 + 8 * s, 4 + 4 + 1 + 1);
            mbar_init(empty0 + 8 * s, 1);
            mbar_init(xloc0 + 8 * s, 1);
        }
        for (int i = 0; i < kMetaSlots; ++i) {
            mbar_init(m_full0 + 8 * i, 32);
            mbar_init(m_empty0 + 8 * i, kDqWarps);
        }
        mbar_init(acc_full0, 1);
        mbar_init(acc_empty0, 2 * kEpiWarps);
        fence_mbar_init();
    }
    if (warp == 1) tmem_alloc_pair(smem_u32(&s_tmem), kTmemCols);
    tc_fence_before();
    __syncwarp();
    cluster_sync_all();   // both CTAs' barriers initialised before any remote arrival or pair commit
    tc_fence_after();
    const uint32_t tmem = s_tmem;

    const int ntiles = pair_tiles(P, pair, npair);
    int own_abort = 0;
    volatile int* abort = &own_abort;

    if (warp == 0) {
        // ---------------------------------------------------------------- TMA: this CTA's half of the x tiles
        if (lane == 0) {
            for (int p = 0; p < P.count; ++p) {
                prefetch_tensormap(&P.d[p].xmap);
                if (P.d[p].a_pad) prefetch_tensormap(&P.d[p].xamap);
            }
            const uint32_t done0 = rank == 0 ? full0 : xloc0;   // where this CTA's x bytes complete
            Ring rs;
            bool ok = true;
            for (int i = 0; ok && i < ntiles; ++i) {
                const int gt = tile_id(P, i, pair, npair);
                const GemmProb& D = P.d[tile_prob(P, gt)];
                const int lt = gt - D.tile_begin, mh = (lt % D.tiles_m) * kBN + (int)rank * kHalfN;
                const int KB = D.K / kBK, NKB = KB + D.a_pad / kBK;
                for (int kb = 0; kb < NKB; ++kb) {
                    if (!(ok = mbar_wait_bounded<true>(empty0 + 8 * rs.s, rs.ph ^ 1, abort, P.status))) break;
                    const uint32_t fb = done0 + 8 * rs.s, dst = smem_u32(btile + rs.s * kBTile);
                    mbar_arrive_expect_tx(fb, kBTile);
                    if (kb < KB) tma_load_2d(dst, &D.xmap, kb * kBK, mh, fb);
                    else tma_load_2d(dst, &D.xamap, (kb - KB) * kBK, mh, fb);   // x at the anchors
                    rs.next(S);
                }
            }
            // every stage's last release has arrived before this CTA may exit
            for (int s = 0; ok && s < S; ++s) {
                ok = mbar_wait_bounded<true>(empty0 + 8 * rs.s, rs.ph ^ 1, abort, P.status);
                rs.next(S);
            }
        }
    } else if (warp == 1) {
        if (rank == 0 && lane == 0) {
            // ------------------------------------------------------------ pair MMA issue (M = 256, N = 256, K = 16)
            const uint32_t idesc = idesc_f16(P.bf16 != 0, kPairM, kBN);
            const uint32_t a_t0 = tmem + kACol0, b_t0 = smem_u32(btile);
            Ring rs;
            bool ok = true;
            for (int i = 0; ok && i < ntiles; ++i) {
                const GemmProb& D = P.d[tile_prob(P, tile_id(P, i, pair, npair))];
                const int NKB = D.K / kBK + D.a_pad / kBK;
                // both CTAs' epilogues have drained the accumulator (the tile before)
                if (!(ok = mbar_wait_bounded<true>(acc_empty0, (i & 1) ^ 1, abort, P.status))) break;
                tc_fence_after();
                for (int kb = 0; kb < NKB; ++kb) {
                    if (!(ok = mbar_wait_bounded<true>(full0 + 8 * rs.s, rs.ph, abort, P.status))) break;
                    tc_fence_after();
                    const uint32_t a_t = a_t0 + 32 * rs.s, b_addr = b_t0 + rs.s * kBTile;
#pragma unroll
                    for (int k = 0; k < kBK / 16; ++k)   // K = 16: 8 columns of A, 32 bytes of each B row
                        tc_mma_f16_ts_pair(tmem, a_t + 8 * k, smem_desc_sw128(b_addr + 32 * k), idesc, (kb | k) != 0);
                    tc_commit_pair(empty0 + 8 * rs.s);   // both CTAs' stage is free once these MMAs have read it
                    rs.next(S);
                }
                if (ok) tc_commit_pair(acc_full0);
            }
        } else if (rank == 1 && lane == 0) {
            // ------------------------------------------------------------ relay: this CTA's x stages to rank 0
            const uint32_t full_r0 = mapa_shared(full0, 0);
            Ring rs;
            bool ok = true;
            for (int i = 0; ok && i < ntiles; ++i) {
                const GemmProb& D = P.d[tile_prob(P, tile_id(P, i, pair, npair))];
                const int NKB = D.K / kBK + D.a_pad / kBK;
                for (int kb = 0; kb < NKB; ++kb) {
                    if (!(ok = mbar_wait_bounded(xloc0 + 8 * rs.s, rs.ph, abort, P.status))) break;
                    mbar_arrive_remote(full_r0 + 8 * rs.s);
                    rs.next(S);
                }
            }
        }
    } else if (warp == 2) {
        // ---------------------------------------------------------------- metadata: codes, scales, anchor bits
        if (lane == 0) {
            for (int p = 0; p < P.count; ++p) {
                prefetch_tensormap(&P.d[p].cmap);
                if (P.d[p].meta_tma) {
                    prefetch_tensormap(&P.d[p].smap);
                    if (!L::kNib) prefetch_tensormap(&P.d[p].omap);
                }
                if (P.d[p].a_pad) prefetch_tensormap(&P.d[p].awmap);
            }
        }
        Ring rm;
        for (int i = 0; i < ntiles; ++i) {
            const int gt = tile_id(P, i, pair, npair);
            const GemmProb& D = P.d[tile_prob(P, gt)];
            const int lt = gt - D.tile_begin, n0 = (lt / D.tiles_m) * kPairM + (int)rank * kBM;   // this CTA's rows
            const int KB = D.K / kBK, NCH = (KB + kChunk - 1) / kChunk;
            for (int c = 0; c < NCH; ++c) {
                if (!__all_sync(0xffffffffu, mbar_wait_bounded(m_empty0 + 8 * rm.s, rm.ph ^ 1, abort, P.status)))
                    goto meta_done;
                uint8_t* ch = meta + rm.s * L::kChunkBytes;
                const uint32_t fb = m_full0 + 8 * rm.s;
                const int kb0 = c * kChunk;
                if (!L::kNib && D.A > 0) {
                    // anchor columns of the chunk's K-blocks and the per-word keep masks
                    const uint4 b01 = *reinterpret_cast<const uint4*>(D.anchor_bits + 2 * kb0);
                    const uint4 b23 = *reinterpret_cast<const uint4*>(D.anchor_bits + 2 * kb0 + 4);
                    const uint32_t bw[8] = {b01.x, b01.y, b01.z, b01.w, b23.x, b23.y, b23.z, b23.w};
                    if (lane == 0) {
                        reinterpret_cast<uint4*>(ch + L::kBitsOff)[0] = b01;
                        reinterpret_cast<uint4*>(ch + L::kBitsOff)[1] = b23;
                    }
#pragma unroll
                    for (int j = 0; j < kChunk; ++j) {
                        const uint32_t half = ((lane >> 4) ? bw[2 * j + 1] : bw[2 * j]) >> (2 * (lane & 15));
                        const uint32_t keep = ((half & 1u) ? 0xFFFF0000u : 0xFFFFFFFFu) & ((half & 2u) ? 0x0000FFFFu : 0xFFFFFFFFu);
                        reinterpret_cast<uint32_t*>(ch + L::kMaskOff + j * 128)[lane] = keep;
                    }
                }
                if (!D.meta_tma) {
                    // scale rows are not 16-byte aligned: 4-byte loads, four rows per lane
                    const int nk = min(kChunk, KB - kb0);
                    for (int rr = lane; rr < kBM; rr += 32) {
                        const int64_t nr = min(n0 + rr, D.N - 1);
                        if (L::kNF4Fmt) {
                            const float* src = static_cast<const float*>(D.scales) + nr * (D.K / 64) + kb0;
                            for (int i = 0; i < nk; ++i)
                                reinterpret_cast<float*>(ch + L::kScaleOff + rr * 16)[i] = __ldg(src + i);
                        } else if (L::kInt4Fmt) {
                            const uint32_t* ss = reinterpret_cast<const uint32_t*>(static_cast<const uint16_t*>(D.scales) +
                                                                                   nr * (D.K / 32) + 2 * kb0);
                            for (int i = 0; i < nk; ++i) reinterpret_cast<uint32_t*>(ch + L::kScaleOff + rr * 16)[i] = __ldg(ss + i);
                        } else {
                            const int64_t g = nr * (D.K / 32) + 2 * kb0;
                            const uint32_t* ss = reinterpret_cast<const uint32_t*>(static_cast<const uint16_t*>(D.scales) + g);
                            const uint32_t* so = reinterpret_cast<const uint32_t*>(D.offsets + g);
                            for (int i = 0; i < nk; ++i) {
                                reinterpret_cast<uint32_t*>(ch + L::kScaleOff + rr * 16)[i] = __ldg(ss + i);
                                reinterpret_cast<uint32_t*>(ch + L::kOffsetOff + rr * 16)[i] = __ldg(so + i);
                            }
                        }
                    }
                }
                if (lane == 0) {
                    uint32_t tx = L::kCodesBytes;
                    if (D.meta_tma) tx += L::kNib ? kBM * 16 : 2 * kBM * 16;
                    mbar_arrive_expect_tx(fb, tx);
                    tma_load_2d(smem_u32(ch), &D.cmap, kb0 * (L::kNib ? 32 : 16), n0, fb);
                    if (D.meta_tma) {
                        tma_load_2d(smem_u32(ch + L::kScaleOff), &D.smap, kb0 * (L::kNF4Fmt ? 1 : 2), n0, fb);
                        if (!L::kNib)
                            tma_load_2d(smem_u32(ch + L::kOffsetOff), &D.omap, kb0 * 2, n0, fb);
                    }
                } else {
                    mbar_arrive(fb);
                }
                rm.next(kMetaSlots);
            }
            // anchor weight tiles of this tile, one per slot
            for (int a = 0; a < D.a_pad / kBK; ++a) {
                if (!__all_sync(0xffffffffu, mbar_wait_bounded(m_empty0 + 8 * rm.s, rm.ph ^ 1, abort, P.status)))
                    goto meta_done;
                const uint32_t fb = m_full0 + 8 * rm.s;
                if (lane == 0) {
                    mbar_arrive_expect_tx(fb, kATile);
                    tma_load_2d(smem_u32(meta + rm.s * L::kChunkBytes), &D.awmap, a * kBK, n0, fb);
                } else {
                    mbar_arrive(fb);
                }
                rm.next(kMetaSlots);
            }
        }
    meta_done:;
    } else if (warp < kEpiWarp0) {
        // ---------------------------------------------------------------- dequant into the A stages
        // kDqGroups groups of four warps take the K-blocks in turn, so that many K-blocks
        // are in flight; each thread turns one row's 64 columns into 16-bit values
        // and stores them to its tensor-memory lane (a warp reaches lanes 32 * (warp % 4) on).
        const int g = (warp - kDqWarp0) >> 2, r = 32 * (warp & 3) + lane;
        const uint32_t a_lane = tmem + ((uint32_t)(32 * (warp & 3)) << 16) + kACol0;
        const uint32_t full_r0 = mapa_shared(full0, 0);   // rank 0's stage barriers
        const int sw = r & 7;
        const float C0 = -1.52f, C1 = -0.45f, C2 = 0.45f, C3 = 1.52f;
        Ring ra, rm;
        for (int i = 0; i < ntiles; ++i) {
          const GemmProb& D = P.d[tile_prob(P, tile_id(P, i, pair, npair))];
          const int KB = D.K / kBK, NKB = KB + D.a_pad / kBK;
          for (int kb = 0; kb < NKB; ++kb) {
            const bool mine = kb % kDqGroups == g;
            if (kb < KB) {
                const int j = kb % kChunk;
                // every warp waits for each metadata chunk and releases it at its end, so a
                // release never runs ahead of the load it frees (count: all dequant warps)
                if (j == 0 && !__all_sync(0xffffffffu, mbar_wait_bounded(m_full0 + 8 * rm.s, rm.ph, abort, P.status)))
                    goto dq_done;
                if (mine) {
                    if (!__all_sync(0xffffffffu, mbar_wait_bounded<true>(empty0 + 8 * ra.s, ra.ph ^ 1, abort, P.status)))
                        goto dq_done;
                    tc_fence_after();   // the MMAs that read this stage have completed
                    const uint8_t* ch = meta + rm.s * L::kChunkBytes;
                    uint32_t c[32];   // c[4q + k]: columns 8q + 2k, 8q + 2k + 1
                    if (FMT == LQ_FMT_2BIT_LM_G32) {
                        const uint4 cw = *reinterpret_cast<const uint4*>(ch + r * 64 + ((j ^ ((r >> 1) & 3)) << 4));
                        const uint32_t s2 = *reinterpret_cast<const uint32_t*>(ch + L::kScaleOff + r * 16 + 4 * j);
                        const uint32_t z2 = *reinterpret_cast<const uint32_t*>(ch + L::kOffsetOff + r * 16 + 4 * j);
                        const float s0 = half_bits_to_float((uint16_t)s2), z0 = half_bits_to_float((uint16_t)z2);
                        const float s1 = half_bits_to_float((uint16_t)(s2 >> 16)), z1 = half_bits_to_float((uint16_t)(z2 >> 16));
                        const uint32_t A01 = pack2(__fmaf_rn(s0, C0, z0), __fmaf_rn(s0, C1, z0), P.bf16);
                        const uint32_t A23 = pack2(__fmaf_rn(s0, C2, z0), __fmaf_rn(s0, C3, z0), P.bf16);
                        const uint32_t B01 = pack2(__fmaf_rn(s1, C0, z1), __fmaf_rn(s1, C1, z1), P.bf16);
                        const uint32_t B23 = pack2(__fmaf_rn(s1, C2, z1), __fmaf_rn(s1, C3, z1), P.bf16);
                        dq2_word(cw.x, A01, A23, *reinterpret_cast<uint32_t(*)[4]>(c + 0), *reinterpret_cast<uint32_t(*)[4]>(c + 4));
                        dq2_word(cw.y, A01, A23, *reinterpret_cast<uint32_t(*)[4]>(c + 8), *reinterpret_cast<uint32_t(*)[4]>(c + 12));
                        dq2_word(cw.z, B01, B23, *reinterpret_cast<uint32_t(*)[4]>(c + 16), *reinterpret_cast<uint32_t(*)[4]>(c + 20));
                        dq2_word(cw.w, B01, B23, *reinterpret_cast<uint32_t(*)[4]>(c + 24), *reinterpret_cast<uint32_t(*)[4]>(c + 28));
                        if (D.A > 0) {
                            // anchor columns replace the 2-bit weights: clear them with the chunk's keep
                            // masks, only in the 16-column words that hold one (the bitmap is warp-uniform)
                            const uint2 bw = *reinterpret_cast<const uint2*>(ch + L::kBitsOff + 8 * j);
                            const uint32_t* km = reinterpret_cast<const uint32_t*>(ch + L::kMaskOff + j * 128);
#pragma unroll
                            for (int wi = 0; wi < 4; ++wi) {
                                if (((wi < 2 ? bw.x : bw.y) >> (16 * (wi & 1))) & 0xFFFFu) {
                                    const uint4 m0 = *reinterpret_cast<const uint4*>(km + 8 * wi);
                                    const uint4 m1 = *reinterpret_cast<const uint4*>(km + 8 * wi + 4);
                                    c[8 * wi + 0] &= m0.x;
                                    c[8 * wi + 1] &= m0.y;
                                    c[8 * wi + 2] &= m0.z;
                                    c[8 * wi + 3] &= m0.w;
                                    c[8 * wi + 4] &= m1.x;
                                    c[8 * wi + 5] &= m1.y;
                                    c[8 * wi + 6] &= m1.z;
                                    c[8 * wi + 7] &= m1.w;
                                }
                            }
                        }
                    } else if (FMT == LQ_FMT_INT4_G32) {
                        // two 32-position groups: each group's 16 values S * q (q the nibble as a 4-bit
                        // two's complement integer; exact in fp32, then one rounding) in byte-split registers
                        const uint8_t* crow = ch + r * 128;
                        const uint4 cw0 = *reinterpret_cast<const uint4*>(crow + (((2 * j) ^ sw) << 4));
                        const uint4 cw1 = *reinterpret_cast<const uint4*>(crow + (((2 * j + 1) ^ sw) << 4));
                        const uint32_t s2 = *reinterpret_cast<const uint32_t*>(ch + L::kScaleOff + r * 16 + 4 * j);
                        // both groups' products q * (S0, S1) per packed fp32 FMA (q * S + (-0) is the exact
                        // product, sign of zero included, as one multiply would give)
                        const float2 sg2 = make_float2(half_bits_to_float((uint16_t)(s2 & 0xFFFFu)),
                                                       half_bits_to_float((uint16_t)(s2 >> 16)));
                        uint32_t BL[2][4], BH[2][4];
#pragma unroll
                        for (int q4 = 0; q4 < 4; ++q4) {
                            float2 v[4];
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const int nib = 4 * q4 + e;
                                v[e] = fma_f32x2(sg2, (float)(nib < 8 ? nib : nib - 16), make_float2(-0.f, -0.f));
                            }
#pragma unroll
                            for (int hh = 0; hh < 2; ++hh) {
                                const uint32_t p01 = pack2(hh ? v[0].y : v[0].x, hh ? v[1].y : v[1].x, P.bf16);
                                const uint32_t p23 = pack2(hh ? v[2].y : v[2].x, hh ? v[3].y : v[3].x, P.bf16);
                                BL[hh][q4] = prmt(p01, p23, 0x6420);
                                BH[hh][q4] = prmt(p01, p23, 0x7531);
                            }
                        }
#pragma unroll
                        for (int hh = 0; hh < 2; ++hh) {
                            const uint4& cw = hh ? cw1 : cw0;
                            const uint32_t ws[4] = {cw.x, cw.y, cw.z, cw.w};
#pragma unroll
                            for (int wi = 0; wi < 4; ++wi) {
                                expand_nf4_fast(ws[wi], 0, BL[hh], BH[hh], c[16 * hh + 4 * wi + 0], c[16 * hh + 4 * wi + 1]);
                                expand_nf4_fast(ws[wi], 1, BL[hh], BH[hh], c[16 * hh + 4 * wi + 2], c[16 * hh + 4 * wi + 3]);
                            }
                        }
                    } else {
                        const uint8_t* crow = ch + r * 128;
                        const uint4 cw0 = *reinterpret_cast<const uint4*>(crow + (((2 * j) ^ sw) << 4));
                        const uint4 cw1 = *reinterpret_cast<const uint4*>(crow + (((2 * j + 1) ^ sw) << 4));
                        const float am = reinterpret_cast<const float*>(ch + L::kScaleOff + r * 16)[j];
                        // this block's 16 values T[q] * absmax, one rounding, in byte-split registers
                        uint32_t BL[4], BH[4];
#pragma unroll
                        for (int q4 = 0; q4 < 4; ++q4) {
                            const uint32_t p01 = pack2(__fmul_rn(kNF4[4 * q4], am), __fmul_rn(kNF4[4 * q4 + 1], am), P.bf16);
                            const uint32_t p23 = pack2(__fmul_rn(kNF4[4 * q4 + 2], am), __fmul_rn(kNF4[4 * q4 + 3], am), P.bf16);
                            BL[q4] = prmt(p01, p23, 0x6420);
                            BH[q4] = prmt(p01, p23, 0x7531);
                        }
                        const uint32_t ws[8] = {cw0.x, cw0.y, cw0.z, cw0.w, cw1.x, cw1.y, cw1.z, cw1.w};
#pragma unroll
                        for (int wi = 0; wi < 8; ++wi) {
                            expand_nf4_fast(ws[wi], 0, BL, BH, c[4 * wi + 0], c[4 * wi + 1]);
                            expand_nf4_fast(ws[wi], 1, BL, BH, c[4 * wi + 2], c[4 * wi + 3]);
                        }
                    }
                    tmem_st32(a_lane + 32 * ra.s, c);
                    tc_fence_before();   // the stores are complete: order them before the arrival
                    __syncwarp();
                    if (lane == 0) mbar_arrive_remote(full_r0 + 8 * ra.s);
                }
                if (j == kChunk - 1 || kb == KB - 1) {
                    if (lane == 0) mbar_arrive(m_empty0 + 8 * rm.s);
                    rm.next(kMetaSlots);
                }
            } else {
                // anchor block: the metadata slot holds 64 binary16 anchor weights per row; the
                // owning group copies them into the stage, zero past A, in bf16 when x is bf16
                if (!__all_sync(0xffffffffu, mbar_wait_bounded(m_full0 + 8 * rm.s, rm.ph, abort, P.status))) goto dq_done;
                if (mine) {
                    if (!__all_sync(0xffffffffu, mbar_wait_bounded<true>(empty0 + 8 * ra.s, ra.ph ^ 1, abort, P.status)))
                        goto dq_done;
                    tc_fence_after();
                    const uint8_t* srow = meta + rm.s * L::kChunkBytes + r * 128;
                    uint32_t c[32];
                    const int a0 = (kb - KB) * kBK;
                    const bool fix = P.bf16 || a0 + kBK > D.A;
#pragma unroll
                    for (int q = 0; q < 8; ++q) {
                        const int off = (q ^ sw) << 4;
                        const uint4 u4 = *reinterpret_cast<const uint4*>(srow + off);
                        uint32_t v[4] = {u4.x, u4.y, u4.z, u4.w};
                        if (fix) {
#pragma unroll
                            for (int i = 0; i < 4; ++i) {
                                const int a = a0 + 8 * q + 2 * i;
                                uint32_t w = a < D.A ? v[i] : 0u;
                                if (a + 1 >= D.A) w &= 0xFFFFu;
                                if (P.bf16)
                                    w = pack2(half_bits_to_float((uint16_t)w), half_bits_to_float((uint16_t)(w >> 16)), 1);
                                v[i] = w;
                            }
                        }
                        c[4 * q] = v[0];
                        c[4 * q + 1] = v[1];
                        c[4 * q + 2] = v[2];
                        c[4 * q + 3] = v[3];
                    }
                    tmem_st32(a_lane + 32 * ra.s, c);
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive_remote(full_r0 + 8 * ra.s);
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(m_empty0 + 8 * rm.s);
                rm.next(kMetaSlots);
            }
            ra.next(S);
          }
        }
        // every stage's last release has arrived before this CTA may exit
        if (warp == kDqWarp0)
            for (int s = 0; s < S; ++s) {
                if (!__all_sync(0xffffffffu, mbar_wait_bounded<true>(empty0 + 8 * ra.s, ra.ph ^ 1, abort, P.status)))
                    break;
                ra.next(S);
            }
    dq_done:;
    } else {
        // ---------------------------------------------------------------- epilogue: TMEM -> y
        // Each CTA holds its 128 rows of the pair's 256 x 256 accumulator.
        const int quarter = warp & 3;   // the TMEM lane quarter this warp may read
        constexpr int kCols = kBN * 4 / kEpiWarps;   // accumulator columns this warp drains
        const int c0 = kCols * ((warp - kEpiWarp0) >> 2);
        const uint32_t acc_empty_r0 = mapa_shared(acc_empty0, 0);
        for (int i = 0; i < ntiles; ++i) {
            const int gt = tile_id(P, i, pair, npair);
            const GemmProb& D = P.d[tile_prob(P, gt)];
            if (!__all_sync(0xffffffffu, mbar_wait_bounded<true>(acc_full0, i & 1, abort, P.status))) break;
            tc_fence_after();
            const int lt = gt - D.tile_begin;
            const int n0 = (lt / D.tiles_m) * kPairM + (int)rank * kBM, m0 = (lt % D.tiles_m) * kBN;
            const int n = n0 + 32 * quarter + lane;
#pragma unroll 1
            for (int cc = c0; cc < c0 + kCols && m0 + cc < D.M; cc += 32) {
                uint32_t v[32];
                tmem_ld32(tmem + ((uint32_t)(32 * quarter) << 16) + cc, v);
                if (n < D.N) {
                    const int mb = m0 + cc, mcount = min(32, D.M - mb);
                    const size_t o = (size_t)mb * D.N + n;
                    if (D.y_dtype == LQ_BF16) {
                        __nv_bfloat16* yp = static_cast<__nv_bfloat16*>(D.y) + o;
#pragma unroll
                        for (int j = 0; j < 32; ++j)
                            if (j < mcount) yp[(size_t)j * D.N] = __float2bfloat16_rn(__uint_as_float(v[j]));
                    } else if (D.y_dtype == LQ_F16) {
                        __half* yp = static_cast<__half*>(D.y) + o;
#pragma unroll
                        for (int j = 0; j < 32; ++j)
                            if (j < mcount) yp[(size_t)j * D.N] = __float2half_rn(__uint_as_float(v[j]));
                    } else {
                        float* yp = static_cast<float*>(D.y) + o;
#pragma unroll
                        for (int j = 0; j < 32; ++j)
                            if (j < mcount) yp[(size_t)j * D.N] = __uint_as_float(v[j]);
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_remote(acc_empty_r0);
        }
    }
    tc_fence_before();
    __syncwarp();
    cluster_sync_all();   // no arrival or tensor-memory access of either CTA is still to come
    tc_fence_after();
    if (warp == 1) tmem_dealloc_pair(tmem, kTmemCols);
}

// x gathered at the anchor columns ([M][a_pad], zero past A) and the anchor bitmap of
// each problem (blockIdx.y); the bitmaps are cleared before this runs.
struct PrepProb {
    const uint16_t* x;
    const int32_t* anchor_idx;
    uint16_t* xa;
    unsigned long long* bits;
    int M, K, A, a_pad;
};

struct GemmPrepParams {
    PrepProb d[kMaxGemmGroup];
};

__global__ void __launch_bounds__(256) gemm_prep_kernel(const __grid_constant__ GemmPrepParams Q) {
    const PrepProb& D = Q.d[blockIdx.y];
    const int64_t total = (int64_t)D.M * D.a_pad;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total || i < D.A;
         i += (int64_t)gridDim.x * blockDim.x) {
        if (i < D.A) {
            const int k = D.anchor_idx[i];
            atomicOr(D.bits + (k >> 6), 1ull << (k & 63));
        }
        if (i < total) {
            const int m = (int)(i / D.a_pad), a = (int)(i - (int64_t)m * D.a_pad);
            D.xa[i] = a < D.A ? D.x[(int64_t)m * D.K + D.anchor_idx[a]] : (uint16_t)0;
        }
    }
}

// INT4 prefill: x in the permuted column order, xp[m][j] = x[m][perm[j]] (zero for a column
// outside [0, K)); one thread per 8 consecutive positions of a token.
__global__ void __launch_bounds__(256) gemm_permute_x_kernel(const uint16_t* __restrict__ x, const int32_t* __restrict__ perm,
                                                             uint16_t* __restrict__ xp, int M, int K) {
    const int64_t n8 = (int64_t)M * (K / 8);
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n8; i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t m = i / (K / 8);
        const int j0 = (int)(i - m * (K / 8)) * 8;
        const int4 c0 = __ldg(reinterpret_cast<const int4*>(perm + j0)), c1 = __ldg(reinterpret_cast<const int4*>(perm + j0 + 4));
        const int cols[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
        uint32_t v[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int a = cols[2 * e], b = cols[2 * e + 1];
            const uint32_t lo = (unsigned)a < (unsigned)K ? x[m * K + a] : 0u, hi = (unsigned)b < (unsigned)K ? x[m * K + b] : 0u;
            v[e] = lo | (hi << 16);
        }
        *reinterpret_cast<uint4*>(xp + m * K + j0) = make_uint4(v[0], v[1], v[2], v[3]);
    }
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn_g() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        cudaDriverEntryPointQueryResult q;
        void* p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// 2-D tiled map over a row-major [rows][cols] matrix with a row pitch of `ld` elements.
bool map_2d(CUtensorMap* m, CUtensorMapDataType dt, int esize, const void* base, uint64_t cols, uint64_t rows,
            uint64_t ld, uint32_t box_cols, uint32_t box_rows, CUtensorMapSwizzle swz) {
    auto fn = encode_fn_g();
    if (!fn) return false;
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {ld * (uint64_t)esize};
    cuuint32_t box[2] = {box_cols, box_rows};
    cuuint32_t estr[2] = {1, 1};
    return fn(m, dt, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool map_16bit(CUtensorMap* m, const void* base, uint64_t cols, uint64_t rows, uint64_t ld, uint32_t box_rows) {
    return map_2d(m, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, base, cols, rows, ld, kBK, box_rows, CU_TENSOR_MAP_SWIZZLE_128B);
}

// CTA pairs of gemm_kernel<FMT> that fit on the device at once (0 on error); the first call
// sets the kernel's shared-memory attribute.  Cached per format and device.
template <int FMT>
int pair_capacity(int device) {
    static std::mutex mu;
    static std::vector<int> cache;
    std::lock_guard<std::mutex> lock(mu);
    if ((int)cache.size() <= device) cache.resize(device + 1, -1);
    if (cache[device] >= 0) return cache[device];
    constexpr int smem = GemmLayout<FMT>::kSmemBytes;
    int n = 0;
    if (cudaFuncSetAttribute(gemm_kernel<FMT>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) == cudaSuccess) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(2, 1, 1);
        cfg.blockDim = dim3(GemmLayout<FMT>::kThreads, 1, 1);
        cfg.dynamicSmemBytes = smem;
        if (cudaOccupancyMaxActiveClusters(&n, gemm_kernel<FMT>, &cfg) != cudaSuccess) n = 0;
    }
    cudaGetLastError();
    cache[device] = n;
    return n;
}

template <int FMT>
lq_status launch_fmt(const GemmParams& P, int npair, cudaStream_t stream) {
    constexpr int smem = GemmLayout<FMT>::kSmemBytes;
    gemm_kernel<FMT><<<2 * npair, GemmLayout<FMT>::kThreads, smem, stream>>>(P);   // (compile-time clusters of two)
    return cudaPeekAtLastError() == cudaSuccess ? LQ_OK : LQ_ERR_CUDA;
}

}  // namespace

// Longest-processing-time assignment of the launch's tiles to `grid` CTA pairs (each tile
// costs its K-blocks), as per-pair lists; kept on the device between calls with the same shapes.
static lq_status upload_schedule(lq_handle h, const GemmParams& P, int grid, cudaStream_t stream) {
    std::vector<int64_t> key = {grid, P.count};
    for (int p = 0; p < P.count; ++p) {
        const GemmProb& D = P.d[p];
        key.insert(key.end(), {D.M, D.N, D.K, D.a_pad, D.tiles_m});
    }
    if (key == h->sched_key) return LQ_OK;
    struct Job {
        int cost, tile;
    };
    std::vector<Job> jobs;
    jobs.reserve(P.total_tiles);
    for (int p = 0; p < P.count; ++p) {
        const GemmProb& D = P.d[p];
        const int ntl = (p + 1 < P.count ? P.d[p + 1].tile_begin : P.total_tiles) - D.tile_begin;
        for (int t = 0; t < ntl; ++t) jobs.push_back({D.K / kBK + D.a_pad / kBK, D.tile_begin + t});
    }
    std::stable_sort(jobs.begin(), jobs.end(), [](const Job& a, const Job& b) { return a.cost > b.cost; });
    std::vector<std::vector<int>> lists(grid);
    std::vector<std::pair<int64_t, int>> heap;   // (load, cta), min-heap
    for (int b = 0; b < grid; ++b) heap.push_back({0, b});
    auto cmp = [](const std::pair<int64_t, int>& a, const std::pair<int64_t, int>& b) { return a > b; };
    std::make_heap(heap.begin(), heap.end(), cmp);
    for (const Job& j : jobs) {
        std::pop_heap(heap.begin(), heap.end(), cmp);
        heap.back().first += j.cost;
        lists[heap.back().second].push_back(j.tile);
        std::push_heap(heap.begin(), heap.end(), cmp);
    }
    std::vector<int> flat(grid + 1);
    for (int b = 0; b < grid; ++b) flat[b + 1] = flat[b] + (int)lists[b].size();
    for (int b = 0; b < grid; ++b) flat.insert(flat.end(), lists[b].begin(), lists[b].end());
    if (flat.size() > h->sched_ints) return LQ_ERR_WORKSPACE;
    if (cudaMemcpyAsync(h->sched, flat.data(), flat.size() * sizeof(int), cudaMemcpyHostToDevice, stream) != cudaSuccess ||
        cudaStreamSynchronize(stream) != cudaSuccess)
        return LQ_ERR_CUDA;
    h->sched_key = key;
    return LQ_OK;
}

lq_status launch_gemm_grouped_limited(lq_handle h, const lq_problem* probs, int count, cudaStream_t stream,
                                      size_t ws_bytes);

// NF4 with double quantization, prefill: the block maxima decoded once into fp32 (one
// fmaf each, as the decode kernels do in registers), then the NF4 GEMM reads them.
__global__ void __launch_bounds__(256) nf4_dq_decode_kernel(const uint8_t* __restrict__ acodes,
                                                            const float* __restrict__ second, float* __restrict__ out,
                                                            int64_t n) {
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x)
        out[i] = nf4_dq_absmax(acodes, second, i);
}

lq_status launch_gemm_grouped(lq_handle h, const lq_problem* probs, int count, cudaStream_t stream) {
    if (count < 1 || count > kMaxGemmGroup) return LQ_ERR_UNSUPPORTED;
    if (probs[0].format == LQ_FMT_NF4_DQ) {
        // decode each problem's maxima into the workspace's tail, then run the NF4 GEMM on copies of
        // the problems that point there
        lq_problem q[kMaxGemmGroup];
        size_t need = 0;
        for (int i = 0; i < count; ++i) {
            if (probs[i].format != LQ_FMT_NF4_DQ) return LQ_ERR_UNSUPPORTED;
            need += ((size_t)probs[i].N * (probs[i].K / 64) * 4 + 255) & ~size_t(255);
        }
        const size_t cap = h->partial_floats * sizeof(float);
        if (need + (size_t(1) << 20) > cap) return LQ_ERR_WORKSPACE;
        char* tail = reinterpret_cast<char*>(h->partials) + ((cap - need) & ~size_t(255));
        for (int i = 0; i < count; ++i) {
            q[i] = probs[i];
            const int64_t n = (int64_t)probs[i].N * (probs[i].K / 64);
            float* dec = reinterpret_cast<float*>(tail);
            tail += ((size_t)n * 4 + 255) & ~size_t(255);
            const int g = (int)std::min<int64_t>((n + 255) / 256, (int64_t)h->num_sms * 16);
            nf4_dq_decode_kernel<<<std::max(g, 1), 256, 0, stream>>>(static_cast<const uint8_t*>(probs[i].scales),
                                                                      static_cast<const float*>(probs[i].offsets), dec, n);
            if (cudaPeekAtLastError() != cudaSuccess) return LQ_ERR_CUDA;
            q[i].format = LQ_FMT_NF4_B64;
            q[i].scales = dec;
            q[i].offsets = nullptr;
        }
        return launch_gemm_grouped_limited(h, q, count, stream, (cap - need) & ~size_t(255));
    }
    return launch_gemm_grouped_limited(h, probs, count, stream, h->partial_floats * sizeof(float));
}

lq_status launch_gemm_grouped_limited(lq_handle h, const lq_problem* probs, int count, cudaStream_t stream,
                                      size_t ws_bytes) {
    GemmParams P;
    GemmPrepParams Q;
    memset(&P, 0, sizeof(P));
    memset(&Q, 0, sizeof(Q));
    const int fmt = probs[0].format;
    const bool nf4 = fmt == LQ_FMT_NF4_B64, int4 = fmt == LQ_FMT_INT4_G32;
    const bool nib = nf4 || int4;   // 4-bit codes
    struct PermJob {
        const uint16_t* x;
        const int32_t* perm;
        uint16_t* xp;
        int M, K;
    } perm_jobs[kMaxGemmGroup];
    int nperm = 0;
    P.count = count;
    P.bf16 = probs[0].x_dtype == LQ_BF16;
    P.status = h->status_flag;
    // workspace per problem: anchor bitmap [K/64 + 4] (a chunk past the last K-block is read whole),
    // all bitmaps first so one memset clears them, then x at the anchor columns [M][a_pad]
    char* ws = reinterpret_cast<char*>(h->partials);
    size_t used = 0, bits_total = 0;
    int tiles = 0, max_prep = 1, prep_count = 0;
    size_t bits_off[kMaxGemmGroup];
    for (int i = 0; i < count; ++i) {
        const lq_problem& p = probs[i];
        if (p.format != fmt || (p.x_dtype == LQ_BF16) != (P.bf16 != 0)) return LQ_ERR_UNSUPPORTED;
        bits_off[i] = bits_total;
        bits_total += ((size_t)(p.K / 64 + kChunk) * 8 + 255) & ~size_t(255);
    }
    used = bits_total;
    for (int i = 0; i < count; ++i) {
        const lq_problem& p = probs[i];
        GemmProb& D = P.d[i];
        const int A = nf4 ? 0 : p.A;
        const int a_pad = A > 0 ? (A + kBK - 1) / kBK * kBK : 0;
        D.scales = p.scales;
        D.offsets = int4 ? nullptr : static_cast<const uint16_t*>(p.offsets);
        D.y = p.y;
        D.M = p.M;
        D.N = p.N;
        D.K = p.K;
        D.A = A;
        D.a_pad = a_pad;
        D.y_dtype = p.y_dtype;
        D.meta_tma = p.K % 256 == 0;   // scale rows 16-byte aligned: TMA boxes; else 4-byte loads
        D.tiles_m = (p.M + kBN - 1) / kBN;
        D.tile_begin = tiles;
        const int64_t t = (int64_t)D.tiles_m * ((p.N + kPairM - 1) / kPairM);
        if (tiles + t > 0x7fffffffLL) return LQ_ERR_UNSUPPORTED;
        tiles += (int)t;
        unsigned long long* bits = reinterpret_cast<unsigned long long*>(ws + bits_off[i]);
        D.anchor_bits = reinterpret_cast<const uint32_t*>(bits);
        uint16_t* xa = reinterpret_cast<uint16_t*>(ws + used);
        used += ((size_t)p.M * a_pad * 2 + 255) & ~size_t(255);
        const void* xsrc = p.x;
        if (int4) {   // INT4: x in the weights' permuted column order, gathered once into the workspace
            uint16_t* xp = reinterpret_cast<uint16_t*>(ws + used);
            used += ((size_t)p.M * p.K * 2 + 255) & ~size_t(255);
            perm_jobs[nperm++] = PermJob{static_cast<const uint16_t*>(p.x), static_cast<const int32_t*>(p.offsets), xp, p.M,
                                         p.K};
            xsrc = xp;
        }
        if (!map_16bit(&D.xmap, xsrc, (uint64_t)p.K, (uint64_t)p.M, (uint64_t)p.K, kHalfN)) return LQ_ERR_CUDA;
        const uint64_t cbytes = (uint64_t)p.K / (nib ? 2 : 4);
        if (!map_2d(&D.cmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, p.codes, cbytes, (uint64_t)p.N, cbytes,
                    kChunk * (nib ? 32 : 16), kBM, nib ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B))
            return LQ_ERR_CUDA;
        if (D.meta_tma) {
            if (nf4) {
                if (!map_2d(&D.smap, CU_TENSOR_MAP_DATA_TYPE_UINT32, 4, p.scales, (uint64_t)p.K / 64, (uint64_t)p.N,
                            (uint64_t)p.K / 64, 4, kBM, CU_TENSOR_MAP_SWIZZLE_NONE))
                    return LQ_ERR_CUDA;
            } else {
                if (!map_2d(&D.smap, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, p.scales, (uint64_t)p.K / 32, (uint64_t)p.N,
                            (uint64_t)p.K / 32, 8, kBM, CU_TENSOR_MAP_SWIZZLE_NONE))
                    return LQ_ERR_CUDA;
                if (!int4 && !map_2d(&D.omap, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, p.offsets, (uint64_t)p.K / 32,
                                     (uint64_t)p.N, (uint64_t)p.K / 32, 8, kBM, CU_TENSOR_MAP_SWIZZLE_NONE))
                    return LQ_ERR_CUDA;
            }
        }
        if (A > 0) {
            if (!map_16bit(&D.xamap, xa, (uint64_t)a_pad, (uint64_t)p.M, (uint64_t)a_pad, kHalfN)) return LQ_ERR_CUDA;
            if (!map_16bit(&D.awmap, p.anchor_w, (uint64_t)p.ld_anchor, (uint64_t)p.N, (uint64_t)p.ld_anchor, kBM))
                return LQ_ERR_CUDA;
            PrepProb& e = Q.d[prep_count++];
            e.x = static_cast<const uint16_t*>(p.x);
            e.anchor_idx = p.anchor_idx;
            e.xa = xa;
            e.bits = bits;
            e.M = p.M;
            e.K = p.K;
            e.A = A;
            e.a_pad = a_pad;
            max_prep = (int)std::max<int64_t>(max_prep, std::max<int64_t>((int64_t)p.M * a_pad, A));
        }
    }
    if (used + 256 > ws_bytes) return LQ_ERR_WORKSPACE;
    P.total_tiles = tiles;
    if (tiles == 0) return LQ_OK;
    if (prep_count > 0) {
        if (cudaMemsetAsync(ws, 0, bits_total, stream) != cudaSuccess) return LQ_ERR_CUDA;
        const int gx = (int)std::min<int64_t>((max_prep + 255) / 256, (int64_t)h->num_sms * 8);
        gemm_prep_kernel<<<dim3(gx, prep_count), 256, 0, stream>>>(Q);
        if (cudaPeekAtLastError() != cudaSuccess) return LQ_ERR_CUDA;
    }
    for (int i = 0; i < nperm; ++i) {
        const PermJob& jb = perm_jobs[i];
        const int64_t n8 = (int64_t)jb.M * (jb.K / 8);
        const int g = (int)std::min<int64_t>((n8 + 255) / 256, (int64_t)h->num_sms * 16);
        gemm_permute_x_kernel<<<std::max(g, 1), 256, 0, stream>>>(jb.x, jb.perm, jb.xp, jb.M, jb.K);
        if (cudaPeekAtLastError() != cudaSuccess) return LQ_ERR_CUDA;
    }
    const int smem = nf4    ? GemmLayout<LQ_FMT_NF4_B64>::kSmemBytes
                     : int4 ? GemmLayout<LQ_FMT_INT4_G32>::kSmemBytes
                            : GemmLayout<LQ_FMT_2BIT_LM_G32>::kSmemBytes;
    if (smem > h->max_smem_optin) return LQ_ERR_UNSUPPORTED;
    const int cap = nf4 ? pair_capacity<LQ_FMT_NF4_B64>(h->device)
                    : int4 ? pair_capacity<LQ_FMT_INT4_G32>(h->device)
                           : pair_capacity<LQ_FMT_2BIT_LM_G32>(h->device);
    if (cap < 1) return LQ_ERR_UNSUPPORTED;
    const int npair = std::min(tiles, cap);
    if (count > 1) {
        // problems of different lengths: balance the pairs' K-blocks
        const lq_status s = upload_schedule(h, P, npair, stream);
        if (s != LQ_OK) return s;
        P.sched_off = h->sched;
        P.sched_tiles = h->sched + npair + 1;
    }
    if (nf4) return launch_fmt<LQ_FMT_NF4_B64>(P, npair, stream);
    if (int4) return launch_fmt<LQ_FMT_INT4_G32>(P, npair, stream);
    return launch_fmt<LQ_FMT_2BIT_LM_G32>(P, npair, stream);
}

lq_status launch_gemm(lq_handle h, const lq_problem& p, cudaStream_t stream) { return launch_gemm_grouped(h, &p, 1, stream); }

}  // namespace lq
