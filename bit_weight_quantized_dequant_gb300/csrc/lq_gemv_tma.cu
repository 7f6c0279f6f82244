// TMA-fed, warp-specialised decode GEMV (the fast path of lq_gemv / lq_gemv_grouped).
//
// Decode streams every weight once per token (otf-llm 4.0.1 README, section 1,
// "The Memory-Bound Bottleneck"), so the kernel's job is to keep HBM busy while
// the SMs dequantize in registers (section 3 reconstruction, section 4 anchors):
//
//  * A tiny pre-pass kernel writes x once per call as binary16, anchor columns
//    zeroed (the anchors replace those weights), in mma-fragment order, plus x
//    gathered at the anchor columns.  It triggers programmatic dependent launch,
//    so the main kernel's prologue overlaps it.
//  * The main kernel is persistent: two CTAs per SM claim work units (128 rows x
//    one K-split, or x one anchor split) from an atomic counter.
//  * Warp 8 is the producer: one thread issues TMA tile loads (codes 128 rows x
//    128 bytes with the 128-byte swizzle, the 128 x 16 scale and offset tiles, or
//    128 x 64 binary16 anchor weights) into a 4-stage shared-memory ring, and one
//    bulk copy of the unit's x slice into a double-buffered x slot.  All copies
//    complete on mbarriers; nothing is held in registers while in flight.
//  * Warps 0-7 are consumers, 16 rows each.  Dequantization is a PRMT lookup in
//    byte-split binary16 tables, the multiply-accumulate is mma.sync m16n8k16
//    (binary16 in, fp32 accumulate) with tokens as the n dimension.
//  * Split-K partials go to the workspace; the last unit of a 128-row strip sums
//    them in a fixed order.  Every mbarrier wait is bounded in time; a wait that
//    runs out raises a status flag and the CTA unwinds.

#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstring>
#include <mutex>

#include "lq_common.cuh"
#include "lq_dq.cuh"
#include "lq_internal.h"
#include "lq_tma.cuh"

namespace lq {
namespace {

constexpr int kRows = 128;               // rows per unit
constexpr int kCWarps = 8;               // consumer warps (16 rows each)
constexpr int kThreadsT = (kCWarps + 2) * 32;   // consumers, producer, epilogue
constexpr int kMaxStages = 4;
constexpr int kStageBytes = 24576;
constexpr int kScalesOff = 16384;        // 2-bit scales tile (128 x 32 B) / NF4 absmax tile (128 x 16 B)
constexpr int kOffsetsOff = 20480;       // 2-bit offsets tile (128 x 32 B)
constexpr int kSC2 = 512;                // K columns per 2-bit code stage
constexpr int kSCNF4 = 256;              // K columns per NF4 code stage
constexpr int kSCA = 64;                 // anchors per anchor stage

struct Maps {
    CUtensorMap codes, scales, offsets, anchors;
};

struct Desc {
    const uint16_t* xperm;       // [batch][Kp/16][M][16] binary16
    const uint16_t* xaperm;      // [batch][a_pad/16][M][16] binary16
    int64_t xperm_stride, xaperm_stride;   // halves per batch member
    void* y;
    int64_t stride_y;
    int N, K, A, batch, Kp, a_pad;
    int KC, S, KA, Sa, parts, merged, strips;
    int64_t unit_begin, strip_begin, partial_begin;
};

struct Params {
    Maps maps[kMaxGroup];
    Desc d[kMaxGroup];
    int count, M, y_dtype, format, x_slot_halves, nstages;
    int64_t total_units;
    float* partials;
    unsigned* counters;   // split-K arrival counters (one per strip)
    unsigned* sched;      // [0] next unit, [1] CTAs done
    int* status;
};

struct Unit {
    int p;
    int64_t l;
    int strip, part;
    int k0, klen;         // code columns (klen = 0: none)
    int a0, alen;         // anchors (alen = 0: none)
};

__device__ __forceinline__ Unit decode_unit(const Params& P, int64_t u) {
    Unit U;
    int p = 0;
    while (p + 1 < P.count && u >= P.d[p + 1].unit_begin) ++p;
    const Desc& D = P.d[p];
    U.p = p;
    const int64_t local = u - D.unit_begin;
    const int64_t per_member = (int64_t)D.strips * D.parts;
    U.l = local / per_member;
    const int rem = (int)(local - U.l * per_member);
    U.strip = rem / D.parts;
    U.part = rem - U.strip * D.parts;
    U.k0 = U.klen = U.a0 = U.alen = 0;
    if (D.merged) {
        U.klen = D.K;
        U.alen = D.A;
    } else if (U.part < D.S) {
        U.k0 = U.part * D.KC;
        U.klen = min(D.KC, D.K - U.k0);
    } else {
        U.a0 = (U.part - D.S) * D.KA;
        U.alen = min(D.KA, D.A - U.a0);
    }
    return U;
}

__device__ __forceinline__ int round_up_d(int a, int b) { return (a + b - 1) / b * b; }

__device__ __forceinline__ uint4 lds128(const uint8_t* p) { return *reinterpret_cast<const uint4*>(p); }
__device__ __forceinline__ uint2 lds64u(const void* p) { return *reinterpret_cast<const uint2*>(p); }
__device__ __forceinline__ uint32_t lds32(const void* p) { return *reinterpret_cast<const uint32_t*>(p); }

template <int NT>
__device__ __forceinline__ void mma_x(float (&acc)[NT][4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                      const uint16_t* xb, int bi, int M, int g, int t) {
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        uint2 b = make_uint2(0u, 0u);
        if (8 * nt + g < M) b = lds64u(xb + ((bi * M) + 8 * nt + g) * 16 + t * 4);
        mma_f16_16816(acc[nt], a0, a1, a2, a3, b.x, b.y);
    }
}

// One 2-bit code stage: 128 rows x 512 columns (steps of 256 beyond `steps` are skipped).
template <int NT>
__device__ __forceinline__ void stage_2bit(const uint8_t* tile, const uint16_t* xb, int steps, int M, int w, int g,
                                           int t, float (&acc)[NT][4]) {
    const int r0 = 16 * w + g, r1 = r0 + 8;
    const uint16_t* sc = reinterpret_cast<const uint16_t*>(tile + kScalesOff);
    const uint16_t* of = reinterpret_cast<const uint16_t*>(tile + kOffsetsOff);
#pragma unroll
    for (int s = 0; s < 2; ++s) {
        if (s >= steps) break;
        const int chunk = ((4 * s + t) ^ g) << 4;
        const uint4 c0 = lds128(tile + r0 * 128 + chunk);
        const uint4 c1 = lds128(tile + r1 * 128 + chunk);
        const uint32_t s0 = lds32(sc + r0 * 16 + 8 * s + 2 * t), z0 = lds32(of + r0 * 16 + 8 * s + 2 * t);
        const uint32_t s1 = lds32(sc + r1 * 16 + 8 * s + 2 * t), z1 = lds32(of + r1 * 16 + 8 * s + 2 * t);
        uint32_t RA[4], RB[4];
        lut2_bits((uint16_t)s0, (uint16_t)z0, RA[0], RB[0]);
        lut2_bits((uint16_t)(s0 >> 16), (uint16_t)(z0 >> 16), RA[1], RB[1]);
        lut2_bits((uint16_t)s1, (uint16_t)z1, RA[2], RB[2]);
        lut2_bits((uint16_t)(s1 >> 16), (uint16_t)(z1 >> 16), RA[3], RB[3]);
        const uint32_t wg[4] = {c0.x, c0.y, c0.z, c0.w};
        const uint32_t wg8[4] = {c1.x, c1.y, c1.z, c1.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int lg = i >> 1;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                uint32_t a0, a1, a2, a3;
                expand2_fast(wg[i], j, RA[lg], RB[lg], a0, a2);
                expand2_fast(wg8[i], j, RA[2 + lg], RB[2 + lg], a1, a3);
                mma_x<NT>(acc, a0, a1, a2, a3, xb, s * 16 + i * 4 + j, M, g, t);
            }
        }
    }
}

// One NF4 code stage: 128 rows x 256 columns = 4 blocks of 64 with their absmax.
template <int NT>
__device__ __forceinline__ void stage_nf4(const uint8_t* tile, const uint16_t* xb, int M, int w, int g, int t,
                                          const uint32_t (&TL)[4], const uint32_t (&TH)[4], float (&acc)[NT][4]) {
    const int r0 = 16 * w + g, r1 = r0 + 8;
    const float* am = reinterpret_cast<const float*>(tile + kScalesOff);
#pragma unroll
    for (int nb = 0; nb < 4; ++nb) {
        const int off = (((2 * nb + (t >> 1)) ^ g) << 4) + ((t & 1) << 3);
        const uint2 cw0 = lds64u(tile + r0 * 128 + off);
        const uint2 cw1 = lds64u(tile + r1 * 128 + off);
        const float am0 = am[r0 * 4 + nb], am1 = am[r1 * 4 + nb];
        float part[NT][4];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) part[nt][0] = part[nt][1] = part[nt][2] = part[nt][3] = 0.f;
#pragma unroll
        for (int b = 0; b < 4; ++b) {
            uint32_t a0, a1, a2, a3;
            expand_nf4_fast(b < 2 ? cw0.x : cw0.y, b & 1, TL, TH, a0, a2);
            expand_nf4_fast(b < 2 ? cw1.x : cw1.y, b & 1, TL, TH, a1, a3);
            mma_x<NT>(part, a0, a1, a2, a3, xb, nb * 4 + b, M, g, t);
        }
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            acc[nt][0] = __fmaf_rn(am0, part[nt][0], acc[nt][0]);
            acc[nt][1] = __fmaf_rn(am0, part[nt][1], acc[nt][1]);
            acc[nt][2] = __fmaf_rn(am1, part[nt][2], acc[nt][2]);
            acc[nt][3] = __fmaf_rn(am1, part[nt][3], acc[nt][3]);
        }
    }
}

// One anchor stage: 128 rows x 64 binary16 anchor weights (128-byte swizzle).
template <int NT>
__device__ __forceinline__ void stage_anchor(const uint8_t* tile, const uint16_t* xb, int M, int w, int g, int t,
                                             float (&acc)[NT][4]) {
    const int r0 = 16 * w + g, r1 = r0 + 8;
#pragma unroll
    for (int ab = 0; ab < 4; ++ab) {
        const int lo = (((2 * ab) ^ g) << 4) + 4 * t, hi = (((2 * ab + 1) ^ g) << 4) + 4 * t;
        const uint32_t a0 = lds32(tile + r0 * 128 + lo), a2 = lds32(tile + r0 * 128 + hi);
        const uint32_t a1 = lds32(tile + r1 * 128 + lo), a3 = lds32(tile + r1 * 128 + hi);
        mma_x<NT>(acc, a0, a1, a2, a3, xb, ab, M, g, t);
    }
}

template <int NT, int FMT>
__global__ void __launch_bounds__(kThreadsT, 2) gemv_tma_kernel(const __grid_constant__ Params P) {
    extern __shared__ uint8_t smem_raw[];
    const int NS = P.nstages, M = P.M;
    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* stages = base;
    uint16_t* xslots = reinterpret_cast<uint16_t*>(base + NS * kStageBytes);
    float* epi = reinterpret_cast<float*>(xslots + 2 * P.x_slot_halves);          // [2][M][kRows]
    uint64_t* bars = reinterpret_cast<uint64_t*>(epi + 2 * M * kRows);
    // bars: full[NS], empty[NS], xfull[2], xempty[2], efull[2], eempty[2]
    __shared__ long long s_unit[2];
    __shared__ long long s_eunit[2];
    __shared__ int s_abort;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t full0 = smem_u32(bars), empty0 = smem_u32(bars + NS);
    const uint32_t xfull0 = smem_u32(bars + 2 * NS), xempty0 = xfull0 + 16;
    const uint32_t efull0 = xfull0 + 32, eempty0 = xfull0 + 48;

    if (tid == 0) {
        for (int s = 0; s < NS; ++s) {
            mbar_init(full0 + 8 * s, 1);
            mbar_init(empty0 + 8 * s, kCWarps);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(xfull0 + 8 * s, 1);
            mbar_init(xempty0 + 8 * s, kCWarps);
            mbar_init(efull0 + 8 * s, kCWarps);
            mbar_init(eempty0 + 8 * s, 1);
        }
        s_abort = 0;
        fence_mbar_init();
    }
    __syncthreads();
    constexpr int SC = FMT == LQ_FMT_2BIT_LM_G32 ? kSC2 : kSCNF4;
    // Every thread gives up only on its own timeout: all threads of a role wait on the
    // same barriers in the same order, so they stop at the same place.
    int own_abort = 0;
    volatile int* abort = &own_abort;

    if (warp == kCWarps) {
        // ------------------------------------------------------------ producer (TMA)
        if (lane == 0) {
            for (int i = 0; i < P.count; ++i) {
                prefetch_tensormap(&P.maps[i].codes);
                prefetch_tensormap(&P.maps[i].scales);
                if (FMT == LQ_FMT_2BIT_LM_G32) {
                    prefetch_tensormap(&P.maps[i].offsets);
                    if (P.d[i].A > 0) prefetch_tensormap(&P.maps[i].anchors);
                }
            }
            int xs = 0, xph = 0, slot = 0, ph = 0;
            bool ok = true, first = true;
            // weight tiles of stage `idx` of unit U (code stages first, then anchor stages)
            auto issue_stage = [&](const Unit& U, int idx) -> bool {
                if (!mbar_wait_bounded(empty0 + 8 * slot, ph ^ 1, abort, P.status)) return false;
                const uint32_t dst = smem_u32(stages + slot * kStageBytes), fb = full0 + 8 * slot;
                const int row0 = U.strip * kRows;
                const int nst = (U.klen + SC - 1) / SC;
                if (idx < nst) {
                    const int col = U.k0 + idx * SC;
                    if (FMT == LQ_FMT_2BIT_LM_G32) {
                        mbar_arrive_expect_tx(fb, 16384 + 4096 + 4096);
                        tma_load_3d(dst, &P.maps[U.p].codes, col / 4, row0, (int)U.l, fb);
                        tma_load_3d(dst + kScalesOff, &P.maps[U.p].scales, col / 32, row0, (int)U.l, fb);
                        tma_load_3d(dst + kOffsetsOff, &P.maps[U.p].offsets, col / 32, row0, (int)U.l, fb);
                    } else {
                        mbar_arrive_expect_tx(fb, 16384 + 2048);
                        tma_load_3d(dst, &P.maps[U.p].codes, col / 2, row0, (int)U.l, fb);
                        tma_load_3d(dst + kScalesOff, &P.maps[U.p].scales, col / 64, row0, (int)U.l, fb);
                    }
                } else {
                    mbar_arrive_expect_tx(fb, 16384);
                    tma_load_3d(dst, &P.maps[U.p].anchors, U.a0 + (idx - nst) * kSCA, row0, (int)U.l, fb);
                }
                if (++slot == NS) {
                    slot = 0;
                    ph ^= 1;
                }
                return true;
            };
            while (ok) {
                const unsigned claimed = atomicAdd(P.sched, 1u);
                const int64_t u = (int64_t)claimed < P.total_units ? (int64_t)claimed : -1;
                if (!(ok = mbar_wait_bounded(xempty0 + 8 * xs, xph ^ 1, abort, P.status))) break;
                s_unit[xs] = u;
                if (u < 0) {
                    mbar_arrive(xfull0 + 8 * xs);
                    break;
                }
                const Unit U = decode_unit(P, u);
                const Desc& D = P.d[U.p];
                const int total = (U.klen + SC - 1) / SC + (U.alen + kSCA - 1) / kSCA;
                // the first unit's weight tiles do not depend on x: start them before waiting
                // for the x pre-pass (at most a ring's worth, the consumers need x to drain it)
                const int pre = first ? min(total, NS) : 0;
                for (int i = 0; i < pre && ok; ++i) ok = issue_stage(U, i);
                if (!ok) break;
                if (first) {
                    pdl_wait();
                    first = false;
                }
                const uint32_t code_b = (uint32_t)(M * round_up_d(U.klen, 256) * 2);
                const uint32_t anch_b = (uint32_t)(M * round_up_d(U.alen, kSCA) * 2);
                const uint32_t xdst = smem_u32(xslots + (size_t)xs * P.x_slot_halves);
                mbar_arrive_expect_tx(xfull0 + 8 * xs, code_b + anch_b);
                if (code_b)
                    bulk_load(xdst, D.xperm + U.l * D.xperm_stride + (int64_t)(U.k0 / 16) * M * 16, code_b,
                              xfull0 + 8 * xs);
                if (anch_b)
                    bulk_load(xdst + (D.merged ? (uint32_t)(M * D.Kp * 2) : 0u),
                              D.xaperm + U.l * D.xaperm_stride + (int64_t)(U.a0 / 16) * M * 16, anch_b,
                              xfull0 + 8 * xs);
                xs ^= 1;
                if (xs == 0) xph ^= 1;
                for (int i = pre; i < total && ok; ++i) ok = issue_stage(U, i);
            }
            if (!ok) {
                // unwinding after a timeout: let the copies already issued land (bounded)
                for (int s = 0; s < NS; ++s) {
                    const unsigned long long t0 = global_timer_ns();
                    while (!mbar_try_wait(full0 + 8 * s, 0) && !mbar_try_wait(full0 + 8 * s, 1) &&
                           global_timer_ns() - t0 < 100000000ull) {
                    }
                }
            }
            // the last CTA to finish resets the scheduler for the next launch
            __threadfence();
            if (atomicAdd(P.sched + 1, 1u) == gridDim.x - 1) {
                atomicExch(P.sched, 0u);
                atomicExch(P.sched + 1, 0u);
            }
        }
        return;
    }

    if (warp == kCWarps + 1) {
        // ------------------------------------------------------------ epilogue warp
        int eb = 0, eph = 0;
        for (;;) {
            if (!mbar_wait_bounded(efull0 + 8 * eb, eph, abort, P.status)) break;
            const int64_t u = s_eunit[eb];
            if (u < 0) break;
            const Unit U = decode_unit(P, u);
            const Desc& D = P.d[U.p];
            const float* acc = epi + (size_t)eb * M * kRows;
            const int N = D.N;
            void* y = static_cast<char*>(D.y) + U.l * D.stride_y;
            if (D.parts == 1) {
                for (int idx = lane; idx < M * kRows; idx += 32) {
                    const int m = idx / kRows, r = idx - m * kRows, n = U.strip * kRows + r;
                    if (n < N) store_out(y, (size_t)m * N + n, P.y_dtype, acc[idx]);
                }
            } else {
                const int64_t strip_id = D.strip_begin + U.l * D.strips + U.strip;
                float* strip_base = P.partials + D.partial_begin + (U.l * D.strips + U.strip) * (int64_t)D.parts * M * kRows;
                float* mine = strip_base + (int64_t)U.part * M * kRows;
                for (int idx = lane; idx < M * kRows; idx += 32) mine[idx] = acc[idx];
                __threadfence();
                __syncwarp();
                unsigned last = 0;
                if (lane == 0) last = atomicAdd(P.counters + strip_id, 1u) == (unsigned)(D.parts - 1);
                last = __shfl_sync(0xffffffffu, last, 0);
                if (last) {
                    __threadfence();
                    for (int idx = lane; idx < M * kRows; idx += 32) {
                        const int m = idx / kRows, r = idx - m * kRows, n = U.strip * kRows + r;
                        if (n >= N) continue;
                        float sum = 0.f;
                        for (int pp = 0; pp < D.parts; ++pp) sum += __ldcg(strip_base + (int64_t)pp * M * kRows + idx);
                        store_out(y, (size_t)m * N + n, P.y_dtype, sum);
                    }
                    if (lane == 0) P.counters[strip_id] = 0u;
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(eempty0 + 8 * eb);
            eb ^= 1;
            if (eb == 0) eph ^= 1;
        }
        return;
    }

    // ---------------------------------------------------------------- consumers
    const int g = lane >> 2, t = lane & 3;
    uint32_t TL[4], TH[4];
    if (FMT == LQ_FMT_NF4_B64) nf4_tables(TL, TH);
    int xs = 0, xph = 0, slot = 0, ph = 0, eb = 0, eph = 0;
    for (;;) {
        if (!mbar_wait_bounded(xfull0 + 8 * xs, xph, abort, P.status)) break;
        const int64_t u = s_unit[xs];
        if (u < 0) {
            // tell the epilogue warp there is no more work
            if (!mbar_wait_bounded(eempty0 + 8 * eb, eph ^ 1, abort, P.status)) break;
            if (tid == 0) s_eunit[eb] = -1;
            __syncwarp();
            if (lane == 0) mbar_arrive(efull0 + 8 * eb);
            break;
        }
        const Unit U = decode_unit(P, u);
        const Desc& D = P.d[U.p];
        const uint16_t* xb = xslots + (size_t)xs * P.x_slot_halves;
        float acc[NT][4];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;
        bool ok = true;
        const int nst = (U.klen + SC - 1) / SC;
        for (int st = 0; st < nst; ++st) {
            if (!(ok = mbar_wait_bounded(full0 + 8 * slot, ph, abort, P.status))) break;
            const uint8_t* tile = stages + slot * kStageBytes;
            if (FMT == LQ_FMT_2BIT_LM_G32) {
                const int steps = min(2, (U.klen - st * SC + 255) / 256);
                stage_2bit<NT>(tile, xb + (st * (SC / 16)) * M * 16, steps, M, warp, g, t, acc);
            } else {
                stage_nf4<NT>(tile, xb + (st * (SC / 16)) * M * 16, M, warp, g, t, TL, TH, acc);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(empty0 + 8 * slot);
            if (++slot == NS) {
                slot = 0;
                ph ^= 1;
            }
        }
        const int nas = ok ? (U.alen + kSCA - 1) / kSCA : 0;
        const uint16_t* xa = xb + (D.merged ? M * D.Kp : 0);
        for (int st = 0; st < nas; ++st) {
            if (!(ok = mbar_wait_bounded(full0 + 8 * slot, ph, abort, P.status))) break;
            stage_anchor<NT>(stages + slot * kStageBytes, xa + st * 4 * M * 16, M, warp, g, t, acc);
            __syncwarp();
            if (lane == 0) mbar_arrive(empty0 + 8 * slot);
            if (++slot == NS) {
                slot = 0;
                ph ^= 1;
            }
        }
        if (!ok) break;
        __syncwarp();
        if (lane == 0) mbar_arrive(xempty0 + 8 * xs);
        xs ^= 1;
        if (xs == 0) xph ^= 1;

        // ---- hand the accumulators to the epilogue warp
        if (!mbar_wait_bounded(eempty0 + 8 * eb, eph ^ 1, abort, P.status)) break;
        float* out = epi + (size_t)eb * M * kRows;
        const int r = 16 * warp + g;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            const int m0 = 8 * nt + 2 * t, m1 = m0 + 1;
            if (m0 < M) {
                out[m0 * kRows + r] = acc[nt][0];
                out[m0 * kRows + r + 8] = acc[nt][2];
            }
            if (m1 < M) {
                out[m1 * kRows + r] = acc[nt][1];
                out[m1 * kRows + r + 8] = acc[nt][3];
            }
        }
        if (tid == 0) s_eunit[eb] = u;
        __syncwarp();
        if (lane == 0) mbar_arrive(efull0 + 8 * eb);
        eb ^= 1;
        if (eb == 0) eph ^= 1;
    }
}

// ---- pre-pass: x -> binary16, anchors zeroed, fragment order ------------------------

struct PrepDesc {
    const uint16_t* x;
    int64_t stride_x;          // bytes
    const int32_t* anchor_idx;
    int64_t stride_anchor_idx; // bytes
    uint16_t* xperm;
    uint16_t* xaperm;
    int64_t xperm_stride, xaperm_stride;   // halves
    int K, Kp, A, a_pad, batch;
    int64_t work_begin;        // first work item (8 halves) of this problem in pass 1
    int64_t anchor_begin;      // first work item (one anchor of one token) in pass 2
};

struct PrepParams {
    PrepDesc d[kMaxGroup];
    int count, M, x_bf16, format;
    int64_t total, total_anchor;
};

__device__ __forceinline__ uint16_t to_half_bits(uint16_t raw, int x_bf16) {
    return x_bf16 ? __half_as_ushort(__float2half_rn(bf16_bits_to_float(raw))) : raw;
}

// Pass 1, output-major: each thread writes 8 consecutive binary16 of the fragment-ordered
// copy of x (one 16-byte store), gathering its 8 source columns from the x row.
__global__ void __launch_bounds__(256) xprep_kernel(const __grid_constant__ PrepParams P) {
    pdl_launch_dependents();
    const int M = P.M;
    for (int64_t w = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; w < P.total; w += (int64_t)gridDim.x * blockDim.x) {
        int p = 0;
        while (p + 1 < P.count && w >= P.d[p + 1].work_begin) ++p;
        const PrepDesc& D = P.d[p];
        const int64_t local = w - D.work_begin;                 // in units of 8 halves
        const int64_t per_member = (int64_t)M * D.Kp / 8;
        const int64_t l = local / per_member;
        const int64_t d0 = 8 * (local - l * per_member);
        const uint16_t* x = reinterpret_cast<const uint16_t*>(reinterpret_cast<const char*>(D.x) + l * D.stride_x);
        const int line = (int)(d0 >> 4), pos0 = (int)(d0 & 15);
        const int bi = line / M, m = line - bi * M;
        uint16_t v[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const int pos = pos0 + e, tt = pos >> 2, hh = pos & 3;
            const int k = P.format == LQ_FMT_2BIT_LM_G32
                ? (bi >> 4) * 256 + tt * 64 + ((bi >> 2) & 3) * 16 + hh * 4 + (bi & 3)
                : (bi >> 2) * 64 + tt * 16 + (bi & 3) * 4 + hh;
            v[e] = k < D.K ? to_half_bits(x[(int64_t)m * D.K + k], P.x_bf16) : (uint16_t)0;
        }
        uint16_t* dst = D.xperm + l * D.xperm_stride + d0;
        *reinterpret_cast<uint4*>(dst) = make_uint4((uint32_t)v[0] | ((uint32_t)v[1] << 16), (uint32_t)v[2] | ((uint32_t)v[3] << 16),
                                                    (uint32_t)v[4] | ((uint32_t)v[5] << 16), (uint32_t)v[6] | ((uint32_t)v[7] << 16));
    }
}

// Pass 2 (after pass 1): zero x at the anchor columns (the anchors replace those weights)
// and write x gathered at the anchor columns, zero-padded to a multiple of 64.
__global__ void __launch_bounds__(256) xanchor_kernel(const __grid_constant__ PrepParams P) {
    pdl_launch_dependents();
    pdl_wait();  // pass 1 has finished writing
    const int M = P.M;
    for (int64_t w = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; w < P.total_anchor; w += (int64_t)gridDim.x * blockDim.x) {
        int p = 0;
        while (p + 1 < P.count && w >= P.d[p + 1].anchor_begin) ++p;
        const PrepDesc& D = P.d[p];
        const int64_t local = w - D.anchor_begin;
        const int64_t per_member = (int64_t)M * D.a_pad;
        const int64_t l = local / per_member;
        const int rem = (int)(local - l * per_member);
        const int m = rem / D.a_pad, a = rem - m * D.a_pad;
        uint16_t v = 0;
        if (a < D.A) {
            const uint16_t* x = reinterpret_cast<const uint16_t*>(reinterpret_cast<const char*>(D.x) + l * D.stride_x);
            const int32_t* aidx =
                reinterpret_cast<const int32_t*>(reinterpret_cast<const char*>(D.anchor_idx) + l * D.stride_anchor_idx);
            const int k = __ldg(aidx + a);
            v = to_half_bits(x[(int64_t)m * D.K + k], P.x_bf16);
            int bi, tt, hh;
            if (P.format == LQ_FMT_2BIT_LM_G32) {
                const int r = k & 255, e = r & 15;
                tt = r >> 6;
                bi = (k >> 8) * 16 + ((r >> 4) & 3) * 4 + (e & 3);
                hh = e >> 2;
            } else {
                const int r = k & 63, e = r & 15;
                tt = r >> 4;
                bi = (k >> 6) * 4 + (e >> 2);
                hh = e & 3;
            }
            D.xperm[l * D.xperm_stride + ((int64_t)bi * M + m) * 16 + tt * 4 + hh] = 0;
        }
        const int s = a & 15;
        const int tt = (s & 7) >> 1, hh = (s & 1) + 2 * (s >> 3);
        D.xaperm[l * D.xaperm_stride + ((int64_t)(a >> 4) * M + m) * 16 + tt * 4 + hh] = v;
    }
}

// ---- host side ---------------------------------------------------------------------

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        cudaDriverEntryPointQueryResult q;
        void* p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// A 3-D tile map over [batch][rows][inner] with the given element type and box.
bool make_map(CUtensorMap* map, CUtensorMapDataType dt, int esize, const void* base, uint64_t inner, uint64_t rows,
              uint64_t batch, uint64_t row_stride_bytes, uint64_t batch_stride_bytes, uint32_t box_inner,
              uint32_t box_rows, CUtensorMapSwizzle sw) {
    auto fn = encode_fn();
    if (!fn) return false;
    (void)esize;
    cuuint64_t dims[3] = {inner, rows, batch};
    cuuint64_t strides[2] = {row_stride_bytes, batch > 1 ? batch_stride_bytes : row_stride_bytes * rows};
    cuuint32_t box[3] = {box_inner, box_rows, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    return fn(map, dt, 3, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int round_up(int a, int b) { return (a + b - 1) / b * b; }

template <int NT, int FMT>
lq_status launch_main(const Params& P, size_t smem, int grid, cudaStream_t stream) {
    auto kern = gemv_tma_kernel<NT, FMT>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
        return LQ_ERR_CUDA;
    cudaLaunchConfig_t cfg;
    memset(&cfg, 0, sizeof(cfg));
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kThreadsT);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, kern, P) != cudaSuccess) return LQ_ERR_CUDA;
    return cudaPeekAtLastError() == cudaSuccess ? LQ_OK : LQ_ERR_CUDA;
}

template <int FMT>
lq_status launch_fmt(const Params& P, size_t smem, int grid, cudaStream_t stream) {
    const int nt = (P.M + 7) / 8;
    if (nt == 1) return launch_main<1, FMT>(P, smem, grid, stream);
    if (nt == 2) return launch_main<2, FMT>(P, smem, grid, stream);
    return launch_main<4, FMT>(P, smem, grid, stream);
}

}  // namespace

bool gemv_tma_eligible(const lq_problem* probs, int count) {
    for (int i = 0; i < count; ++i) {
        if (probs[i].K % 256 != 0) return false;   // TMA row strides of the scale tiles need K/16 % 16 == 0
        if (probs[i].N >= (1 << 30) || probs[i].batch >= (1 << 30)) return false;
    }
    return encode_fn() != nullptr;
}

lq_status launch_gemv_tma(const GemvWorkspace& ws, const lq_problem* probs, int count, cudaStream_t stream) {
    static Params P;          // large (tensor maps); built on the host, passed by value
    static PrepParams Q;
    static std::mutex mu;
    std::lock_guard<std::mutex> lock(mu);
    memset(&P, 0, sizeof(P));
    memset(&Q, 0, sizeof(Q));
    const int M = probs[0].M;
    const int fmt = probs[0].format;
    const int SC = fmt == LQ_FMT_2BIT_LM_G32 ? kSC2 : kSCNF4;
    P.count = Q.count = count;
    P.M = Q.M = M;
    P.format = Q.format = fmt;
    P.y_dtype = probs[0].y_dtype;
    Q.x_bf16 = probs[0].x_dtype == LQ_BF16;

    // columns per split: the x slot (M x KC binary16) stays <= 16 KiB
    int kc_target = M <= 4 ? 2048 : 512;
    kc_target = std::max(kc_target, SC);

    // first pass: splits
    int S[kMaxGroup], Sa[kMaxGroup], merged[kMaxGroup], KC[kMaxGroup], KA[kMaxGroup];
    int64_t units = 0;
    for (int i = 0; i < count; ++i) {
        const lq_problem& q = probs[i];
        const int A = fmt == LQ_FMT_2BIT_LM_G32 ? q.A : 0;
        const int Kp = round_up(q.K, 256);
        const int a_pad = A > 0 ? round_up(A, kSCA) : 0;
        KC[i] = std::min(round_up(q.K, SC), kc_target);
        S[i] = (q.K + KC[i] - 1) / KC[i];
        KA[i] = kc_target;
        Sa[i] = A > 0 ? (A + KA[i] - 1) / KA[i] : 0;
        merged[i] = (S[i] == 1 && Sa[i] <= 1 && Kp + a_pad <= kc_target) ? 1 : 0;
        const int parts = merged[i] ? 1 : S[i] + Sa[i];
        units += (int64_t)q.batch * ((q.N + kRows - 1) / kRows) * parts;
    }
    // small launches: split K further so that every SM has work
    const int64_t want = 2LL * ws.num_sms;
    if (units < want) {
        units = 0;
        for (int i = 0; i < count; ++i) {
            const lq_problem& q = probs[i];
            const int64_t strips = (int64_t)q.batch * ((q.N + kRows - 1) / kRows);
            const int target_s = (int)std::min<int64_t>(std::max<int64_t>(1, want / std::max<int64_t>(1, strips)),
                                                         (q.K + SC - 1) / SC);
            if (target_s > S[i]) {
                KC[i] = round_up((q.K + target_s - 1) / target_s, SC);
                S[i] = (q.K + KC[i] - 1) / KC[i];
                merged[i] = 0;
            }
            const int parts = merged[i] ? 1 : S[i] + Sa[i];
            units += strips * parts;
        }
    }

    int64_t unit = 0, strip = 0, partial_floats = 0, prep = 0, prep_a = 0, xperm_halves = 0;
    int x_slot = 0;
    for (int i = 0; i < count; ++i) {
        const lq_problem& q = probs[i];
        const int A = fmt == LQ_FMT_2BIT_LM_G32 ? q.A : 0;
        Desc& d = P.d[i];
        PrepDesc& e = Q.d[i];
        d.N = q.N;
        d.K = q.K;
        d.A = A;
        d.batch = q.batch;
        d.Kp = round_up(q.K, 256);
        d.a_pad = A > 0 ? round_up(A, kSCA) : 0;
        d.KC = KC[i];
        d.S = S[i];
        d.KA = KA[i];
        d.Sa = Sa[i];
        d.merged = merged[i];
        d.parts = merged[i] ? 1 : S[i] + Sa[i];
        d.strips = (q.N + kRows - 1) / kRows;
        d.y = q.y;
        d.stride_y = q.stride_y;
        d.unit_begin = unit;
        unit += (int64_t)q.batch * d.strips * d.parts;
        if (d.parts > 1) {
            d.strip_begin = strip;
            d.partial_begin = partial_floats;
            strip += (int64_t)q.batch * d.strips;
            partial_floats += (int64_t)q.batch * d.strips * d.parts * M * kRows;
        }
        d.xperm_stride = (int64_t)M * d.Kp;
        d.xaperm_stride = (int64_t)M * d.a_pad;
        const int slot_cols = d.merged ? d.Kp + d.a_pad : std::max(round_up(std::min(d.KC, q.K), 256), std::min(d.KA, d.a_pad));
        x_slot = std::max(x_slot, M * slot_cols);
        // x pre-pass
        e.x = static_cast<const uint16_t*>(q.x);
        e.stride_x = q.stride_x;
        e.anchor_idx = A > 0 ? q.anchor_idx : nullptr;
        e.stride_anchor_idx = q.stride_anchor_idx;
        e.K = q.K;
        e.Kp = d.Kp;
        e.A = A;
        e.a_pad = d.a_pad;
        e.batch = q.batch;
        e.xperm_stride = d.xperm_stride;
        e.xaperm_stride = d.xaperm_stride;
        e.work_begin = prep;
        prep += (int64_t)q.batch * M * d.Kp / 8;
        e.anchor_begin = prep_a;
        prep_a += (int64_t)q.batch * M * d.a_pad;
        xperm_halves += (int64_t)q.batch * M * (d.Kp + d.a_pad);
    }
    // workspace: [partials | x pre-pass output] in the float area, [sched(2) | strip counters] in the counters
    const int64_t xperm_floats = (xperm_halves + 1) / 2 + 64 * (count + 1);
    if ((size_t)(strip + 2) > ws.num_counters || (size_t)(partial_floats + xperm_floats + 64) > ws.partial_floats)
        return LQ_ERR_WORKSPACE;
    uint16_t* xp = reinterpret_cast<uint16_t*>(
        (reinterpret_cast<uintptr_t>(ws.partials + partial_floats) + 255) & ~uintptr_t(255));
    for (int i = 0; i < count; ++i) {
        const int64_t member = (int64_t)M * (P.d[i].Kp + P.d[i].a_pad);
        Q.d[i].xperm = xp;
        Q.d[i].xaperm = xp + (int64_t)probs[i].batch * P.d[i].xperm_stride;
        P.d[i].xperm = Q.d[i].xperm;
        P.d[i].xaperm = Q.d[i].xaperm;
        xp += (int64_t)probs[i].batch * member;
        xp = reinterpret_cast<uint16_t*>((reinterpret_cast<uintptr_t>(xp) + 255) & ~uintptr_t(255));
    }
    P.x_slot_halves = round_up(std::max(x_slot, 8), 8);
    P.total_units = unit;
    P.partials = ws.partials;
    P.sched = ws.counters;
    P.counters = ws.counters + 2;
    P.status = ws.status;
    Q.total = prep;
    Q.total_anchor = prep_a;

    // tensor maps
    for (int i = 0; i < count; ++i) {
        const lq_problem& q = probs[i];
        const uint64_t rows = q.N, b = q.batch;
        bool ok;
        if (fmt == LQ_FMT_2BIT_LM_G32) {
            ok = make_map(&P.maps[i].codes, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, q.codes, q.K / 4, rows, b, q.K / 4,
                          q.stride_codes, 128, kRows, CU_TENSOR_MAP_SWIZZLE_128B) &&
                 make_map(&P.maps[i].scales, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, q.scales, q.K / 32, rows, b,
                          (uint64_t)q.K / 16, q.stride_scales, 16, kRows, CU_TENSOR_MAP_SWIZZLE_NONE) &&
                 make_map(&P.maps[i].offsets, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, q.offsets, q.K / 32, rows, b,
                          (uint64_t)q.K / 16, q.stride_offsets, 16, kRows, CU_TENSOR_MAP_SWIZZLE_NONE);
            if (ok && q.A > 0)
                ok = make_map(&P.maps[i].anchors, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, q.anchor_w, q.A, rows, b,
                              (uint64_t)q.ld_anchor * 2, q.stride_anchor_w, kSCA, kRows, CU_TENSOR_MAP_SWIZZLE_128B);
        } else {
            ok = make_map(&P.maps[i].codes, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, q.codes, q.K / 2, rows, b, q.K / 2,
                          q.stride_codes, 128, kRows, CU_TENSOR_MAP_SWIZZLE_128B) &&
                 make_map(&P.maps[i].scales, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, q.scales, q.K / 64, rows, b,
                          (uint64_t)q.K / 16, q.stride_scales, 4, kRows, CU_TENSOR_MAP_SWIZZLE_NONE);
        }
        if (!ok) return LQ_ERR_UNSUPPORTED;   // the register-fed kernel takes over
    }

    if (ws.clear_counters && cudaMemsetAsync(ws.counters, 0, sizeof(unsigned) * (size_t)(strip + 2), stream) != cudaSuccess)
        return LQ_ERR_CUDA;

    // x passes, then the main kernel, chained by programmatic dependent launch
    const int prep_grid = (int)std::min<int64_t>((Q.total + 255) / 256, (int64_t)ws.num_sms * 8);
    xprep_kernel<<<std::max(1, prep_grid), 256, 0, stream>>>(Q);
    if (cudaPeekAtLastError() != cudaSuccess) return LQ_ERR_CUDA;
    if (Q.total_anchor > 0) {
        cudaLaunchConfig_t cfg;
        memset(&cfg, 0, sizeof(cfg));
        cfg.gridDim = dim3((unsigned)std::max<int64_t>(1, std::min<int64_t>((Q.total_anchor + 255) / 256, (int64_t)ws.num_sms * 8)));
        cfg.blockDim = dim3(256);
        cfg.stream = stream;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        if (cudaLaunchKernelEx(&cfg, xanchor_kernel, Q) != cudaSuccess) return LQ_ERR_CUDA;
    }

    auto smem_for = [&](int ns) {
        return 1024 + (size_t)ns * kStageBytes + 2 * (size_t)P.x_slot_halves * 2 + 2 * (size_t)M * kRows * 4 +
               (2 * ns + 8) * 8;
    };
    // two CTAs per SM when they fit (4 stages, else 3), otherwise one CTA with 4 stages
    int per_sm = 2;
    P.nstages = kMaxStages;
    if (2 * (smem_for(kMaxStages) + 1024) > 228 * 1024) P.nstages = 3;
    if (2 * (smem_for(P.nstages) + 1024) > 228 * 1024) {
        per_sm = 1;
        P.nstages = kMaxStages;
    }
    const size_t smem = smem_for(P.nstages);
    if (smem > (size_t)ws.max_smem_optin) return LQ_ERR_UNSUPPORTED;
    const int grid = (int)std::min<int64_t>((int64_t)ws.num_sms * per_sm, unit);
    if (fmt == LQ_FMT_2BIT_LM_G32) return launch_fmt<LQ_FMT_2BIT_LM_G32>(P, smem, grid, stream);
    return launch_fmt<LQ_FMT_NF4_B64>(P, smem, grid, stream);
}

}  // namespace lq
