// lq_gemm: prefill-sized y = x * W_eff^T on tcgen05 tensor cores.
//
// A dense contraction at M = 2048 tokens, so the weights are dequantized into
// shared memory and multiplied on the 5th-generation tensor cores:
//
//  * Persistent CTAs, one per SM, walk output tiles of 128 weight rows x 256
//    tokens.  The fp32 accumulator (128 lanes x 256 columns) lives in tensor
//    memory.
//  * Warp 0 streams x tiles (256 tokens x 64 columns, 16-bit, 128-byte swizzle)
//    by TMA into a 4-stage ring.
//  * Warps 2-9 dequantize: each thread turns 32 columns of one weight row into
//    16-bit values (2-bit: fmaf(S, C[q], Z) per group, otf-llm README sections
//    2-3; NF4: T[q] * absmax, AirQuant README NF4) and writes them in the
//    canonical K-major 128-byte-swizzled layout.  Anchor columns (section 4) are
//    zeroed in the weight tile, and the anchors join as extra K-blocks: binary16
//    anchor weights against x gathered at the anchor columns.
//  * Warp 1 (one thread) issues tcgen05.mma (M=128, N=256, K=16) from the two
//    shared-memory descriptors and commits each stage back to the producers.
//  * The same eight warps read the accumulator back with tcgen05.ld and write y.
// The multiply runs in the dtype of x (bf16 or binary16) with fp32 accumulation.
// Every mbarrier wait is bounded in time.

#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstring>
#include <mutex>

#include "lq_common.cuh"
#include "lq_dq.cuh"
#include "lq_internal.h"
#include "lq_tcgen05.cuh"
#include "lq_tma.cuh"

namespace lq {
namespace {

constexpr int kBM = 128;                 // weight rows per tile (MMA M)
constexpr int kBN = 256;                 // tokens per tile (MMA N)
constexpr int kBK = 64;                  // columns per stage (one 128-byte swizzle row of 16-bit values)
constexpr int kStagesG = 4;
constexpr int kATile = kBM * kBK * 2;    // 16 KiB
constexpr int kBTile = kBN * kBK * 2;    // 32 KiB
constexpr int kDqWarps = 8;
constexpr int kGemmThreads = (2 + kDqWarps) * 32;
constexpr int kTmemCols = 256;

struct GemmParams {
    CUtensorMap xmap;          // x [M][K] 16-bit, box 64 x 256, 128-byte swizzle
    CUtensorMap xamap;         // x at the anchor columns [M][a_pad], same box
    const uint8_t* codes;
    const void* scales;
    const uint16_t* offsets;
    const uint16_t* anchor_w;
    const unsigned long long* anchor_bits;   // [K/64] anchor columns of each 64-column block
    void* y;
    int M, N, K, A, ld_anchor, a_pad, format, bf16, y_dtype;
    int tiles_m, total_tiles;
    int* status;
};

__device__ __forceinline__ uint32_t pack2(float lo, float hi, int bf16) {
    uint32_t d;
    if (bf16)
        asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
    else
        asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
    return d;
}

__device__ __forceinline__ void sts128(uint8_t* p, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    *reinterpret_cast<uint4*>(p) = make_uint4(a, b, c, d);
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

template <int FMT>
__global__ void __launch_bounds__(kGemmThreads, 1) gemm_kernel(const __grid_constant__ GemmParams P) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* base = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
    uint8_t* atile = base;                                  // [kStagesG][128 rows][128 B]
    uint8_t* btile = base + kStagesG * kATile;              // [kStagesG][256 rows][128 B]
    uint64_t* bars = reinterpret_cast<uint64_t*>(btile + kStagesG * kBTile);
    // bars: a_full[S], b_full[S], empty[S], accum_full, tmem_empty
    __shared__ uint32_t s_tmem;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t a_full0 = smem_u32(bars), b_full0 = smem_u32(bars + kStagesG), empty0 = smem_u32(bars + 2 * kStagesG);
    const uint32_t accum_full = smem_u32(bars + 3 * kStagesG), tmem_empty = accum_full + 8;

    if (tid == 0) {
        for (int s = 0; s < kStagesG; ++s) {
            mbar_init(a_full0 + 8 * s, kDqWarps);
            mbar_init(b_full0 + 8 * s, 1);
            mbar_init(empty0 + 8 * s, 1);
        }
        mbar_init(accum_full, 1);
        mbar_init(tmem_empty, kDqWarps);
        fence_mbar_init();
    }
    if (warp == 1) tmem_alloc(smem_u32(&s_tmem), kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = s_tmem;

    const int KB = P.K / kBK, AB = P.a_pad / kBK, NKB = KB + AB;
    int own_abort = 0;
    volatile int* abort = &own_abort;

    if (warp == 0) {
        // ---------------------------------------------------------------- TMA: x tiles
        if (lane == 0) {
            prefetch_tensormap(&P.xmap);
            if (AB) prefetch_tensormap(&P.xamap);
            int s = 0, ph = 0;
            for (int tile = blockIdx.x; tile < P.total_tiles; tile += gridDim.x) {
                const int m0 = (tile % P.tiles_m) * kBN;
                for (int kb = 0; kb < NKB; ++kb) {
                    if (!mbar_wait_bounded(empty0 + 8 * s, ph ^ 1, abort, P.status)) goto tma_done;
                    mbar_arrive_expect_tx(b_full0 + 8 * s, kBTile);
                    if (kb < KB) tma_load_2d(smem_u32(btile + s * kBTile), &P.xmap, kb * kBK, m0, b_full0 + 8 * s);
                    else tma_load_2d(smem_u32(btile + s * kBTile), &P.xamap, (kb - KB) * kBK, m0, b_full0 + 8 * s);
                    if (++s == kStagesG) {
                        s = 0;
                        ph ^= 1;
                    }
                }
            }
        tma_done:;
        }
    } else if (warp == 1) {
        // ---------------------------------------------------------------- MMA issue
        if (lane == 0) {
            const uint32_t idesc = idesc_f16(P.bf16 != 0, kBM, kBN);
            int s = 0, ph = 0, tph = 0;
            for (int tile = blockIdx.x; tile < P.total_tiles; tile += gridDim.x) {
                // the epilogue has drained the accumulator of the previous tile
                if (!mbar_wait_bounded(tmem_empty, tph ^ 1, abort, P.status)) break;
                tph ^= 1;
                tc_fence_after();
                bool ok = true;
                for (int kb = 0; kb < NKB; ++kb) {
                    if (!(ok = mbar_wait_bounded(a_full0 + 8 * s, ph, abort, P.status))) break;
                    if (!(ok = mbar_wait_bounded(b_full0 + 8 * s, ph, abort, P.status))) break;
                    tc_fence_after();
                    const uint32_t a_addr = smem_u32(atile + s * kATile), b_addr = smem_u32(btile + s * kBTile);
#pragma unroll
                    for (int k = 0; k < kBK / 16; ++k)
                        tc_mma_f16(tmem, smem_desc_sw128(a_addr + 32 * k), smem_desc_sw128(b_addr + 32 * k), idesc,
                                   (kb | k) != 0);
                    tc_commit(empty0 + 8 * s);   // the stage is free once these MMAs have read it
                    if (++s == kStagesG) {
                        s = 0;
                        ph ^= 1;
                    }
                }
                if (!ok) break;
                tc_commit(accum_full);
            }
        }
    } else {
        // ---------------------------------------------------------------- dequant + epilogue
        const int d = tid - 64, r = d & (kBM - 1), h = d >> 7;   // row of the tile, half of the 64 columns
        const int K = P.K, N = P.N;
        const float C0 = -1.52f, C1 = -0.45f, C2 = 0.45f, C3 = 1.52f;
        int s = 0, ph = 0, aph = 0;
        for (int tile = blockIdx.x; tile < P.total_tiles; tile += gridDim.x) {
            const int n0 = (tile / P.tiles_m) * kBM, m0 = (tile % P.tiles_m) * kBN;
            const int64_t nr = min(n0 + r, N - 1);   // rows past N read the last row; never stored
            bool ok = true;
            for (int kb = 0; kb < NKB; ++kb) {
                // warp-uniform: a lane that gives up takes its whole warp out
                if (!(ok = __all_sync(0xffffffffu, mbar_wait_bounded(empty0 + 8 * s, ph ^ 1, abort, P.status))))
                    break;
                uint8_t* arow = atile + s * kATile + r * 128;
                const int sw = r & 7;
                if (kb < KB) {
                    uint32_t c[4][4];
                    if (FMT == LQ_FMT_2BIT_LM_G32) {
                        const uint2 cw = ldg64(P.codes + nr * (K / 4) + kb * 16 + h * 8);
                        const int64_t gi = nr * (K / 32) + kb * 2 + h;
                        const float sf = half_bits_to_float(static_cast<const uint16_t*>(P.scales)[gi]);
                        const float zf = half_bits_to_float(P.offsets[gi]);
                        const uint32_t P01 = pack2(__fmaf_rn(sf, C0, zf), __fmaf_rn(sf, C1, zf), P.bf16);
                        const uint32_t P23 = pack2(__fmaf_rn(sf, C2, zf), __fmaf_rn(sf, C3, zf), P.bf16);
                        dq2_word(cw.x, P01, P23, c[0], c[1]);
                        dq2_word(cw.y, P01, P23, c[2], c[3]);
                    } else {
                        const uint4 cw = ldg128(P.codes + nr * (K / 2) + kb * 32 + h * 16);
                        const float am = static_cast<const float*>(P.scales)[nr * (K / 64) + kb];
                        // this block's 16 values T[q] * absmax, one rounding, in byte-split registers
                        uint32_t BL[4], BH[4];
#pragma unroll
                        for (int q4 = 0; q4 < 4; ++q4) {
                            const uint32_t p01 = pack2(__fmul_rn(kNF4[4 * q4], am), __fmul_rn(kNF4[4 * q4 + 1], am), P.bf16);
                            const uint32_t p23 = pack2(__fmul_rn(kNF4[4 * q4 + 2], am), __fmul_rn(kNF4[4 * q4 + 3], am), P.bf16);
                            BL[q4] = prmt(p01, p23, 0x6420);
                            BH[q4] = prmt(p01, p23, 0x7531);
                        }
                        const uint32_t ws[4] = {cw.x, cw.y, cw.z, cw.w};
#pragma unroll
                        for (int wi = 0; wi < 4; ++wi) {
                            expand_nf4_fast(ws[wi], 0, BL, BH, c[wi][0], c[wi][1]);
                            expand_nf4_fast(ws[wi], 1, BL, BH, c[wi][2], c[wi][3]);
                        }
                    }
#pragma unroll
                    for (int q = 0; q < 4; ++q) sts128(arow + (((4 * h + q) ^ sw) << 4), c[q][0], c[q][1], c[q][2], c[q][3]);
                    if (FMT == LQ_FMT_2BIT_LM_G32 && P.A > 0) {
                        // anchor columns replace the 2-bit weights: zero them in the tile
                        uint32_t bits = (uint32_t)(P.anchor_bits[kb] >> (32 * h));
                        while (bits) {
                            const int i = __ffs(bits) - 1;
                            bits &= bits - 1;
                            const int col = 32 * h + i;
                            *reinterpret_cast<uint16_t*>(arow + (((col >> 3) ^ sw) << 4) + (col & 7) * 2) = 0;
                        }
                    }
                } else {
                    // anchor block: 32 binary16 anchor weights of this row, zero past A
                    const int a0 = (kb - KB) * kBK + 32 * h;
                    const uint16_t* src = P.anchor_w + nr * P.ld_anchor + a0;
                    uint32_t v[16];
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const uint4 u = (a0 + 8 * q < P.A) ? *reinterpret_cast<const uint4*>(src + 8 * q) : make_uint4(0, 0, 0, 0);
                        v[4 * q] = u.x;
                        v[4 * q + 1] = u.y;
                        v[4 * q + 2] = u.z;
                        v[4 * q + 3] = u.w;
                    }
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const int a = a0 + 2 * i;
                        uint32_t w = a < P.A ? v[i] : 0u;
                        if (a + 1 >= P.A) w &= 0xFFFFu;
                        if (P.bf16) {
                            const float lo = half_bits_to_float((uint16_t)w), hi = half_bits_to_float((uint16_t)(w >> 16));
                            w = pack2(lo, hi, 1);
                        }
                        v[i] = w;
                    }
#pragma unroll
                    for (int q = 0; q < 4; ++q) sts128(arow + (((4 * h + q) ^ sw) << 4), v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
                }
                fence_proxy_async_smem();   // generic-proxy stores -> visible to the tensor core
                __syncwarp();
                if (lane == 0) mbar_arrive(a_full0 + 8 * s);
                if (++s == kStagesG) {
                    s = 0;
                    ph ^= 1;
                }
            }
            if (!ok) break;
            // ---- epilogue: accumulator rows of this warp's lane quarter, half of the 256 columns
            if (!__all_sync(0xffffffffu, mbar_wait_bounded(accum_full, aph, abort, P.status))) break;
            aph ^= 1;
            tc_fence_after();
            const int quarter = warp & 3, colhalf = (warp - 2) >> 2;
            const int n = n0 + 32 * quarter + lane;
#pragma unroll 1
            for (int cc = 0; cc < 4; ++cc) {
                const int col = 128 * colhalf + 32 * cc;
                uint32_t v[32];
                tmem_ld32(tmem + ((uint32_t)(32 * quarter) << 16) + col, v);
                if (n < N) {
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        const int m = m0 + col + j;
                        if (m < P.M) store_out(P.y, (size_t)m * N + n, P.y_dtype, __uint_as_float(v[j]));
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(tmem_empty);
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

// x gathered at the anchor columns ([M][a_pad], zero past A) and the anchor bitmap
__global__ void __launch_bounds__(256) gemm_prep_kernel(const uint16_t* __restrict__ x, int M, int K,
                                                        const int32_t* __restrict__ anchor_idx, int A, int a_pad,
                                                        uint16_t* __restrict__ xa, unsigned long long* bits) {
    const int64_t total = (int64_t)M * a_pad;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total || i < A;
         i += (int64_t)gridDim.x * blockDim.x) {
        if (i < A) {
            const int k = anchor_idx[i];
            atomicOr(bits + (k >> 6), 1ull << (k & 63));
        }
        if (i < total) {
            const int m = (int)(i / a_pad), a = (int)(i - (int64_t)m * a_pad);
            xa[i] = a < A ? x[(int64_t)m * K + anchor_idx[a]] : (uint16_t)0;
        }
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

// 2-D map over a row-major [rows][cols] 16-bit matrix, box 64 columns x 256 rows, 128-byte swizzle.
bool map_x(CUtensorMap* m, const void* base, uint64_t cols, uint64_t rows) {
    auto fn = encode_fn_g();
    if (!fn) return false;
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {cols * 2};
    cuuint32_t box[2] = {(cuuint32_t)kBK, (cuuint32_t)kBN};
    cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, const_cast<void*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

lq_status launch_gemm(lq_handle h, const lq_problem& p, cudaStream_t stream) {
    GemmParams P;
    memset(&P, 0, sizeof(P));
    const int A = p.format == LQ_FMT_2BIT_LM_G32 ? p.A : 0;
    const int a_pad = A > 0 ? (A + kBK - 1) / kBK * kBK : 0;
    P.codes = p.codes;
    P.scales = p.scales;
    P.offsets = p.offsets;
    P.anchor_w = p.anchor_w;
    P.y = p.y;
    P.M = p.M;
    P.N = p.N;
    P.K = p.K;
    P.A = A;
    P.ld_anchor = p.ld_anchor;
    P.a_pad = a_pad;
    P.format = p.format;
    P.bf16 = p.x_dtype == LQ_BF16;
    P.y_dtype = p.y_dtype;
    P.tiles_m = (p.M + kBN - 1) / kBN;
    const int64_t tiles = (int64_t)P.tiles_m * ((p.N + kBM - 1) / kBM);
    if (tiles > 0x7fffffffLL) return LQ_ERR_UNSUPPORTED;
    P.total_tiles = (int)tiles;
    P.status = h->status_flag;

    // workspace: anchor bitmap [K/64] | x at the anchor columns [M][a_pad]
    char* ws = reinterpret_cast<char*>(h->partials);
    const size_t bits_bytes = ((size_t)(p.K / 64) * 8 + 255) & ~size_t(255);
    const size_t xa_bytes = (size_t)p.M * a_pad * 2;
    if (bits_bytes + xa_bytes + 256 > h->partial_floats * sizeof(float)) return LQ_ERR_WORKSPACE;
    unsigned long long* bits = reinterpret_cast<unsigned long long*>(ws);
    uint16_t* xa = reinterpret_cast<uint16_t*>(ws + bits_bytes);
    P.anchor_bits = bits;
    if (!map_x(&P.xmap, p.x, (uint64_t)p.K, (uint64_t)p.M)) return LQ_ERR_CUDA;
    if (A > 0) {
        if (!map_x(&P.xamap, xa, (uint64_t)a_pad, (uint64_t)p.M)) return LQ_ERR_CUDA;
        if (cudaMemsetAsync(bits, 0, (size_t)(p.K / 64) * 8, stream) != cudaSuccess) return LQ_ERR_CUDA;
        const int64_t work = std::max<int64_t>((int64_t)p.M * a_pad, A);
        const int grid = (int)std::min<int64_t>((work + 255) / 256, (int64_t)h->num_sms * 8);
        gemm_prep_kernel<<<grid, 256, 0, stream>>>(static_cast<const uint16_t*>(p.x), p.M, p.K, p.anchor_idx, A, a_pad,
                                                   xa, bits);
        if (cudaPeekAtLastError() != cudaSuccess) return LQ_ERR_CUDA;
    }

    const size_t smem = 1024 + (size_t)kStagesG * (kATile + kBTile) + (3 * kStagesG + 2) * 8;
    if (smem > (size_t)h->max_smem_optin) return LQ_ERR_UNSUPPORTED;
    const int grid = (int)std::min<int64_t>(tiles, h->num_sms);
    if (p.format == LQ_FMT_2BIT_LM_G32) {
        if (cudaFuncSetAttribute(gemm_kernel<LQ_FMT_2BIT_LM_G32>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
            return LQ_ERR_CUDA;
        gemm_kernel<LQ_FMT_2BIT_LM_G32><<<grid, kGemmThreads, smem, stream>>>(P);
    } else {
        if (cudaFuncSetAttribute(gemm_kernel<LQ_FMT_NF4_B64>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
            return LQ_ERR_CUDA;
        gemm_kernel<LQ_FMT_NF4_B64><<<grid, kGemmThreads, smem, stream>>>(P);
    }
    return cudaPeekAtLastError() == cudaSuccess ? LQ_OK : LQ_ERR_CUDA;
}

}  // namespace lq
