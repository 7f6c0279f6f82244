// Quantizers on the GPU: the converter step that produces the stored formats the
// hot path reads (otf-llm 4.0.1 README, "Theoretical & Mathematical Foundations"
// sections 3-4 and its converter's G / anchor-fraction arguments; AirQuant README,
// "Fundamentacao Teorica" item 2 for NF4).
//
// Every output is reproducible bit for bit: each floating-point decision is taken in
// fp64 with the operations of the definition, one IEEE rounding each (the _rn
// intrinsics keep the compiler from fusing a multiply into an add), and every sum
// runs in one fixed order:
//   * along a group (mean, variance, the least-squares sums): pairwise with eight
//     interleaved partial sums r[j] (element i goes to r[i % 8] while a full round of
//     eight remains), combined as ((r0+r1)+(r2+r3))+((r4+r5)+(r6+r7)), then the last
//     n % 8 elements one by one; fewer than eight elements are added one by one;
//   * down a column (anchor scores): row by row.
// These are the orders numpy's reductions use, so the results equal a numpy
// implementation of the same definitions exactly.
//
//  * lq_select_anchors: score_c = sqrt(sum_n W[n][c]^2) * profile_c (section 4), the
//    A largest scores, ties to the lower column, written in ascending column order.
//    One thread per column sums its column; one CTA then finds the A-th largest key
//    by an 8-pass radix select and compacts the chosen columns in column order.
//  * lq_quantize_2bit: per row and group of 32 columns, the non-anchor values V are
//    normalised by their mean and population standard deviation (z = 0 when it is 0),
//    each z takes the nearest codebook level (lowest index on a tie), and (S, Z) is the
//    closed-form least-squares fit of V on C[q] (section 3); S and Z are stored as
//    binary16 (round to nearest even).  Anchor columns store code 0 and their binary16
//    value in anchor_w.  One thread per (row, group).
//  * lq_quantize_nf4: per block of 64 columns, absmax = max|w| (fp32) and
//    q = argmin_k |w/absmax - T[k]| in fp64 (lowest index on a tie; q = index of 0
//    when absmax = 0).  One warp per block: lane l owns columns 2l and 2l+1 and
//    writes byte l of the block.

#include <cuda_fp16.h>

#include "lq_common.cuh"
#include "lq_internal.h"

namespace lq {
namespace {

// otf-llm README section 2: the four Lloyd-Max levels, as fp64 (the decimal values).
__device__ __constant__ const double kLevels[4] = {-1.52, -0.45, 0.45, 1.52};
constexpr double kOlsEps = 1e-12;   // the "+ eps" of the least-squares denominator (section 3)

// Pairwise sum of term(0..n) in the fixed order described at the top of the file.
// The result is +0 when every term is a zero (a sum that starts from +0).
template <class F>
__device__ __forceinline__ double pairwise_sum(int n, F term) {
    double res;
    if (n < 8) {
        res = 0.0;
        for (int i = 0; i < n; ++i) res = __dadd_rn(res, term(i));
        return res;
    }
    double r[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) r[j] = term(j);
    const int n8 = n - (n % 8);
    int i = 8;
    for (; i < n8; i += 8) {
#pragma unroll
        for (int j = 0; j < 8; ++j) r[j] = __dadd_rn(r[j], term(i + j));
    }
    res = __dadd_rn(__dadd_rn(__dadd_rn(r[0], r[1]), __dadd_rn(r[2], r[3])),
                    __dadd_rn(__dadd_rn(r[4], r[5]), __dadd_rn(r[6], r[7])));
    for (; i < n; ++i) res = __dadd_rn(res, term(i));
    return __dadd_rn(0.0, res);
}

__device__ __forceinline__ uint16_t half_bits_rn(double v) { return __half_as_ushort(__double2half(v)); }

// ---- anchor selection -------------------------------------------------------------

// score[c] = sqrt(sum_n W[n][c]^2) * profile[c] (profile NULL: 1).  W is fp32 [N][K].
// One thread per column: the sum must run row by row, so parallelism comes from the
// columns and from keeping 32 rows of loads in flight per thread.
constexpr int kScoreThreads = 64;

__global__ void __launch_bounds__(kScoreThreads) anchor_score_kernel(const float* __restrict__ W, int N, int K,
                                                                     const double* __restrict__ profile, double* score) {
    const int c = blockIdx.x * blockDim.x + threadIdx.x;
    if (c >= K) return;
    const float* col = W + c;
    double acc = 0.0;
    int n = 0;
    for (; n + 32 <= N; n += 32) {
        float v[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] = __ldg(col + (size_t)(n + j) * K);
#pragma unroll
        for (int j = 0; j < 32; ++j) acc = __dadd_rn(acc, __dmul_rn((double)v[j], (double)v[j]));
    }
    for (; n < N; ++n) {
        const double v = (double)__ldg(col + (size_t)n * K);
        acc = __dadd_rn(acc, __dmul_rn(v, v));
    }
    const double s = __dsqrt_rn(acc);
    score[c] = __dadd_rn(profile ? __dmul_rn(s, profile[c]) : s, 0.0);   // + 0: a -0 score orders as +0
}

// Order-preserving map of a (non-NaN) double to an unsigned key.
__device__ __forceinline__ unsigned long long order_key(double d) {
    const unsigned long long b = (unsigned long long)__double_as_longlong(d);
    return (b >> 63) ? ~b : (b | (1ull << 63));
}

constexpr int kSelThreads = 1024;

// Exclusive prefix sum of `v` over the CTA; `total` receives the CTA's sum.
__device__ __forceinline__ int block_exclusive_scan(int v, int* warp_sums, int& total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) warp_sums[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int s = lane < kSelThreads / 32 ? warp_sums[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, s, o);
            if (lane >= o) s += y;
        }
        warp_sums[lane] = s;   // inclusive sums of the warp totals
    }
    __syncthreads();
    total = warp_sums[kSelThreads / 32 - 1];
    const int before = warp == 0 ? 0 : warp_sums[warp - 1];
    const int res = before + x - v;
    __syncthreads();   // warp_sums is reused by the next scan
    return res;
}

// The A largest scores (ties: lower column first), written to idx[] in ascending column order.
__global__ void __launch_bounds__(kSelThreads) anchor_select_kernel(const double* __restrict__ score, int K, int A,
                                                                    int32_t* __restrict__ idx) {
    __shared__ unsigned hist[256];
    __shared__ unsigned long long s_prefix;
    __shared__ int s_need;
    __shared__ int warp_sums[32];
    const int tid = threadIdx.x;
    unsigned long long prefix = 0, mask = 0;
    int need = A;
    // radix select, 8 bits per pass from the top: the key of the A-th largest score
    for (int shift = 56; shift >= 0; shift -= 8) {
        for (int i = tid; i < 256; i += kSelThreads) hist[i] = 0u;
        __syncthreads();
        for (int c = tid; c < K; c += kSelThreads) {
            const unsigned long long k = order_key(score[c]);
            if ((k & mask) == prefix) atomicAdd(&hist[(k >> shift) & 255u], 1u);
        }
        __syncthreads();
        if (tid == 0) {
            int above = 0;
            for (int b = 255; b >= 0; --b) {
                if (above + (int)hist[b] >= need) {
                    s_prefix = prefix | ((unsigned long long)b << shift);
                    s_need = need - above;
                    break;
                }
                above += (int)hist[b];
            }
        }
        __syncthreads();
        prefix = s_prefix;
        need = s_need;
        mask |= 0xFFull << shift;
        __syncthreads();
    }
    // every key above the A-th is taken; of the keys equal to it, the `need` lowest columns
    int taken = 0, equal = 0;
    for (int c0 = 0; c0 < K; c0 += kSelThreads) {
        const int c = c0 + tid;
        const unsigned long long k = c < K ? order_key(score[c]) : 0ull;
        const int gt = c < K && k > prefix, eq = c < K && k == prefix;
        int eq_total = 0, take_total = 0;
        const int eq_rank = equal + block_exclusive_scan(eq, warp_sums, eq_total);
        const int take = gt || (eq && eq_rank < need);
        const int pos = taken + block_exclusive_scan(take, warp_sums, take_total);
        if (take && pos < A) idx[pos] = c;
        taken += take_total;
        equal += eq_total;
    }
}

// ---- 2-bit group quantizer ---------------------------------------------------------

// bits[k / 32] bit k % 32 set for every anchor column k (columns outside [0, K) are skipped).
__global__ void anchor_bits_kernel(const int32_t* __restrict__ anchor_idx, int A, int K, uint32_t* bits) {
    const int a = blockIdx.x * blockDim.x + threadIdx.x;
    if (a >= A) return;
    const int k = anchor_idx[a];
    if (k >= 0 && k < K) atomicOr(bits + (k >> 5), 1u << (k & 31));
}

// Nearest level of z = d / sd, lowest index on a tie, exactly as the fp64 quotient and the
// four fp64 distances decide it.  The decision only changes at the level midpoints -0.985, 0
// and +0.985 (within a few ulps of them, where rounding can tie two distances).  d * (1/sd) is
// within a few ulps of the quotient, so when it lies more than 1e-9 from every midpoint the
// side it lies on is the answer; otherwise the exact quotient and distances are computed.
// (`fast` is false when 1/sd is not a finite number, or sd is 0.)
__device__ __forceinline__ uint32_t nearest_level(double d, double sd, double inv_sd, bool fast) {
    if (fast) {
        const double za = __dmul_rn(d, inv_sd);
        const long long bits = __double_as_longlong(za);
        const long long mag = bits & 0x7FFFFFFFFFFFFFFFll;      // |za|, ordered as an integer
        if (mag > __double_as_longlong(1e-9) &&
            (mag < __double_as_longlong(0.985 - 1e-9) || mag > __double_as_longlong(0.985 + 1e-9))) {
            const uint32_t outer = mag > __double_as_longlong(0.985);
            return bits < 0 ? 1u - outer : 2u + outer;
        }
    }
    const double z = sd > 0.0 ? __ddiv_rn(d, sd) : 0.0;
    uint32_t best = 0;
    double bd = fabs(__dsub_rn(z, kLevels[0]));
#pragma unroll
    for (int k = 1; k < 4; ++k) {
        const double dk = fabs(__dsub_rn(z, kLevels[k]));
        if (dk < bd) {
            bd = dk;
            best = k;
        }
    }
    return best;
}

__device__ __forceinline__ double pick4(uint32_t q, double a0, double a1, double a2, double a3) {
    return (q & 2u) ? ((q & 1u) ? a3 : a2) : ((q & 1u) ? a1 : a0);
}

__global__ void __launch_bounds__(128) quantize_2bit_kernel(const float* __restrict__ W, int N, int K,
                                                            const uint32_t* __restrict__ bits,
                                                            uint8_t* __restrict__ codes, uint16_t* __restrict__ scales,
                                                            uint16_t* __restrict__ offsets) {
    const int groups = K / 32;
    const int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (t >= (int64_t)N * groups) return;
    const int64_t n = t / groups;
    const int g = (int)(t - n * groups);
    const uint32_t am = bits ? bits[g] : 0u;
    // the group's non-anchor values, in column order
    float v[32];
    int nv = 0;
    const float4* src = reinterpret_cast<const float4*>(W + n * K + 32 * g);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const float4 f = __ldg(src + i);
        const float e[4] = {f.x, f.y, f.z, f.w};
#pragma unroll
        for (int j = 0; j < 4; ++j)
            if (!((am >> (4 * i + j)) & 1u)) v[nv++] = e[j];
    }
    uint64_t packed = 0;
    double S = 0.0, Z = 0.0;
    if (nv > 0) {
        const double dn = (double)nv;
        const double mu = __ddiv_rn(pairwise_sum(nv, [&](int j) { return (double)v[j]; }), dn);
        const double var = __ddiv_rn(pairwise_sum(nv, [&](int j) {
                                         const double d = __dsub_rn((double)v[j], mu);
                                         return __dmul_rn(d, d);
                                     }), dn);
        const double sd = __dsqrt_rn(var);
        const double inv_sd = sd > 0.0 ? __ddiv_rn(1.0, sd) : 0.0;
        const bool fast = sd > 0.0 && isfinite(inv_sd);
        uint64_t q = 0;   // code of the j-th value in bits 2j..2j+1
        for (int j = 0; j < nv; ++j)
            q |= (uint64_t)nearest_level(__dsub_rn((double)v[j], mu), sd, inv_sd, fast) << (2 * j);
        auto code = [&](int j) { return (uint32_t)(q >> (2 * j)) & 3u; };
        const double c0 = kLevels[0], c1 = kLevels[1], c2 = kLevels[2], c3 = kLevels[3];
        const double cb = __ddiv_rn(pairwise_sum(nv, [&](int j) { return pick4(code(j), c0, c1, c2, c3); }), dn);
        // C_q - cb and its square take four values per group
        const double t0 = __dsub_rn(c0, cb), t1 = __dsub_rn(c1, cb), t2 = __dsub_rn(c2, cb), t3 = __dsub_rn(c3, cb);
        const double s0 = __dmul_rn(t0, t0), s1 = __dmul_rn(t1, t1), s2 = __dmul_rn(t2, t2), s3 = __dmul_rn(t3, t3);
        const double num = pairwise_sum(nv, [&](int j) {
            return __dmul_rn(__dsub_rn((double)v[j], mu), pick4(code(j), t0, t1, t2, t3));
        });
        const double den = __dadd_rn(pairwise_sum(nv, [&](int j) { return pick4(code(j), s0, s1, s2, s3); }), kOlsEps);
        S = __ddiv_rn(num, den);
        Z = __dsub_rn(mu, __dmul_rn(S, cb));
        // scatter the codes back to their columns (anchor columns keep code 0)
        int j = 0;
        for (int k = 0; k < 32; ++k) {
            if (!((am >> k) & 1u)) {
                packed |= ((q >> (2 * j)) & 3u) << (2 * k);
                ++j;
            }
        }
    }
    *reinterpret_cast<uint2*>(codes + n * (K / 4) + 8 * g) = make_uint2((uint32_t)packed, (uint32_t)(packed >> 32));
    scales[n * groups + g] = half_bits_rn(S);
    offsets[n * groups + g] = half_bits_rn(Z);
}

// anchor_w[n][a] = binary16(W[n][anchor_idx[a]]) for a < A, 0 for A <= a < ld_anchor.
__global__ void anchor_weights_kernel(const float* __restrict__ W, int N, int K, const int32_t* __restrict__ anchor_idx,
                                      int A, uint16_t* __restrict__ anchor_w, int ld_anchor) {
    const int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (t >= (int64_t)N * ld_anchor) return;
    const int64_t n = t / ld_anchor;
    const int a = (int)(t - n * ld_anchor);
    uint16_t h = 0;
    if (a < A) {
        const int k = anchor_idx[a];
        if (k >= 0 && k < K) h = __half_as_ushort(__float2half_rn(__ldg(W + n * K + k)));
    }
    anchor_w[t] = h;
}

// ---- NF4 block quantizer ----------------------------------------------------------

__global__ void __launch_bounds__(256) quantize_nf4_kernel(const float* __restrict__ W, int N, int K,
                                                           uint8_t* __restrict__ codes, float* __restrict__ absmax) {
    __shared__ double T[16];   // the levels in fp64, ascending
    if (threadIdx.x < 16) T[threadIdx.x] = (double)kNF4[threadIdx.x];
    __syncthreads();
    const int lane = threadIdx.x & 31;
    const int64_t blk = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int per_row = K / 64;
    if (blk >= (int64_t)N * per_row) return;
    const int64_t n = blk / per_row;
    const int b = (int)(blk - n * per_row);
    const float2 w = __ldg(reinterpret_cast<const float2*>(W + n * K + 64 * b) + lane);
    float m = fmaxf(fabsf(w.x), fabsf(w.y));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    const double am = (double)m;
    // argmin_k |r - T[k]| (lowest k on a tie) from the two levels around r: |r| <= 1 = T[15] = -T[0],
    // and every other level is at least 0.07 further from r than the nearer of the two, far more than
    // the fp64 rounding of a distance, so no other level can reach (or tie) their minimum.
    auto code = [&](float x) {
        const double r = am > 0.0 ? __ddiv_rn((double)x, am) : 0.0;
        int i = 0;   // the largest i with T[i] <= r
#pragma unroll
        for (int step = 8; step >= 1; step >>= 1)
            if (T[i + step] <= r) i += step;
        if (i == 15) return 15u;
        const double d0 = fabs(__dsub_rn(r, T[i])), d1 = fabs(__dsub_rn(r, T[i + 1]));
        return (uint32_t)(d1 < d0 ? i + 1 : i);
    };
    codes[n * (K / 2) + 32 * b + lane] = (uint8_t)(code(w.x) | (code(w.y) << 4));
    if (lane == 0) absmax[n * per_row + b] = m;
}

unsigned blocks_for(int64_t threads, int per_block) { return (unsigned)((threads + per_block - 1) / per_block); }

}  // namespace

lq_status launch_select_anchors(lq_handle h, const float* W, int N, int K, const double* profile, int A,
                                int32_t* anchor_idx, cudaStream_t stream) {
    if (A == 0) return LQ_OK;
    if ((size_t)K * sizeof(double) > h->partial_floats * sizeof(float)) return LQ_ERR_WORKSPACE;
    double* score = reinterpret_cast<double*>(h->partials);
    anchor_score_kernel<<<blocks_for(K, kScoreThreads), kScoreThreads, 0, stream>>>(W, N, K, profile, score);
    if (cudaPeekAtLastError() != cudaSuccess) return LQ_ERR_CUDA;
    anchor_select_kernel<<<1, kSelThreads, 0, stream>>>(score, K, A, anchor_idx);
    return cudaPeekAtLastError() == cudaSuccess ? LQ_OK : LQ_ERR_CUDA;
}

lq_status launch_quantize_2bit(lq_handle h, const float* W, int N, int K, const int32_t* anchor_idx, int A,
                               uint8_t* codes, uint16_t* scales, uint16_t* offsets, uint16_t* anchor_w, int ld_anchor,
                               cudaStream_t stream) {
    uint32_t* bits = nullptr;
    if (A > 0) {
        const size_t bytes = (size_t)(K / 32) * sizeof(uint32_t);
        if (bytes > h->partial_floats * sizeof(float)) return LQ_ERR_WORKSPACE;
        bits = reinterpret_cast<uint32_t*>(h->partials);
        if (cudaMemsetAsync(bits, 0, bytes, stream) != cudaSuccess) return LQ_ERR_CUDA;
        anchor_bits_kernel<<<blocks_for(A, 256), 256, 0, stream>>>(anchor_idx, A, K, bits);
        if (cudaPeekAtLastError() != cudaSuccess) return LQ_ERR_CUDA;
    }
    const int64_t groups = (int64_t)N * (K / 32);
    quantize_2bit_kernel<<<blocks_for(groups, 128), 128, 0, stream>>>(W, N, K, bits, codes, scales, offsets);
    if (cudaPeekAtLastError() != cudaSuccess) return LQ_ERR_CUDA;
    if (anchor_w && ld_anchor > 0) {
        anchor_weights_kernel<<<blocks_for((int64_t)N * ld_anchor, 256), 256, 0, stream>>>(W, N, K, anchor_idx, A,
                                                                                          anchor_w, ld_anchor);
        if (cudaPeekAtLastError() != cudaSuccess) return LQ_ERR_CUDA;
    }
    return LQ_OK;
}

lq_status launch_quantize_nf4(const float* W, int N, int K, uint8_t* codes, float* absmax, cudaStream_t stream) {
    const int64_t threads = (int64_t)N * (K / 64) * 32;
    quantize_nf4_kernel<<<blocks_for(threads, 256), 256, 0, stream>>>(W, N, K, codes, absmax);
    return cudaPeekAtLastError() == cudaSuccess ? LQ_OK : LQ_ERR_CUDA;
}

}  // namespace lq
