/*
 * lq.h — C ABI of liblq.so: fused dequantize-and-multiply for linear layers whose
 * weights are stored low-bit, on one GB300 (sm_103a).
 *
 * y[m][n] = sum_k x[m][k] * W_eff[n][k]      (x: M x K tokens, W: N x K, out x in)
 *
 * Weight formats
 * --------------
 * LQ_FMT_2BIT_LM_G32 — the otf-llm 4.0.1 README, "Theoretical & Mathematical
 *   Foundations": 2-bit codes q index the Lloyd-Max codebook
 *   C = {-1.52, -0.45, +0.45, +1.52} (section 2), a group of G = 32 consecutive
 *   input columns of one output row shares a binary16 scale S_g and offset Z_g
 *   fitted by least squares (section 3), and a sorted set of input columns
 *   ("outlier anchors", section 4) is kept exactly in binary16:
 *       W_eff[n][k] = fmaf(S_g, C[q], Z_g)          (fp32, one rounding)
 *       W_eff[n][anchor_idx[a]] = anchor_w[n][a]    (replaces the 2-bit value)
 *   Storage (all row-major, device memory):
 *       codes      uint8   [N][K/4]   column 4j+i of a row in bits 2i..2i+1 of byte j
 *       scales     binary16[N][K/32]  S_g
 *       offsets    binary16[N][K/32]  Z_g
 *       anchor_idx int32   [A]        strictly increasing columns in [0, K)
 *       anchor_w   binary16[N][ld_anchor], ld_anchor >= A, ld_anchor % 8 == 0
 *   Anchor columns store code 0 in `codes`; their code is never used.
 *
 * LQ_FMT_INT4_G32 — the same README's v3.2 engine ("Comparative Analysis: INT4
 *   (v3.2) vs INT2 Non-Uniform (v4.0)" and the "Method Comparison Table"): 2 weights
 *   per byte on a uniform grid with zero-point 0, input columns stored in a global
 *   static permutation, the top-1 % columns kept in binary16.  Position j of the
 *   permuted order holds input column perm[j]; 32 consecutive positions of a row
 *   share a binary16 scale S:
 *       W_eff[n][perm[j]] = S * q[n][j]     (fp32, exact; q a 4-bit two's complement)
 *       W_eff[n][anchor_idx[a]] = anchor_w[n][a]    (replaces the grid value)
 *   Storage: codes uint8 [N][K/2] (position 2j in the low nibble of byte j, 2j+1 in
 *   the high nibble), scales binary16 [N][K/32], `offsets` = perm int32 [K] (each
 *   column once), anchors as for the 2-bit format (anchor positions store q = 0).
 *
 * LQ_FMT_NF4_B64 — the AirQuant README, "Fundamentacao Teorica" item 2 (NF4,
 *   block-wise, the QLoRA NormalFloat data type): blocks of 64 consecutive input
 *   columns share an fp32 absmax, codes index the 16 NF4 levels T:
 *       W_eff[n][k] = T[q] * absmax_b                 (fp32, one rounding)
 *   Storage: codes uint8 [N][K/2] (column 2j in the low nibble of byte j, 2j+1 in
 *   the high nibble), scales = absmax float32 [N][K/64]; offsets, anchor_idx and
 *   anchor_w are NULL and A = 0.
 *
 * LQ_FMT_NF4_DQ — NF4 with double quantization (QLoRA, the method the AirQuant README
 *   cites for NF4): the block maxima themselves are stored as 8-bit floats (E4M3: bias
 *   7, 3 mantissa bits, no infinities, largest 448).  The maxima of a matrix, in
 *   row-major order of [N][K/64], form blocks of 256; with `second` = [mean, s2_0,
 *   s2_1, ...] (fp32):
 *       c'_i = fmaf(E4M3(acode_i), s2_(i/256), mean)   (fp32, one rounding)
 *       W_eff[n][k] = T[q] * c'_(n*(K/64) + k/64)      (fp32, one rounding)
 *   Storage: codes as for NF4; scales = acode uint8 [N][K/64]; offsets = second
 *   float32 [1 + ceil(N*K/64 / 256)]; anchor_idx and anchor_w NULL and A = 0.
 *   Decode (lq_gemv) needs K % 256 == 0.  lq_gemm decodes the maxima into fp32 in the
 *   handle's workspace (one small kernel per problem) and runs the NF4 GEMM on them.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - Ownership: the caller owns every buffer passed in.  The library owns the
 *   handle and the device workspace that lq_create allocates, and the two device
 *   slots that lq_stream_create allocates; no other call allocates memory.
 * - Asynchrony: compute calls enqueue work on `stream` (a cudaStream_t, NULL for
 *   the legacy default stream) and return without waiting.  A returned LQ_OK
 *   means the arguments were valid and the launch was accepted.
 * - Errors: arguments are validated on the host before anything is launched; an
 *   invalid call returns an error status and enqueues nothing.  No call traps
 *   on the device.  Device-side waits are bounded; a wait that runs out records
 *   a flag that lq_sync() reports as LQ_ERR_TIMEOUT.
 * - Alignment: every device pointer must be 16-byte aligned.
 * - Workspace: calls that split K across thread blocks keep partial sums and
 *   arrival counters in the handle's workspace.  One handle serves one stream
 *   at a time; calls on one handle that overlap on the GPU race.
 * - Device: a handle belongs to the device given to lq_create; calls switch to
 *   that device for the launch and switch back.
 * - Arithmetic: dequantized weights follow the definitions above exactly
 *   (lq_dequant is bit-exact).  lq_gemv multiplies binary16-rounded weights by
 *   binary16 x on tensor cores with fp32 accumulation (|error| <= 1e-3 *
 *   sum_k |W_eff||x|).  bf16 x: each token's x is scaled by the power of two that
 *   brings its largest |x| into [2^14, 2^15), rounded to binary16, and the fp32
 *   result is scaled back (both factors exact), so bf16 x of any finite magnitude
 *   keeps the bound.  Weight domain of lq_gemv (2-bit): the four table values
 *   fmaf(S, C[q], Z) of a group are rounded to binary16, so they must satisfy
 *   |S*C+Z| < 65520 (a group that breaks this raises LQ_ERR_RANGE at the next
 *   lq_sync); values below 2^-14 keep an absolute error of at most 2^-25, so the
 *   bound needs each row's weights to be mostly above that size (NF4: the levels
 *   T[q] are in [-1, 1] and absmax scales in fp32; no range limit).
 *   lq_gemm multiplies in the dtype of x (bf16 or binary16) with fp32
 *   accumulation (|error| <= 4e-3 * sum_k |W_eff||x| for bf16).  The quantizers'
 *   outputs (codes, scales, offsets, anchors, absmax) are deterministic bit
 *   patterns.
 * - CUDA graphs: compute calls may be captured into a graph once each shape has
 *   been called outside capture (the first call of a kernel variant sets its
 *   attributes; a grouped GEMM uploads its tile list when its shapes change).
 */
#ifndef LQ_H_
#define LQ_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(_WIN32)
#define LQ_API __declspec(dllexport)
#else
#define LQ_API __attribute__((visibility("default")))
#endif

typedef enum lq_status {
    LQ_OK = 0,
    LQ_ERR_INVALID_ARG = 1,   /* null pointer, bad size, bad enum, unsorted anchors ... */
    LQ_ERR_UNSUPPORTED = 2,   /* valid but not handled by this entry point (e.g. M out of range) */
    LQ_ERR_ALIGNMENT = 3,     /* a pointer or leading dimension breaks the 16-byte rule */
    LQ_ERR_WORKSPACE = 4,     /* the handle's workspace is too small for this call */
    LQ_ERR_CUDA = 5,          /* a CUDA runtime call or launch failed */
    LQ_ERR_TIMEOUT = 6,       /* a bounded device-side wait ran out (reported by lq_sync) */
    LQ_ERR_RANGE = 7          /* a decode GEMV met a weight table value |S*C+Z| >= 65520, outside the
                                 binary16 range of its tensor-core operands (reported by lq_sync) */
} lq_status;

typedef enum lq_format {
    LQ_FMT_2BIT_LM_G32 = 1,
    LQ_FMT_NF4_B64 = 2,
    LQ_FMT_INT4_G32 = 3,
    LQ_FMT_NF4_DQ = 4
} lq_format;

typedef enum lq_dtype {
    LQ_F32 = 0,
    LQ_F16 = 1,
    LQ_BF16 = 2
} lq_dtype;

typedef struct lq_handle_s* lq_handle;

/*
 * One problem of a grouped call: `batch` independent products of the same
 * shape.  Member b of the batch reads and writes at the base pointers plus
 * b * stride_* BYTES.  Pointers, strides and layouts as described above; x is
 * [M][K] and y is [M][N], both row-major.
 */
typedef struct lq_problem {
    int format;                /* lq_format */
    int M, N, K;
    const uint8_t* codes;
    const void* scales;        /* binary16 S_g (2-bit, INT4), fp32 absmax (NF4) or E4M3 maxima (NF4-DQ) */
    const void* offsets;       /* binary16 Z_g (2-bit), int32 perm[K] (INT4), NULL (NF4) or fp32 second level (NF4-DQ) */
    const int32_t* anchor_idx; /* 2-bit and INT4, may be NULL when A == 0 */
    const uint16_t* anchor_w;  /* 2-bit and INT4, may be NULL when A == 0 */
    int A;
    int ld_anchor;
    const void* x;
    int x_dtype;               /* LQ_F16 or LQ_BF16 */
    void* y;
    int y_dtype;               /* LQ_F32, LQ_F16 or LQ_BF16 */
    int batch;                 /* >= 1 */
    int64_t stride_codes, stride_scales, stride_offsets, stride_anchor_idx, stride_anchor_w;
    int64_t stride_x, stride_y;
} lq_problem;

/*
 * lq_create — make a handle for CUDA device `device`.
 *   workspace_bytes: device scratch for split-K partial sums and counters;
 *   0 selects the default (256 MiB).  Allocated and zeroed here, once.
 *   Returns LQ_ERR_INVALID_ARG for a null `out` or a bad device, LQ_ERR_CUDA when
 *   the allocation fails.  On failure *out is set to NULL.
 */
LQ_API lq_status lq_create(lq_handle* out, int device, size_t workspace_bytes);

/* lq_destroy — synchronize the handle's device and free the handle and its workspace. NULL is a no-op. */
LQ_API lq_status lq_destroy(lq_handle h);

/* lq_status_string — static English text for a status code; never NULL. */
LQ_API const char* lq_status_string(int status);

/*
 * lq_sync — wait for the device and report errors raised on it: LQ_ERR_CUDA for
 * an asynchronous CUDA error, LQ_ERR_TIMEOUT when a bounded device wait ran out
 * since the last lq_sync (the flag is cleared).
 */
LQ_API lq_status lq_sync(lq_handle h);

/*
 * lq_dequant — W_eff as dense [N][K] in out_dtype (LQ_F32, LQ_F16 or LQ_BF16).
 * fp32 output is bit-exact to the definitions above; binary16/bf16 outputs are
 * the round-to-nearest-even conversion of that fp32 value.
 * Format rules: K % 32 == 0 (2-bit) or K % 64 == 0 (NF4); N >= 1; anchors as above.
 */
LQ_API lq_status lq_dequant(lq_handle h, int format,
                            const uint8_t* codes, const void* scales, const void* offsets,
                            const int32_t* anchor_idx, const uint16_t* anchor_w, int A, int ld_anchor,
                            void* w_out, int out_dtype, int N, int K, void* stream);

/*
 * lq_gemv — decode-sized product y = x * W_eff^T for 1 <= M <= 32 tokens, the
 * weights streamed once and dequantized in registers, the anchor columns folded
 * into the same fp32 accumulator.  x: [M][K] binary16 or bf16; y: [M][N] in
 * y_dtype.  LQ_ERR_UNSUPPORTED for M outside 1..32, and for INT4 or NF4-DQ when
 * K % 256 != 0.
 */
LQ_API lq_status lq_gemv(lq_handle h, int format,
                         const uint8_t* codes, const void* scales, const void* offsets,
                         const int32_t* anchor_idx, const uint16_t* anchor_w, int A, int ld_anchor,
                         const void* x, int x_dtype, void* y, int y_dtype,
                         int M, int N, int K, void* stream);

/*
 * lq_gemv_grouped — several lq_gemv problems (e.g. the seven projections of one
 * decoder layer, or many small matrices as a batch) in ONE launch.  `problems`
 * is a host array of `count` entries, read before the call returns.  All
 * problems must share format, M, x_dtype and y_dtype.
 */
LQ_API lq_status lq_gemv_grouped(lq_handle h, const lq_problem* problems, int count, void* stream);

/*
 * lq_gemv_layers — consecutive decode layers in one call: layer l is a grouped
 * call of counts[l] problems (lq_gemv_grouped's rules), taken in order from
 * `problems` (host array of sum(counts) entries, read before the call returns).
 * Layer l's problems may read, as x, what any earlier layer of the call wrote as
 * y (an LLM decode step: the next layer's input is the previous layer's output);
 * results are those of one lq_gemv_grouped call per layer, in order, and that is
 * how it runs: one launch per layer on `stream`, each overlapping its start with
 * the end of the launch before (programmatic dependent launch).  Errors as
 * lq_gemv_grouped; LQ_ERR_INVALID_ARG for layers < 1 or a count < 1.  (The
 * decode loop this serves is the memory-bound one of the otf-llm README, "The
 * Memory-Bound Bottleneck in Autoregressive LLM Decoding": one pass over every
 * layer's weights per generated token.)
 */
LQ_API lq_status lq_gemv_layers(lq_handle h, const lq_problem* problems, const int* counts, int layers, void* stream);

/*
 * lq_gemm — prefill-sized product for M >= 1 (tuned for M >= 256) on the
 * tcgen05 tensor cores, run by clusters of two CTAs (one per SM) that share each
 * 256-row x 256-token tile through one cta_group::2 MMA: each CTA TMA-loads its
 * half of the x tile and dequantizes its 128 weight rows into its tensor memory,
 * the fp32 accumulator lives in tensor memory, and the anchor columns are
 * appended as extra K-blocks of the same accumulator.  LQ_ERR_UNSUPPORTED when
 * the device cannot hold one such pair.
 * x: [M][K] bf16 or binary16 (the multiply runs in that dtype); y: [M][N] in
 * y_dtype.  K % 64 == 0, every format.  INT4 first writes x in the permuted
 * column order into the handle's workspace (M * K values per problem), and NF4-DQ
 * its decoded block maxima (N * K / 64 floats per problem); LQ_ERR_WORKSPACE when
 * they do not fit.
 */
LQ_API lq_status lq_gemm(lq_handle h, int format,
                         const uint8_t* codes, const void* scales, const void* offsets,
                         const int32_t* anchor_idx, const uint16_t* anchor_w, int A, int ld_anchor,
                         const void* x, int x_dtype, void* y, int y_dtype,
                         int M, int N, int K, void* stream);

/*
 * lq_gemm_grouped — several lq_gemm problems (e.g. the seven projections of one
 * decoder layer at prefill) in ONE persistent launch.  `problems` is a host
 * array of `count` (1..8) entries, read before the call returns; batch must be
 * 1 (strides ignored).  All problems share format and x_dtype; M, N, K, anchors
 * and y_dtype may differ.  The CTA pairs' tile lists balance the problems' K-blocks
 * (longest first); the lists are built on the host and kept in the handle's
 * workspace, so the first call with new shapes waits for their upload (the
 * stream is synchronized once) and later calls with the same shapes do not.
 * Errors as lq_gemm; LQ_ERR_UNSUPPORTED for count > 8 or mixed format/x_dtype.
 */
LQ_API lq_status lq_gemm_grouped(lq_handle h, const lq_problem* problems, int count, void* stream);

/*
 * lq_gemv_noalloc — lq_gemv for callers that cannot allocate device memory.
 * The paper has no counterpart to this entry point; it exists for deployment.
 *
 * Some callers may not call cudaMalloc at all: a plugin running inside a host
 * application whose own allocator owns every byte of device memory, or a
 * service that must not grow or fragment its memory after start-up.  Such a
 * caller cannot create an lq handle, because lq_create allocates the handle's
 * workspace.  This entry point takes no handle and allocates nothing (no
 * cudaMalloc, cudaFree or allocating library call).  The caller still provides
 * x, y and the packed weights; the scratch is a fixed file-scope device array of
 * 8.06 MiB (16384 arrival counters + 2^21 fp32 words) that every GPU loading the
 * library holds until the process exits.
 *
 * - Runs on the CURRENT device.  Its first call on a device looks up the
 *   array's device address (cudaGetSymbolAddress); make that first call before
 *   any stream capture.
 * - Scratch needs (fp32 words), as for lq_gemv: K % 256 == 0 uses a copy of x in
 *   the kernels' layout (about M * (K + A) / 2 words; none for small problems at
 *   up to 8 tokens, which build it in shared memory) plus one 16- or 32-row slot
 *   of M * rows words per warp that shares a row block; otherwise the split-K
 *   kernel uses M * 64 words per 64-row strip per K-split (plus one split for the
 *   anchors), and one word per token for bf16 x.  A launch that does not fit the
 *   streaming kernel's needs falls back to split-K; one that fits neither returns
 *   LQ_ERR_WORKSPACE before anything is launched.
 * - All calls share the one array: each call clears the counters it uses on
 *   `stream` before its kernel runs, and calls that overlap on the GPU (other
 *   streams, other threads) race and give wrong results.
 * - There is no handle and no lq_sync here, so nothing reports device-side status:
 *   the decode kernels have no waits to time out, and a weight past the binary16
 *   range (LQ_ERR_RANGE through lq_gemv) is not reported.
 * Arguments, layouts, results and the other errors are those of lq_gemv.
 */
LQ_API lq_status lq_gemv_noalloc(int format,
                                 const uint8_t* codes, const void* scales, const void* offsets,
                                 const int32_t* anchor_idx, const uint16_t* anchor_w, int A, int ld_anchor,
                                 const void* x, int x_dtype, void* y, int y_dtype,
                                 int M, int N, int K, void* stream);

/* ---- Quantizers: the converter step that produces the formats above ----------
 *
 * These run the quantizers of the formats' definitions on the GPU, so that a caller
 * with fp32 weights in device memory can produce the stored formats in place.  Every
 * output is deterministic and equal bit for bit to an fp64 evaluation of the
 * definitions below with sums in a fixed pairwise order (eight interleaved partial
 * sums along a group, row by row down a column).  W is fp32 [N][K] row-major, finite.
 * Ownership, asynchrony, device and error rules are the shared ones; the selection
 * and the 2-bit quantizer use the handle's workspace (K doubles, K/8 bytes).
 */

/*
 * lq_select_anchors — outlier anchor columns (otf-llm 4.0.1 README, section 4):
 *     score_c = sqrt(sum_n W[n][c]^2) * profile[c]          (fp64)
 * the A largest scores, ties to the lower column, written to anchor_idx[A]
 * (int32, device) in ascending column order.  profile: fp64 [K] in device memory,
 * non-negative (mean |X_c| of a calibration profile), or NULL for all ones.  The
 * README keeps the top 3.5 %: A < 0 selects lq_anchor_count(K) columns (anchor_idx
 * must then hold that many).  0 <= A <= K otherwise; A = 0 launches nothing.
 * Errors: LQ_ERR_INVALID_ARG (shape, NULL), LQ_ERR_ALIGNMENT (W, profile or
 * anchor_idx not 16-byte aligned), LQ_ERR_WORKSPACE (K doubles do not fit).
 */
/* lq_anchor_count — the otf-llm README's outlier-anchor count for K input columns
 * (section 4, "Top-3.5%"): floor(0.035 * K), computed exactly as (35 K) / 1000;
 * 0 for K <= 0.  Host-only, needs no device. */
LQ_API int lq_anchor_count(int K);

LQ_API lq_status lq_select_anchors(lq_handle h, const float* W, int N, int K, const double* profile, int A,
                                   int32_t* anchor_idx, void* stream);

/*
 * lq_quantize_2bit — the 2-bit Lloyd-Max G = 32 quantizer (otf-llm 4.0.1 README,
 * sections 2-4).  For each row n and group g (columns 32g..32g+31), with V the
 * group's columns that are not anchors:
 *     mu = mean(W_V), sd = population std of W_V           (fp64)
 *     z  = (W - mu) / sd, or 0 when sd == 0
 *     q  = argmin_k |z - C_k|, C = {-1.52, -0.45, 0.45, 1.52}, lowest k on a tie
 *     S  = sum (W - mu)(C_q - mean C_q) / (sum (C_q - mean C_q)^2 + 1e-12)
 *     Z  = mu - S * mean C_q
 *     scales[n][g] = binary16(S), offsets[n][g] = binary16(Z)   (round to nearest even)
 * A group whose columns are all anchors stores S = Z = 0.  Anchor columns store
 * code 0, and anchor_w[n][a] = binary16(W[n][anchor_idx[a]]) for a < A, 0 up to
 * ld_anchor.  Outputs use the storage layout of LQ_FMT_2BIT_LM_G32 (codes
 * [N][K/4], scales/offsets [N][K/32], anchor_w [N][ld_anchor]).  anchor_idx:
 * strictly increasing columns in [0, K) (LQ_VALIDATE=1 checks them on the host;
 * otherwise a column outside [0, K) is ignored).  Rules: K % 32 == 0, N >= 1,
 * 0 <= A <= K, ld_anchor >= A and % 8 == 0 when A > 0 (anchor_idx and anchor_w may
 * be NULL when A = 0).  Errors: LQ_ERR_INVALID_ARG, LQ_ERR_ALIGNMENT,
 * LQ_ERR_WORKSPACE.
 */
LQ_API lq_status lq_quantize_2bit(lq_handle h, const float* W, int N, int K, const int32_t* anchor_idx, int A,
                                  uint8_t* codes, uint16_t* scales, uint16_t* offsets, uint16_t* anchor_w,
                                  int ld_anchor, void* stream);

/*
 * lq_quantize_nf4 — NF4 block-64 quantizer (AirQuant README, "Fundamentacao
 * Teorica" item 2; the QLoRA NormalFloat levels T):
 *     absmax_b = max |w| over the block (fp32, exact)
 *     q = argmin_k |w / absmax_b - T[k]| in fp64, lowest k on a tie (0 when absmax_b = 0
 *         gives the index of the level 0)
 * Outputs use the LQ_FMT_NF4_B64 layout: codes uint8 [N][K/2], absmax float32
 * [N][K/64].  Rules: K % 64 == 0, N >= 1.  Errors: LQ_ERR_INVALID_ARG,
 * LQ_ERR_ALIGNMENT.
 */
LQ_API lq_status lq_quantize_nf4(lq_handle h, const float* W, int N, int K, uint8_t* codes, float* absmax,
                                 void* stream);

/* ---- Layer streaming: decode over a stack whose weights live in host memory ------
 *
 * The airllm README ("Efficient Memory Usage") runs models larger than GPU memory by
 * loading one layer at a time; the otf-llm README (section 1) notes that decode
 * reads every weight once per token.  An lq_layer_stream holds two device slots of
 * slot_bytes each, a copy stream and events.  lq_stream_run runs the L layers of a
 * stack in order on `stream`:
 *   - layer l's packed weights are the layer_bytes bytes at
 *     host_layers + l * host_stride (host memory; pinned memory makes the copies
 *     asynchronous and lets them overlap the computation);
 *   - they are copied (one cudaMemcpyAsync) into slot l % 2 on the object's copy
 *     stream, after the layer that used that slot before (l - 2) has finished, so the
 *     copy of layer l runs while layer l - 1 computes;
 *   - layer l then runs lq_gemv_grouped(problems) on `stream` against its slot.
 * `problems` (count <= 16, batch 1) describe one layer: their codes, scales,
 * offsets, anchor_idx and anchor_w fields hold BYTE OFFSETS into the layer's bytes
 * (cast to pointers; each 16-byte aligned and inside layer_bytes); x and y are device
 * pointers; layer l writes y at y + l * y_layer_stride bytes (0: every layer writes
 * the same y).  Every layer has the same problem list, as in a decoder stack.
 * lq_stream_create allocates the slots (the one allocating call besides
 * lq_create); lq_stream_destroy waits for the copy stream and frees them.  A stream
 * object serves one pass at a time; its handle's workspace rules apply.
 * Errors: LQ_ERR_INVALID_ARG (shapes, offsets outside the layer),
 * LQ_ERR_ALIGNMENT, LQ_ERR_WORKSPACE (layer_bytes > slot_bytes), LQ_ERR_UNSUPPORTED
 * (count > 16, or an INT4 or NF4-DQ layer: the stream carries 2-bit and NF4 layers),
 * then those of lq_gemv_grouped; LQ_ERR_CUDA from the runtime.
 */
typedef struct lq_layer_stream_s* lq_layer_stream;

LQ_API lq_status lq_stream_create(lq_layer_stream* out, lq_handle h, size_t slot_bytes);
LQ_API lq_status lq_stream_run(lq_layer_stream s, const void* host_layers, size_t host_stride, size_t layer_bytes,
                               int L, const lq_problem* problems, int count, int64_t y_layer_stride, void* stream);
LQ_API lq_status lq_stream_destroy(lq_layer_stream s);

/*
 * lq_stream_run_direct — the same pass with no copies and no slots: the GEMV kernels
 * read each layer's weights straight from host memory over the CPU-GPU link.
 * host_layers must be pinned memory with a device mapping that covers the whole
 * stack (checked with cudaPointerGetAttributes at its first and last byte; otherwise
 * LQ_ERR_UNSUPPORTED and nothing is launched).  Other arguments and errors are those
 * of lq_stream_run.
 */
LQ_API lq_status lq_stream_run_direct(lq_handle h, const void* host_layers, size_t host_stride, size_t layer_bytes,
                                      int L, const lq_problem* problems, int count, int64_t y_layer_stride,
                                      void* stream);

/*
 * lq_selftest_wait — exercises the timeout path of the kernels' bounded waits.  One
 * thread of one CTA waits, with the routine the pipelined kernels use, on a
 * shared-memory barrier that nothing completes.  After limit_us microseconds
 * (1 .. 1000000) the wait gives up, raises the handle's status word and the kernel
 * returns; the next lq_sync reports LQ_ERR_TIMEOUT and clears the status word and
 * the arrival counters.  Nothing faults and the context stays usable.  Errors:
 * LQ_ERR_INVALID_ARG (null handle, limit out of range), LQ_ERR_CUDA.
 */
LQ_API lq_status lq_selftest_wait(lq_handle h, unsigned limit_us, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* LQ_H_ */
