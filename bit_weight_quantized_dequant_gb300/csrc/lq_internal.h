// Host-side internals of liblq: the handle and the launch entry points that the
// C ABI (lq_api.cu) dispatches to after validating arguments.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <vector>

#include "../../include/lq.h"

struct lq_handle_s {
    int device = 0;
    int num_sms = 0;
    int max_smem_optin = 0;
    void* workspace = nullptr;          // device scratch: [counters | partial sums]
    size_t workspace_bytes = 0;
    unsigned* counters = nullptr;       // per-strip arrival counters (zero between calls)
    size_t num_counters = 0;
    float* partials = nullptr;          // split-K partial sums
    size_t partial_floats = 0;
    int* status_flag = nullptr;         // device word: nonzero after a bounded wait ran out
    int* sched = nullptr;               // grouped-GEMM tile lists, kept between calls with the same shapes
    size_t sched_ints = 0;
    std::vector<int64_t> sched_key;     // the shapes `sched` was built for
};

namespace lq {

constexpr int kMaxGroup = 16;           // problems per grouped GEMV launch
constexpr int kMaxGemmGroup = 8;        // problems per grouped GEMM launch
constexpr int kGemvStripRows = 64;      // output rows per GEMV thread block (4 warps x 16)
constexpr int kGemvThreads = 128;

// One problem of a grouped GEMV launch as the kernel sees it.
struct GemvDesc {
    const uint8_t* codes;
    const void* scales;
    const uint16_t* offsets;
    const int32_t* anchor_idx;
    const uint16_t* anchor_w;
    const void* x;
    void* y;
    int64_t stride_codes, stride_scales, stride_offsets, stride_anchor_idx, stride_anchor_w, stride_x, stride_y;
    int N, K, A, ld_anchor, batch;
    int KC;            // K columns per code split (multiple of 256 unless the split is the whole row)
    int S;             // code splits
    int parts;         // S, plus one anchor part when S > 1 and A > 0
    int strips;        // ceil(N / 64)
    int64_t unit_begin;   // first global unit of this problem
    int64_t strip_begin;  // first global strip (counters index)
    int64_t partial_begin;  // first float of this problem's split-K partial sums
    const uint32_t* xmax; // bf16 x: max |x| word of each (member, token) row of this problem
};

struct GemvParams {
    GemvDesc d[kMaxGroup];
    int count;
    int M;
    int format;
    int x_bf16;
    int y_dtype;
    int kc_pad;        // smem columns reserved for one code split (multiple of 256)
    int a_pad;         // smem columns reserved for anchors (multiple of 16)
    float* partials;
    unsigned* counters;
    int* status;       // device status word: bit 2 is raised when a weight table value overflows binary16
    int64_t total_units;
};

lq_status launch_dequant(lq_handle h, int format, const uint8_t* codes, const void* scales, const void* offsets,
                         const int32_t* anchor_idx, const uint16_t* anchor_w, int A, int ld_anchor, void* w_out,
                         int out_dtype, int N, int K, cudaStream_t stream);

// Device scratch a GEMV launch may use for split-K partial sums and arrival counters.
struct GemvWorkspace {
    int num_sms;
    int max_smem_optin;
    float* partials;
    size_t partial_floats;
    unsigned* counters;
    size_t num_counters;
    bool clear_counters;   // zero the counters this launch uses before it runs
    int* status;           // device word raised when a bounded wait runs out
};

lq_status launch_gemv(lq_handle h, const lq_problem* problems, int count, cudaStream_t stream);
lq_status launch_gemv_ws(const GemvWorkspace& ws, const lq_problem* problems, int count, cudaStream_t stream);
bool gemv_stream_eligible(const lq_problem* problems, int count);
lq_status launch_gemv_regs(const GemvWorkspace& ws, const lq_problem* problems, int count, cudaStream_t stream);
lq_status launch_gemv_stream(const GemvWorkspace& ws, const lq_problem* problems, int count, cudaStream_t stream);
// Consecutive layers of grouped calls (counts[l] problems each), one launch per layer in
// stream order; layer l may read what layer l - 1 wrote.
lq_status launch_gemv_layers(lq_handle h, const lq_problem* problems, const int* counts, int layers,
                             cudaStream_t stream);
// bf16 x: each (member, token) row's max |x| (fp32 bit pattern) into words[], rows in problem order.
lq_status launch_xmax_rows(const lq_problem* problems, int count, uint32_t* words, cudaStream_t stream);

lq_status launch_gemm(lq_handle h, const lq_problem& p, cudaStream_t stream);

lq_status launch_select_anchors(lq_handle h, const float* W, int N, int K, const double* profile, int A,
                                int32_t* anchor_idx, cudaStream_t stream);
lq_status launch_quantize_2bit(lq_handle h, const float* W, int N, int K, const int32_t* anchor_idx, int A,
                               uint8_t* codes, uint16_t* scales, uint16_t* offsets, uint16_t* anchor_w, int ld_anchor,
                               cudaStream_t stream);
lq_status launch_quantize_nf4(const float* W, int N, int K, uint8_t* codes, float* absmax, cudaStream_t stream);
lq_status launch_gemm_grouped(lq_handle h, const lq_problem* problems, int count, cudaStream_t stream);

}  // namespace lq
