// The C ABI of liblq: handle management, host-side argument validation and
// dispatch to the kernels.  Nothing is launched unless every check passes.

#include <cuda_runtime.h>
#include <stdlib.h>
#include <string.h>

#include <mutex>
#include <vector>

#include "lq_internal.h"

namespace {

constexpr size_t kDefaultWorkspace = 256ull << 20;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool valid_dtype(int d) { return d == LQ_F32 || d == LQ_F16 || d == LQ_BF16; }

// Restores the caller's current device on scope exit.
struct DeviceGuard {
    int prev = -1;
    bool ok = true;
    explicit DeviceGuard(int dev) {
        if (cudaGetDevice(&prev) != cudaSuccess) {
            ok = false;
            return;
        }
        if (prev != dev && cudaSetDevice(dev) != cudaSuccess) ok = false;
    }
    ~DeviceGuard() {
        int cur = -1;
        if (prev >= 0 && cudaGetDevice(&cur) == cudaSuccess && cur != prev) cudaSetDevice(prev);
    }
};

bool env_validate() {
    const char* v = getenv("LQ_VALIDATE");
    return v && v[0] == '1';
}

// Optional deep check (LQ_VALIDATE=1): anchor_idx strictly increasing in [0, K).
// Reads device memory, so it synchronizes the stream.
lq_status check_anchor_order(const int32_t* anchor_idx, int A, int K, cudaStream_t stream) {
    if (A <= 0 || !env_validate()) return LQ_OK;
    std::vector<int32_t> host(A);
    if (cudaMemcpyAsync(host.data(), anchor_idx, sizeof(int32_t) * A, cudaMemcpyDeviceToHost, stream) != cudaSuccess)
        return LQ_ERR_CUDA;
    if (cudaStreamSynchronize(stream) != cudaSuccess) return LQ_ERR_CUDA;
    for (int a = 0; a < A; ++a) {
        if (host[a] < 0 || host[a] >= K) return LQ_ERR_INVALID_ARG;
        if (a > 0 && host[a] <= host[a - 1]) return LQ_ERR_INVALID_ARG;
    }
    return LQ_OK;
}

// Shape, pointer and alignment rules shared by every compute entry point.
lq_status check_weights(int format, const uint8_t* codes, const void* scales, const void* offsets,
                        const int32_t* anchor_idx, const uint16_t* anchor_w, int A, int ld_anchor, int N, int K) {
    if (format != LQ_FMT_2BIT_LM_G32 && format != LQ_FMT_NF4_B64 && format != LQ_FMT_INT4_G32 &&
        format != LQ_FMT_NF4_DQ)
        return LQ_ERR_INVALID_ARG;
    if (N < 1 || K < 1) return LQ_ERR_INVALID_ARG;
    if (!codes || !scales) return LQ_ERR_INVALID_ARG;
    if (!aligned16(codes) || !aligned16(scales)) return LQ_ERR_ALIGNMENT;
    if (format == LQ_FMT_2BIT_LM_G32 || format == LQ_FMT_INT4_G32) {
        if (K % 32 != 0) return LQ_ERR_INVALID_ARG;
        if (!offsets) return LQ_ERR_INVALID_ARG;   // (binary16 Z_g, or the INT4 permutation)
        if (!aligned16(offsets)) return LQ_ERR_ALIGNMENT;
        if (A < 0 || A > K) return LQ_ERR_INVALID_ARG;
        if (A > 0) {
            if (!anchor_idx || !anchor_w) return LQ_ERR_INVALID_ARG;
            if (ld_anchor < A) return LQ_ERR_INVALID_ARG;
            if (!aligned16(anchor_idx) || !aligned16(anchor_w) || ld_anchor % 8 != 0) return LQ_ERR_ALIGNMENT;
        }
    } else {
        if (K % 64 != 0) return LQ_ERR_INVALID_ARG;
        if (A != 0 || anchor_idx || anchor_w) return LQ_ERR_INVALID_ARG;
        if (format == LQ_FMT_NF4_DQ) {   // (offsets: the second-level constants [mean, s2_0, ...])
            if (!offsets) return LQ_ERR_INVALID_ARG;
            if (!aligned16(offsets)) return LQ_ERR_ALIGNMENT;
        }
    }
    return LQ_OK;
}

lq_status check_problem(const lq_problem& p) {
    lq_status s = check_weights(p.format, p.codes, p.scales, p.offsets, p.anchor_idx, p.anchor_w, p.A, p.ld_anchor,
                                p.N, p.K);
    if (s != LQ_OK) return s;
    if (!p.x || !p.y) return LQ_ERR_INVALID_ARG;
    if (!aligned16(p.x) || !aligned16(p.y)) return LQ_ERR_ALIGNMENT;
    if (p.x_dtype != LQ_F16 && p.x_dtype != LQ_BF16) return LQ_ERR_INVALID_ARG;
    if (!valid_dtype(p.y_dtype)) return LQ_ERR_INVALID_ARG;
    if (p.batch < 1) return LQ_ERR_INVALID_ARG;
    if (p.batch > 1) {
        const int64_t st[] = {p.stride_codes, p.stride_scales, p.stride_offsets, p.stride_anchor_idx,
                              p.stride_anchor_w, p.stride_x, p.stride_y};
        for (int64_t v : st)
            if (v < 0) return LQ_ERR_INVALID_ARG;
        for (int64_t v : st)
            if (v % 16 != 0) return LQ_ERR_ALIGNMENT;
    }
    return LQ_OK;
}

lq_problem make_problem(int format, const uint8_t* codes, const void* scales, const void* offsets,
                        const int32_t* anchor_idx, const uint16_t* anchor_w, int A, int ld_anchor, const void* x,
                        int x_dtype, void* y, int y_dtype, int M, int N, int K) {
    lq_problem p;
    memset(&p, 0, sizeof(p));
    p.format = format;
    p.M = M;
    p.N = N;
    p.K = K;
    p.codes = codes;
    p.scales = scales;
    p.offsets = offsets;   // (a binary16 array, or the INT4 permutation)
    p.anchor_idx = anchor_idx;
    p.anchor_w = anchor_w;
    p.A = A;
    p.ld_anchor = ld_anchor;
    p.x = x;
    p.x_dtype = x_dtype;
    p.y = y;
    p.y_dtype = y_dtype;
    p.batch = 1;
    return p;
}

}  // namespace

extern "C" {

LQ_API const char* lq_status_string(int status) {
    switch (status) {
        case LQ_OK: return "ok";
        case LQ_ERR_INVALID_ARG: return "invalid argument";
        case LQ_ERR_UNSUPPORTED: return "unsupported by this entry point";
        case LQ_ERR_ALIGNMENT: return "pointer, stride or leading dimension breaks the 16-byte alignment rule";
        case LQ_ERR_WORKSPACE: return "handle workspace too small for this call";
        case LQ_ERR_CUDA: return "CUDA error";
        case LQ_ERR_TIMEOUT: return "a bounded device-side wait ran out";
        case LQ_ERR_RANGE: return "a dequantized weight is outside the binary16 range of the decode GEMV's operands";
        default: return "unknown status";
    }
}

LQ_API lq_status lq_create(lq_handle* out, int device, size_t workspace_bytes) {
    if (!out) return LQ_ERR_INVALID_ARG;
    *out = nullptr;
    int count = 0;
    if (cudaGetDeviceCount(&count) != cudaSuccess) return LQ_ERR_CUDA;
    if (device < 0 || device >= count) return LQ_ERR_INVALID_ARG;
    DeviceGuard guard(device);
    if (!guard.ok) return LQ_ERR_CUDA;
    lq_handle h = new lq_handle_s();
    h->device = device;
    if (cudaDeviceGetAttribute(&h->num_sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess ||
        cudaDeviceGetAttribute(&h->max_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, device) != cudaSuccess) {
        delete h;
        return LQ_ERR_CUDA;
    }
    const size_t bytes = workspace_bytes ? workspace_bytes : kDefaultWorkspace;
    if (bytes < (1u << 16)) {
        delete h;
        return LQ_ERR_INVALID_ARG;
    }
    if (cudaMalloc(&h->workspace, bytes) != cudaSuccess) {
        delete h;
        return LQ_ERR_CUDA;
    }
    if (cudaMemset(h->workspace, 0, bytes) != cudaSuccess || cudaDeviceSynchronize() != cudaSuccess) {
        cudaFree(h->workspace);
        delete h;
        return LQ_ERR_CUDA;
    }
    h->workspace_bytes = bytes;
    // layout: [status word (256 B) | counters (1/16 of the rest) | partial sums | GEMM tile lists (1/64)]
    char* base = static_cast<char*>(h->workspace);
    h->status_flag = reinterpret_cast<int*>(base);
    const size_t rest = bytes - 256;
    const size_t counter_bytes = (rest / 16) & ~size_t(255);
    const size_t sched_bytes = (rest / 64) & ~size_t(255);
    h->counters = reinterpret_cast<unsigned*>(base + 256);
    h->num_counters = counter_bytes / sizeof(unsigned);
    h->partials = reinterpret_cast<float*>(base + 256 + counter_bytes);
    h->partial_floats = (rest - counter_bytes - sched_bytes) / sizeof(float);
    h->sched = reinterpret_cast<int*>(base + bytes - sched_bytes);
    h->sched_ints = sched_bytes / sizeof(int);
    *out = h;
    return LQ_OK;
}

LQ_API lq_status lq_destroy(lq_handle h) {
    if (!h) return LQ_OK;
    lq_status st = LQ_OK;
    {
        DeviceGuard guard(h->device);
        if (!guard.ok || cudaDeviceSynchronize() != cudaSuccess) st = LQ_ERR_CUDA;
        if (h->workspace && cudaFree(h->workspace) != cudaSuccess) st = LQ_ERR_CUDA;
    }
    delete h;
    return st;
}

LQ_API lq_status lq_sync(lq_handle h) {
    if (!h) return LQ_ERR_INVALID_ARG;
    DeviceGuard guard(h->device);
    if (!guard.ok) return LQ_ERR_CUDA;
    if (cudaDeviceSynchronize() != cudaSuccess) return LQ_ERR_CUDA;
    int flag = 0;
    if (cudaMemcpy(&flag, h->status_flag, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return LQ_ERR_CUDA;
    if (flag & 1) {
        // a wait ran out: the launch that timed out may have left arrival counts behind, so they
        // are cleared with the flag
        if (cudaMemset(h->status_flag, 0, 256) != cudaSuccess ||
            cudaMemset(h->counters, 0, h->num_counters * sizeof(unsigned)) != cudaSuccess ||
            cudaDeviceSynchronize() != cudaSuccess)
            return LQ_ERR_CUDA;
        return LQ_ERR_TIMEOUT;
    }
    if (flag & 2) {
        // a decode GEMV met a weight outside the binary16 range of its tensor-core operands
        if (cudaMemset(h->status_flag, 0, 256) != cudaSuccess || cudaDeviceSynchronize() != cudaSuccess)
            return LQ_ERR_CUDA;
        return LQ_ERR_RANGE;
    }
    return LQ_OK;
}

LQ_API lq_status lq_dequant(lq_handle h, int format, const uint8_t* codes, const void* scales,
                            const void* offsets, const int32_t* anchor_idx, const uint16_t* anchor_w, int A,
                            int ld_anchor, void* w_out, int out_dtype, int N, int K, void* stream) {
    if (!h) return LQ_ERR_INVALID_ARG;
    lq_status s = check_weights(format, codes, scales, offsets, anchor_idx, anchor_w, A, ld_anchor, N, K);
    if (s != LQ_OK) return s;
    if (!w_out) return LQ_ERR_INVALID_ARG;
    if (!aligned16(w_out)) return LQ_ERR_ALIGNMENT;
    if (!valid_dtype(out_dtype)) return LQ_ERR_INVALID_ARG;
    DeviceGuard guard(h->device);
    if (!guard.ok) return LQ_ERR_CUDA;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if ((s = check_anchor_order(anchor_idx, A, K, st)) != LQ_OK) return s;
    return lq::launch_dequant(h, format, codes, scales, offsets, anchor_idx, anchor_w, A, ld_anchor, w_out, out_dtype,
                              N, K, st);
}

LQ_API lq_status lq_gemv_grouped(lq_handle h, const lq_problem* problems, int count, void* stream) {
    if (!h || !problems || count < 1) return LQ_ERR_INVALID_ARG;
    if (count > lq::kMaxGroup) return LQ_ERR_UNSUPPORTED;
    for (int i = 0; i < count; ++i) {
        lq_status s = check_problem(problems[i]);
        if (s != LQ_OK) return s;
        if (problems[i].M < 1 || problems[i].M > 32) return LQ_ERR_UNSUPPORTED;
        if (problems[i].format != problems[0].format || problems[i].M != problems[0].M ||
            problems[i].x_dtype != problems[0].x_dtype || problems[i].y_dtype != problems[0].y_dtype)
            return LQ_ERR_UNSUPPORTED;
    }
    DeviceGuard guard(h->device);
    if (!guard.ok) return LQ_ERR_CUDA;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    for (int i = 0; i < count; ++i) {
        if (problems[i].batch == 1 || problems[i].stride_anchor_idx == 0) {
            lq_status s = check_anchor_order(problems[i].anchor_idx, problems[i].A, problems[i].K, st);
            if (s != LQ_OK) return s;
        }
    }
    return lq::launch_gemv(h, problems, count, st);
}

LQ_API lq_status lq_gemv_layers(lq_handle h, const lq_problem* problems, const int* counts, int layers, void* stream) {
    if (!h || !problems || !counts || layers < 1) return LQ_ERR_INVALID_ARG;
    int total = 0;
    for (int l = 0; l < layers; ++l) {
        if (counts[l] < 1) return LQ_ERR_INVALID_ARG;
        if (counts[l] > lq::kMaxGroup) return LQ_ERR_UNSUPPORTED;
        const lq_problem* g = problems + total;
        for (int i = 0; i < counts[l]; ++i) {
            lq_status s = check_problem(g[i]);
            if (s != LQ_OK) return s;
            if (g[i].M < 1 || g[i].M > 32) return LQ_ERR_UNSUPPORTED;
            if (g[i].format != g[0].format || g[i].M != g[0].M || g[i].x_dtype != g[0].x_dtype ||
                g[i].y_dtype != g[0].y_dtype)
                return LQ_ERR_UNSUPPORTED;
        }
        total += counts[l];
    }
    DeviceGuard guard(h->device);
    if (!guard.ok) return LQ_ERR_CUDA;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    for (int i = 0; i < total; ++i) {
        if (problems[i].batch == 1 || problems[i].stride_anchor_idx == 0) {
            lq_status s = check_anchor_order(problems[i].anchor_idx, problems[i].A, problems[i].K, st);
            if (s != LQ_OK) return s;
        }
    }
    return lq::launch_gemv_layers(h, problems, counts, layers, st);
}

LQ_API lq_status lq_gemv(lq_handle h, int format, const uint8_t* codes, const void* scales, const void* offsets,
                         const int32_t* anchor_idx, const uint16_t* anchor_w, int A, int ld_anchor, const void* x,
                         int x_dtype, void* y, int y_dtype, int M, int N, int K, void* stream) {
    lq_problem p = make_problem(format, codes, scales, offsets, anchor_idx, anchor_w, A, ld_anchor, x, x_dtype, y,
                                y_dtype, M, N, K);
    return lq_gemv_grouped(h, &p, 1, stream);
}

LQ_API lq_status lq_gemm(lq_handle h, int format, const uint8_t* codes, const void* scales, const void* offsets,
                         const int32_t* anchor_idx, const uint16_t* anchor_w, int A, int ld_anchor, const void* x,
                         int x_dtype, void* y, int y_dtype, int M, int N, int K, void* stream) {
    if (!h) return LQ_ERR_INVALID_ARG;
    lq_problem p = make_problem(format, codes, scales, offsets, anchor_idx, anchor_w, A, ld_anchor, x, x_dtype, y,
                                y_dtype, M, N, K);
    lq_status s = check_problem(p);
    if (s != LQ_OK) return s;
    if (M < 1) return LQ_ERR_INVALID_ARG;
    if (K % 64 != 0) return LQ_ERR_UNSUPPORTED;
    DeviceGuard guard(h->device);
    if (!guard.ok) return LQ_ERR_CUDA;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if ((s = check_anchor_order(anchor_idx, A, K, st)) != LQ_OK) return s;
    return lq::launch_gemm(h, p, st);
}

LQ_API lq_status lq_gemm_grouped(lq_handle h, const lq_problem* problems, int count, void* stream) {
    if (!h || !problems || count < 1) return LQ_ERR_INVALID_ARG;
    if (count > lq::kMaxGemmGroup) return LQ_ERR_UNSUPPORTED;
    for (int i = 0; i < count; ++i) {
        const lq_problem& p = problems[i];
        const lq_status s = check_problem(p);
        if (s != LQ_OK) return s;
        if (p.M < 1 || p.batch != 1) return LQ_ERR_UNSUPPORTED;
        if (p.K % 64 != 0) return LQ_ERR_UNSUPPORTED;
        if (p.format != problems[0].format || p.x_dtype != problems[0].x_dtype) return LQ_ERR_UNSUPPORTED;
    }
    DeviceGuard guard(h->device);
    if (!guard.ok) return LQ_ERR_CUDA;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    for (int i = 0; i < count; ++i) {
        const lq_status s = check_anchor_order(problems[i].anchor_idx, problems[i].A, problems[i].K, st);
        if (s != LQ_OK) return s;
    }
    return lq::launch_gemm_grouped(h, problems, count, st);
}

// ---- quantizers ------------------------------------------------------------------

LQ_API int lq_anchor_count(int K) {
    // the otf-llm README's top 3.5 % of input columns, floor(0.035 K), in exact integer arithmetic
    return K > 0 ? (int)(((int64_t)K * 35) / 1000) : 0;
}

LQ_API lq_status lq_select_anchors(lq_handle h, const float* W, int N, int K, const double* profile, int A,
                                   int32_t* anchor_idx, void* stream) {
    if (A < 0) A = lq_anchor_count(K);
    if (!h || !W || N < 1 || K < 1 || A > K) return LQ_ERR_INVALID_ARG;
    if (A > 0 && !anchor_idx) return LQ_ERR_INVALID_ARG;
    if (!aligned16(W) || (profile && !aligned16(profile)) || (anchor_idx && !aligned16(anchor_idx)))
        return LQ_ERR_ALIGNMENT;
    DeviceGuard guard(h->device);
    if (!guard.ok) return LQ_ERR_CUDA;
    return lq::launch_select_anchors(h, W, N, K, profile, A, anchor_idx, static_cast<cudaStream_t>(stream));
}

LQ_API lq_status lq_quantize_2bit(lq_handle h, const float* W, int N, int K, const int32_t* anchor_idx, int A,
                                  uint8_t* codes, uint16_t* scales, uint16_t* offsets, uint16_t* anchor_w,
                                  int ld_anchor, void* stream) {
    if (!h || !W || !codes || !scales || !offsets) return LQ_ERR_INVALID_ARG;
    if (N < 1 || K < 1 || K % 32 != 0 || A < 0 || A > K) return LQ_ERR_INVALID_ARG;
    if (!aligned16(W) || !aligned16(codes) || !aligned16(scales) || !aligned16(offsets)) return LQ_ERR_ALIGNMENT;
    if (A > 0) {
        if (!anchor_idx || !anchor_w || ld_anchor < A) return LQ_ERR_INVALID_ARG;
        if (!aligned16(anchor_idx) || !aligned16(anchor_w) || ld_anchor % 8 != 0) return LQ_ERR_ALIGNMENT;
    } else if (anchor_w && (ld_anchor < 0 || ld_anchor % 8 != 0 || !aligned16(anchor_w))) {
        return LQ_ERR_ALIGNMENT;
    }
    DeviceGuard guard(h->device);
    if (!guard.ok) return LQ_ERR_CUDA;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    lq_status s = check_anchor_order(anchor_idx, A, K, st);
    if (s != LQ_OK) return s;
    return lq::launch_quantize_2bit(h, W, N, K, anchor_idx, A, codes, scales, offsets, anchor_w, anchor_w ? ld_anchor : 0,
                                    st);
}

LQ_API lq_status lq_quantize_nf4(lq_handle h, const float* W, int N, int K, uint8_t* codes, float* absmax,
                                 void* stream) {
    if (!h || !W || !codes || !absmax) return LQ_ERR_INVALID_ARG;
    if (N < 1 || K < 1 || K % 64 != 0) return LQ_ERR_INVALID_ARG;
    if (!aligned16(W) || !aligned16(codes) || !aligned16(absmax)) return LQ_ERR_ALIGNMENT;
    DeviceGuard guard(h->device);
    if (!guard.ok) return LQ_ERR_CUDA;
    return lq::launch_quantize_nf4(W, N, K, codes, absmax, static_cast<cudaStream_t>(stream));
}

// ---- the allocation-free GEMV entry point ---------------------------------------
//
// Scratch for split-K partial sums and arrival counters lives in this file-scope
// device array instead of a handle's cudaMalloc'd workspace.  Every GPU that loads
// the library holds it until the process exits.  In host code the array's name is
// only a host-side stand-in, so its device address is looked up once per device
// (cudaGetSymbolAddress, with that device current) and passed to the kernel.

namespace {

constexpr size_t kStaticCounters = 16384;           // 64 KiB of arrival counters
constexpr size_t kStaticPartialFloats = 2u << 20;   // 8 MiB of split-K partial sums
constexpr size_t kStaticScratchBytes = kStaticCounters * sizeof(unsigned) + kStaticPartialFloats * sizeof(float);
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

struct StaticScratchSlot {
    bool ready = false;
    void* base = nullptr;
    int num_sms = 0;
    int max_smem_optin = 0;
};

std::mutex g_static_mutex;
StaticScratchSlot g_static_slots[kMaxDevices];

// Device address of the scratch array on the current device (set up on first use).
lq_status static_scratch(StaticScratchSlot& out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return LQ_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return LQ_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_static_mutex);
    StaticScratchSlot& slot = g_static_slots[dev];
    if (!slot.ready) {
        void* ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_static_scratch) != cudaSuccess || ptr == nullptr) return LQ_ERR_CUDA;
        if (cudaDeviceGetAttribute(&slot.num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&slot.max_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
            return LQ_ERR_CUDA;
        slot.base = ptr;
        slot.ready = true;
    }
    out = slot;
    return LQ_OK;
}

}  // namespace

LQ_API lq_status lq_gemv_noalloc(int format, const uint8_t* codes, const void* scales, const void* offsets,
                                 const int32_t* anchor_idx, const uint16_t* anchor_w, int A, int ld_anchor,
                                 const void* x, int x_dtype, void* y, int y_dtype, int M, int N, int K,
                                 void* stream) {
    lq_problem p = make_problem(format, codes, scales, offsets, anchor_idx, anchor_w, A, ld_anchor, x, x_dtype, y,
                                y_dtype, M, N, K);
    lq_status s = check_problem(p);
    if (s != LQ_OK) return s;
    if (M < 1 || M > 32) return LQ_ERR_UNSUPPORTED;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if ((s = check_anchor_order(anchor_idx, A, K, st)) != LQ_OK) return s;
    StaticScratchSlot slot;
    if ((s = static_scratch(slot)) != LQ_OK) return s;
    lq::GemvWorkspace ws;
    ws.num_sms = slot.num_sms;
    ws.max_smem_optin = slot.max_smem_optin;
    ws.counters = static_cast<unsigned*>(slot.base);
    ws.num_counters = kStaticCounters;
    ws.status = nullptr;   // (no handle, so no lq_sync to report device-side status through)
    ws.partials = reinterpret_cast<float*>(static_cast<char*>(slot.base) + kStaticCounters * sizeof(unsigned));
    ws.partial_floats = kStaticPartialFloats;
    ws.clear_counters = true;
    return lq::launch_gemv_ws(ws, &p, 1, st);
}

}  // extern "C"
