// Layer streaming: one decode pass over a stack of layers whose packed weights live
// in host memory (the airllm README's layer-by-layer loading, "Efficient Memory
// Usage"; the otf-llm README section 1: decode reads every weight once per token).
//
// Two device slots hold layer weights.  Layer l is copied into slot l % 2 on a copy
// stream of this object while layer l - 1 computes on the caller's stream; the copy
// of layer l waits until layer l - 2 (the slot's previous user) has finished.  Each
// layer then runs one grouped GEMV on its slot.  Host code only: it enqueues copies
// (one cudaMemcpyAsync per layer), event waits and the GEMV launches.

#include <cuda_runtime.h>
#include <string.h>

#include <vector>

#include "lq_internal.h"

struct lq_layer_stream_s {
    lq_handle h = nullptr;
    size_t slot_bytes = 0;
    void* slot[2] = {nullptr, nullptr};
    cudaStream_t copy = nullptr;
    cudaEvent_t ready[2] = {nullptr, nullptr};   // slot filled (copy stream)
    cudaEvent_t freed[2] = {nullptr, nullptr};   // slot's layer computed (caller's stream)
    cudaEvent_t start = nullptr;                 // caller's stream reached the pass
};

namespace {

bool aligned16(uint64_t v) { return (v & 15u) == 0; }

// Bytes each weight array of a (batch 1) problem occupies.
void extents(const lq_problem& p, uint64_t (&ext)[5]) {
    const uint64_t N = (uint64_t)p.N, K = (uint64_t)p.K;
    const bool two = p.format == LQ_FMT_2BIT_LM_G32;
    ext[0] = two ? N * K / 4 : N * K / 2;                  // codes
    ext[1] = two ? N * (K / 32) * 2 : N * (K / 64) * 4;    // scales / absmax
    ext[2] = two ? N * (K / 32) * 2 : 0;                   // offsets
    ext[3] = two ? (uint64_t)p.A * 4 : 0;                  // anchor_idx
    ext[4] = two ? N * (uint64_t)p.ld_anchor * 2 : 0;      // anchor_w
}

// The weight fields of a layer's problems are byte offsets into the layer's bytes:
// each array must be 16-byte aligned and lie inside layer_bytes.
lq_status check_layer(const lq_problem* problems, int count, size_t layer_bytes) {
    for (int i = 0; i < count; ++i) {
        const lq_problem& p = problems[i];
        if (p.batch != 1 || p.N < 1 || p.K < 1) return LQ_ERR_INVALID_ARG;
        if (p.format == LQ_FMT_INT4_G32 || p.format == LQ_FMT_NF4_DQ)
            return LQ_ERR_UNSUPPORTED;   // (the stream object carries 2-bit and NF4 layers)
        if (p.format != LQ_FMT_2BIT_LM_G32 && p.format != LQ_FMT_NF4_B64) return LQ_ERR_INVALID_ARG;
        if (p.K % (p.format == LQ_FMT_2BIT_LM_G32 ? 32 : 64) != 0 || p.A < 0 || p.ld_anchor < 0) return LQ_ERR_INVALID_ARG;
        uint64_t ext[5];
        extents(p, ext);
        const uint64_t off[5] = {(uint64_t)(uintptr_t)p.codes, (uint64_t)(uintptr_t)p.scales,
                                 (uint64_t)(uintptr_t)p.offsets, (uint64_t)(uintptr_t)p.anchor_idx,
                                 (uint64_t)(uintptr_t)p.anchor_w};
        for (int a = 0; a < 5; ++a) {
            if (ext[a] == 0) continue;
            if (!aligned16(off[a])) return LQ_ERR_ALIGNMENT;
            if (off[a] > layer_bytes || ext[a] > layer_bytes - off[a]) return LQ_ERR_INVALID_ARG;
        }
    }
    return LQ_OK;
}

void destroy(lq_layer_stream s) {
    for (int i = 0; i < 2; ++i) {
        if (s->slot[i]) cudaFree(s->slot[i]);
        if (s->ready[i]) cudaEventDestroy(s->ready[i]);
        if (s->freed[i]) cudaEventDestroy(s->freed[i]);
    }
    if (s->start) cudaEventDestroy(s->start);
    if (s->copy) cudaStreamDestroy(s->copy);
    delete s;
}

}  // namespace

extern "C" {

LQ_API lq_status lq_stream_create(lq_layer_stream* out, lq_handle h, size_t slot_bytes) {
    if (!out || !h || slot_bytes == 0) return LQ_ERR_INVALID_ARG;
    *out = nullptr;
    int prev = -1;
    if (cudaGetDevice(&prev) != cudaSuccess || cudaSetDevice(h->device) != cudaSuccess) return LQ_ERR_CUDA;
    lq_layer_stream s = new lq_layer_stream_s();
    s->h = h;
    s->slot_bytes = slot_bytes;
    bool ok = cudaStreamCreateWithFlags(&s->copy, cudaStreamNonBlocking) == cudaSuccess &&
              cudaEventCreateWithFlags(&s->start, cudaEventDisableTiming) == cudaSuccess;
    for (int i = 0; ok && i < 2; ++i)
        ok = cudaMalloc(&s->slot[i], slot_bytes) == cudaSuccess &&
             cudaEventCreateWithFlags(&s->ready[i], cudaEventDisableTiming) == cudaSuccess &&
             cudaEventCreateWithFlags(&s->freed[i], cudaEventDisableTiming) == cudaSuccess;
    cudaSetDevice(prev);
    if (!ok) {
        destroy(s);
        return LQ_ERR_CUDA;
    }
    *out = s;
    return LQ_OK;
}

LQ_API lq_status lq_stream_destroy(lq_layer_stream s) {
    if (!s) return LQ_OK;
    int prev = -1;
    cudaGetDevice(&prev);
    cudaSetDevice(s->h->device);
    const lq_status st = cudaStreamSynchronize(s->copy) == cudaSuccess ? LQ_OK : LQ_ERR_CUDA;
    destroy(s);
    cudaSetDevice(prev);
    return st;
}

LQ_API lq_status lq_stream_run(lq_layer_stream s, const void* host_layers, size_t host_stride, size_t layer_bytes,
                               int L, const lq_problem* problems, int count, int64_t y_layer_stride, void* stream) {
    if (!s || !host_layers || !problems || L < 1 || count < 1 || layer_bytes == 0) return LQ_ERR_INVALID_ARG;
    if (count > lq::kMaxGroup) return LQ_ERR_UNSUPPORTED;
    if (layer_bytes > s->slot_bytes) return LQ_ERR_WORKSPACE;
    if (L > 1 && host_stride < layer_bytes) return LQ_ERR_INVALID_ARG;
    if (y_layer_stride < 0) return LQ_ERR_INVALID_ARG;
    if (!aligned16((uint64_t)(uintptr_t)host_layers) || !aligned16(host_stride) || !aligned16((uint64_t)y_layer_stride))
        return LQ_ERR_ALIGNMENT;
    lq_status v = check_layer(problems, count, layer_bytes);
    if (v != LQ_OK) return v;
    lq_handle h = s->h;
    int prev = -1;
    if (cudaGetDevice(&prev) != cudaSuccess || cudaSetDevice(h->device) != cudaSuccess) return LQ_ERR_CUDA;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    lq_status res = LQ_OK;
    std::vector<lq_problem> abs(problems, problems + count);
    // slots may still be read by the caller's earlier work, and by the last two layers of an
    // earlier pass (which may have run on another stream): the copies wait for both
    if (cudaEventRecord(s->start, st) != cudaSuccess || cudaStreamWaitEvent(s->copy, s->start, 0) != cudaSuccess ||
        cudaStreamWaitEvent(s->copy, s->freed[0], 0) != cudaSuccess ||
        cudaStreamWaitEvent(s->copy, s->freed[1], 0) != cudaSuccess)
        res = LQ_ERR_CUDA;
    for (int l = 0; l < L && res == LQ_OK; ++l) {
        const int k = l & 1;
        char* base = static_cast<char*>(s->slot[k]);
        if (l >= 2 && cudaStreamWaitEvent(s->copy, s->freed[k], 0) != cudaSuccess) {
            res = LQ_ERR_CUDA;
            break;
        }
        const char* src = static_cast<const char*>(host_layers) + (size_t)l * host_stride;
        if (cudaMemcpyAsync(base, src, layer_bytes, cudaMemcpyHostToDevice, s->copy) != cudaSuccess ||
            cudaEventRecord(s->ready[k], s->copy) != cudaSuccess || cudaStreamWaitEvent(st, s->ready[k], 0) != cudaSuccess) {
            res = LQ_ERR_CUDA;
            break;
        }
        for (int i = 0; i < count; ++i) {
            const lq_problem& p = problems[i];
            lq_problem& q = abs[i];
            q.codes = reinterpret_cast<const uint8_t*>(base + (uintptr_t)p.codes);
            q.scales = base + (uintptr_t)p.scales;
            q.offsets = p.format == LQ_FMT_2BIT_LM_G32 ? reinterpret_cast<const uint16_t*>(base + (uintptr_t)p.offsets) : nullptr;
            q.anchor_idx = p.A > 0 ? reinterpret_cast<const int32_t*>(base + (uintptr_t)p.anchor_idx) : nullptr;
            q.anchor_w = p.A > 0 ? reinterpret_cast<const uint16_t*>(base + (uintptr_t)p.anchor_w) : nullptr;
            q.y = static_cast<char*>(p.y) + (int64_t)l * y_layer_stride;
        }
        res = lq_gemv_grouped(h, abs.data(), count, stream);
        if (res == LQ_OK && cudaEventRecord(s->freed[k], st) != cudaSuccess) res = LQ_ERR_CUDA;
    }
    cudaSetDevice(prev);
    return res;
}

// The same pass with no copies: the kernels read each layer's weights from host
// memory themselves (over the CPU-GPU link).  The memory must be pinned memory with a
// device mapping that covers the whole stack (cudaPointerGetAttributes at its first
// and last byte); otherwise LQ_ERR_UNSUPPORTED and nothing is launched.
LQ_API lq_status lq_stream_run_direct(lq_handle h, const void* host_layers, size_t host_stride, size_t layer_bytes,
                                      int L, const lq_problem* problems, int count, int64_t y_layer_stride,
                                      void* stream) {
    if (!h || !host_layers || !problems || L < 1 || count < 1 || layer_bytes == 0) return LQ_ERR_INVALID_ARG;
    if (count > lq::kMaxGroup) return LQ_ERR_UNSUPPORTED;
    if (L > 1 && host_stride < layer_bytes) return LQ_ERR_INVALID_ARG;
    if (y_layer_stride < 0) return LQ_ERR_INVALID_ARG;
    if (!aligned16((uint64_t)(uintptr_t)host_layers) || !aligned16(host_stride) || !aligned16((uint64_t)y_layer_stride))
        return LQ_ERR_ALIGNMENT;
    lq_status v = check_layer(problems, count, layer_bytes);
    if (v != LQ_OK) return v;
    int prev = -1;
    if (cudaGetDevice(&prev) != cudaSuccess || cudaSetDevice(h->device) != cudaSuccess) return LQ_ERR_CUDA;
    // the device address of the host bytes, or UNSUPPORTED when the device cannot read them
    const char* dbase = nullptr;
    cudaPointerAttributes attr;
    memset(&attr, 0, sizeof(attr));
    if (cudaPointerGetAttributes(&attr, host_layers) != cudaSuccess) {
        cudaGetLastError();
        cudaSetDevice(prev);
        return LQ_ERR_CUDA;
    }
    if (attr.type != cudaMemoryTypeHost || attr.devicePointer == nullptr) {
        cudaSetDevice(prev);
        return LQ_ERR_UNSUPPORTED;
    }
    dbase = static_cast<const char*>(attr.devicePointer);
    // the whole range must belong to the same mapping (checked at its last byte)
    {
        cudaPointerAttributes last;
        memset(&last, 0, sizeof(last));
        const char* end = static_cast<const char*>(host_layers) + (size_t)(L - 1) * host_stride + layer_bytes - 1;
        if (cudaPointerGetAttributes(&last, end) != cudaSuccess || last.type != cudaMemoryTypeHost ||
            static_cast<const char*>(last.devicePointer) != dbase + (end - static_cast<const char*>(host_layers))) {
            cudaGetLastError();
            cudaSetDevice(prev);
            return LQ_ERR_UNSUPPORTED;
        }
    }
    std::vector<lq_problem> abs(problems, problems + count);
    lq_status res = LQ_OK;
    for (int l = 0; l < L && res == LQ_OK; ++l) {
        const char* base = dbase + (size_t)l * host_stride;
        for (int i = 0; i < count; ++i) {
            const lq_problem& p = problems[i];
            lq_problem& q = abs[i];
            q.codes = reinterpret_cast<const uint8_t*>(base + (uintptr_t)p.codes);
            q.scales = base + (uintptr_t)p.scales;
            q.offsets = p.format == LQ_FMT_2BIT_LM_G32 ? reinterpret_cast<const uint16_t*>(base + (uintptr_t)p.offsets) : nullptr;
            q.anchor_idx = p.A > 0 ? reinterpret_cast<const int32_t*>(base + (uintptr_t)p.anchor_idx) : nullptr;
            q.anchor_w = p.A > 0 ? reinterpret_cast<const uint16_t*>(base + (uintptr_t)p.anchor_w) : nullptr;
            q.y = static_cast<char*>(p.y) + (int64_t)l * y_layer_stride;
        }
        res = lq_gemv_grouped(h, abs.data(), count, stream);
    }
    cudaSetDevice(prev);
    return res;
}

}  // extern "C"
