// Self-test of the timeout path shared by the pipelined kernels: one thread waits,
// with the same bounded-wait routine, on a shared-memory barrier that nothing
// completes.  The wait gives up after the requested time, raises the handle's
// status word and the kernel returns; lq_sync then reports LQ_ERR_TIMEOUT.

#include <cuda_runtime.h>

#include "lq_internal.h"
#include "lq_tma.cuh"

namespace lq {
namespace {

__global__ void selftest_wait_kernel(int* status, unsigned long long limit_ns) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x != 0) return;
    abort_flag = 0;
    mbar_init(smem_u32(&bar), 1);   // one arrival completes phase 0; none is ever made
    fence_mbar_init();
    mbar_wait_bounded(smem_u32(&bar), 0, &abort_flag, status, limit_ns);
}

}  // namespace
}  // namespace lq

extern "C" LQ_API lq_status lq_selftest_wait(lq_handle h, unsigned limit_us, void* stream) {
    if (!h || limit_us == 0 || limit_us > 1000000u) return LQ_ERR_INVALID_ARG;
    int prev = -1;
    if (cudaGetDevice(&prev) != cudaSuccess || cudaSetDevice(h->device) != cudaSuccess) return LQ_ERR_CUDA;
    lq::selftest_wait_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(h->status_flag,
                                                                             1000ull * (unsigned long long)limit_us);
    const lq_status st = cudaPeekAtLastError() == cudaSuccess ? LQ_OK : LQ_ERR_CUDA;
    cudaSetDevice(prev);
    return st;
}
