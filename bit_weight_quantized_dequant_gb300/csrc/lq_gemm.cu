// lq_gemm: prefill-sized product on tcgen05 tensor cores (placeholder until the
// tensor-memory kernel lands).
#include "lq_internal.h"

namespace lq {

lq_status launch_gemm(lq_handle, const lq_problem&, cudaStream_t) { return LQ_ERR_UNSUPPORTED; }

}  // namespace lq
