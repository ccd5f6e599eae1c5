// Hessian accumulation H += 2 X^T X for bf16 X on the fifth-generation tensor
// cores (tcgen05, TMEM accumulators, TMA loads).  Placeholder until the kernel
// lands: the SIMT float32 GEMM serves every shape meanwhile.
#include "common.cuh"

namespace gq {

bool hessian_bf16_tc_supported(int64_t cols, const void *X, int64_t ldx) {
    (void)cols; (void)X; (void)ldx;
    return false;
}

cudaError_t hessian_bf16_tc(float *H, int64_t cols, const __nv_bfloat16 *X, int64_t n, int64_t ldx, cudaStream_t s) {
    (void)H; (void)cols; (void)X; (void)n; (void)ldx; (void)s;
    return cudaErrorNotSupported;
}

}  // namespace gq
