// gemm_tc.cu -- small-batch (M >= 9) decode-GEMM on the tcgen05 tensor cores.
#include "q4_internal.cuh"

namespace q4 {
namespace {
// Sticky device-side error word (e.g. a bounded mbarrier wait that ran out).
__device__ int g_device_error;
}  // namespace

cudaError_t launch_gemm_tc(const Tensor &, const void *, q4_dtype, float *, int64_t, cudaStream_t,
                           bool *handled) {
    *handled = false;
    return cudaSuccess;
}

int gemv_read_and_clear_error();

int read_and_clear_device_error() {
    int v = 0;
    const int zero = 0;
    if (cudaDeviceSynchronize() != cudaSuccess) return Q4_ECUDA;
    if (cudaMemcpyFromSymbol(&v, g_device_error, sizeof(v)) != cudaSuccess) return Q4_ECUDA;
    if (cudaMemcpyToSymbol(g_device_error, &zero, sizeof(zero)) != cudaSuccess) return Q4_ECUDA;
    const int g = gemv_read_and_clear_error();
    return v ? v : g;
}

}  // namespace q4

extern "C" int q4_last_error(void) { return q4::read_and_clear_device_error(); }
