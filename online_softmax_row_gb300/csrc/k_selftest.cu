// k_selftest.cu -- test support (include/osr_test.h): the kernels' exponential
// evaluated beside CUDA's expf, so tests can hold it to its error bound.
#include <cuda_runtime.h>

#include "../../include/osr_test.h"
#include "device_common.cuh"

namespace osr {
namespace {

__global__ void exp_shifted_kernel(const float *x, const float *m, float *approx, float *ref,
                                   int64_t n) {
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
         i += (int64_t)gridDim.x * blockDim.x) {
        approx[i] = exp_shifted(x[i], m[i]);
        ref[i] = expf(x[i] - m[i]);
    }
}

}  // namespace
}  // namespace osr

extern "C" osr_status osr_test_exp_shifted(const float *x, const float *m, float *approx, float *ref,
                                           int64_t n, void *stream) {
    if (n < 0 || !x || !m || !approx || !ref) return OSR_ERR_INVALID;
    if (n == 0) return OSR_OK;
    const int64_t blocks = (n + 255) / 256;
    osr::exp_shifted_kernel<<<(unsigned)(blocks < 4096 ? blocks : 4096), 256, 0, (cudaStream_t)stream>>>(
        x, m, approx, ref, n);
    if (cudaGetLastError() != cudaSuccess) return OSR_ERR_CUDA;
    return OSR_OK;
}
