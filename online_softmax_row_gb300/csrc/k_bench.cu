// k_bench.cu -- 128-bit copy kernel and device-to-device memcpy for the
// measured HBM peak (include/osr_bench.h).
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/osr_bench.h"

namespace {

__global__ void __launch_bounds__(512) copy16_kernel(const uint4 *__restrict__ src,
                                                      uint4 *__restrict__ dst, int64_t n) {
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    // four independent 16-byte loads in flight per thread, then four stores
    for (; i + 3 * stride < n; i += 4 * stride) {
        const uint4 a = __ldcs(src + i), b = __ldcs(src + i + stride);
        const uint4 c = __ldcs(src + i + 2 * stride), d = __ldcs(src + i + 3 * stride);
        __stcs(dst + i, a);
        __stcs(dst + i + stride, b);
        __stcs(dst + i + 2 * stride, c);
        __stcs(dst + i + 3 * stride, d);
    }
    for (; i < n; i += stride) __stcs(dst + i, __ldcs(src + i));
}

}  // namespace

extern "C" osr_status osr_bench_copy(const void *src, void *dst, size_t bytes, void *stream) {
    if (bytes == 0) return OSR_OK;
    if (!src || !dst || (bytes & 15) || ((uintptr_t)src & 15) || ((uintptr_t)dst & 15))
        return OSR_ERR_INVALID;
    const char *s = (const char *)src, *d = (const char *)dst;
    if (s < d + bytes && d < s + bytes) return OSR_ERR_ALIAS;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return OSR_ERR_CUDA;
    copy16_kernel<<<4 * sms, 512, 0, (cudaStream_t)stream>>>((const uint4 *)src, (uint4 *)dst,
                                                              (int64_t)(bytes / 16));
    return cudaGetLastError() == cudaSuccess ? OSR_OK : OSR_ERR_CUDA;
}

extern "C" osr_status osr_bench_memcpy(const void *src, void *dst, size_t bytes, void *stream) {
    if (bytes == 0) return OSR_OK;
    if (!src || !dst) return OSR_ERR_INVALID;
    const char *s = (const char *)src, *d = (const char *)dst;
    if (s < d + bytes && d < s + bytes) return OSR_ERR_ALIAS;
    if (cudaMemcpyAsync(dst, src, bytes, cudaMemcpyDeviceToDevice, (cudaStream_t)stream) != cudaSuccess) {
        cudaGetLastError();
        return OSR_ERR_CUDA;
    }
    return OSR_OK;
}
