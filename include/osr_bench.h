/*
 * osr_bench.h -- measurement helpers that ship with the library but are not
 * part of the row-wise path: a 128-bit device-to-device copy kernel and the
 * runtime's device-to-device memcpy, used to measure the achievable HBM
 * bandwidth in the same run as the row kernels.
 */
#ifndef OSR_BENCH_H
#define OSR_BENCH_H

#include <stddef.h>

#include "osr.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * dst[0, bytes) <- src[0, bytes) with 16-byte loads and streaming 16-byte
 * stores, grid-stride over (4 x SM count) CTAs of 512 threads.
 *   src, dst  device pointers, 16-byte aligned, non-overlapping
 *   bytes     a multiple of 16 (0 is a no-op)
 * Returns OSR_ERR_INVALID on a NULL pointer, misalignment or a size that is
 * not a multiple of 16, OSR_ERR_ALIAS on overlap, OSR_ERR_CUDA on a launch
 * failure.  Asynchronous on `stream`.
 */
osr_status osr_bench_copy(const void *src, void *dst, size_t bytes, void *stream);

/*
 * dst[0, bytes) <- src[0, bytes) by the runtime's cudaMemcpyAsync
 * (device to device): a second reading of the achievable copy bandwidth,
 * beside the copy kernel above.  Same arguments and errors as
 * osr_bench_copy; any size and alignment.  Asynchronous on `stream`.
 */
osr_status osr_bench_memcpy(const void *src, void *dst, size_t bytes, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* OSR_BENCH_H */
