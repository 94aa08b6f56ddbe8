// topk.h -- arguments, limits and launcher of the top-k sampling prologue
// (k_topk.cu), declared apart from launch.h so the row kernels do not depend
// on it.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "device_common.cuh"

namespace osr {

struct TopkArgs {
    const void *x;     // [M][N] input rows
    float *values;     // [M][k] the k largest values, largest first
    int64_t *indices;  // [M][k] their column indices
    float *probs;      // [M][k] softmax of the k values, may be null
    float *lse;        // [M] log-sum-exp of the whole row, may be null
    int64_t M, N, k;
    int64_t chunk;     // elements per cluster CTA (a multiple of the vector width)
    int cs;            // CTAs per row (cluster size)
    int sort_n;        // power of two >= k: the sorting network's width
    uint32_t region0;  // bytes of the piece / sort region at the start of shared memory
};

constexpr int kTopkThreads = 256;
constexpr int64_t kTopkMaxK = 1024;
constexpr int64_t kTopkMaxPieceBytes = 192 << 10;  // largest piece a CTA caches
// the sweep keeps one bit per 16-byte vector of a thread in a 64-bit word
static_assert(kTopkMaxPieceBytes / 16 / kTopkThreads <= 64, "vectors a thread sweeps");
constexpr int kTopkMaxCluster = 16;
constexpr int kTopkListCap = 1024;  // keys at or above a CTA's bound kept in a short list
constexpr int64_t kTopkRankMaxK = 256;  // k up to this: outputs placed by counting, no sort
constexpr int64_t kTopkMinWords = 2048;  // the piece region holds at least this many 8-byte words
// the kernel's static shared memory (1552 bytes as built), for the planner's
// estimate of CTAs per SM
constexpr int64_t kTopkStaticSmem = 1600;

// Dynamic shared memory of one CTA: piece (or sort buffer), the histogram,
// the published histogram (two buffers), the short list, the candidates.
inline size_t topk_smem_bytes(uint32_t region0, int64_t k) {
    return (size_t)region0 + 256 * 4 + 2 * 256 * 4 + (size_t)kTopkListCap * 8 + (size_t)k * 8;
}

template <Dt DI>
cudaError_t launch_topk(const TopkArgs &a, bool vec, size_t smem, cudaStream_t st);
template <Dt DI>
cudaError_t topk_occupancy(bool vec, int cs, size_t smem, int *n);

}  // namespace osr
