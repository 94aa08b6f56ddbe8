// staged.h -- shapes and launcher of the staged softmax tier (k_staged.cu),
// declared apart from launch.h so the register-cached row kernels do not
// depend on it.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>

#include "row_common.cuh"

namespace osr {

// Kernel shapes: (threads per CTA, 16-byte units a thread holds in
// registers).  The rest of each CTA's piece is bulk-copied into shared memory.
// Measured against 128 threads of 16 units (96 registers, five CTAs an SM):
// within 2 % either way, up to 20 % slower on some shapes.
constexpr int kStagedThreads = 256;            // shared-memory-only CTAs
constexpr int kStagedRegThreads = 256;         // CTAs holding part of the piece in registers ...
constexpr int kStagedRegUnits = 8;             // ... this many units a thread (64 registers)
constexpr int kStagedPieceIoBytes = 80 << 10;  // bytes a CTA reads and writes, without registers
constexpr int kStagedMaxSmem = 200 << 10;      // largest staged piece + header
constexpr int kStagedRegPieceBytes = 76 << 10; // largest piece when part of it is in registers
constexpr int kStagedMaxCluster = 16;          // CTAs per row at most

// Whether (threads, ru) is one of the compiled kernel shapes.
constexpr bool staged_shape_ok(int threads, int ru) {
    return (threads == kStagedThreads && ru == 0) ||
           (threads == kStagedRegThreads && ru == kStagedRegUnits);
}

// grid = rows * a.cs CTAs of `threads`, clusters of a.cs, `smem` bytes of
// dynamic shared memory; each thread holds `ru` units of its CTA's piece in
// registers.
template <Dt DI, Dt DO>
cudaError_t launch_softmax_staged(const RowArgs &a, int64_t grid, size_t smem, int threads, int ru,
                                  cudaStream_t st);
// Resident clusters of cs CTAs the shape could have at once.
template <Dt DI, Dt DO>
cudaError_t softmax_staged_occupancy(int cs, size_t smem, int threads, int ru, int *n);

}  // namespace osr
