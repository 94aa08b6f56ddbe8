// launch.h -- host-side plan and launcher declarations shared by the
// dispatcher (dispatch.cu) and the per-dtype kernel translation units.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>
#include <stdlib.h>

#include "row_common.cuh"

namespace osr {

enum class Op : int { RmsNorm = 0, FusedAddRmsNorm = 1, Softmax = 2, LayerNorm = 3 };

// Rows    : register-cached, one group / CTA per row        (one launch)
// Cluster : register-cached, a CTA cluster per row (DSMEM)  (one launch)
// Split   : S CTAs per row, partials in a workspace         (two launches)
// Staged  : softmax only, 16-byte rows: a cluster per row, each CTA's piece
//           bulk-copied into shared memory                  (one launch)
enum class Tier : int { Rows = 0, Cluster = 1, Split = 2, Staged = 3 };

// Which kernel of a tier a launch runs.
enum class Kind : int { Rows = 0, Cluster = 1, SplitStats = 2, SplitApply = 3 };

constexpr int kEpt = 16;           // elements per thread per tile (softmax; fp32 norms)
// Single-input norm kernels on 16-byte bfloat16 rows keep them packed, so a
// thread can hold 32 elements (64 bytes of loads in flight, like 16 fp32
// elements): measured 14 % faster for LayerNorm bf16 8192 x 4096.  The fused
// kernel already reads two rows per thread and measured 5 % slower with 32.
template <Dt D, int U, bool FUSED = false>
constexpr int norm_ept() {
    return D == Dt::BF16 && U == 8 && !FUSED ? 32 : 16;
}
// Softmax on 16-byte bfloat16 rows: 32 elements per thread in the register
// tiers, so a thread keeps 64 bytes of loads in flight like the fp32 kernels
// (the cached values are fp32 either way).  The split-row kernels stay at 16:
// at 32 the pass-2 kernel needs 99 registers, one 512-thread CTA per SM.
template <Dt DI, int U>
constexpr int softmax_ept() {
    return DI == Dt::BF16 && U == 8 ? 32 : 16;
}
constexpr int kSplitThreads = 512;  // threads per split-row CTA
constexpr int kMaxPieces = kSplitThreads;

// Launch with programmatic dependent launch (default on; OSR_PDL=0 turns it
// off).  Read once per process.
inline bool use_pdl() {
    static const bool on = [] {
        const char *e = getenv("OSR_PDL");
        return !(e && e[0] == '0');
    }();
    return on;
}

struct Plan {
    Tier tier = Tier::Rows;
    int g = 1;               // threads per row (Rows) or per CTA (Cluster, Split)
    int cs = 1;              // Cluster: CTAs per row; Split: pieces per row
    int64_t chunk = 0;       // Cluster / Split: units per CTA piece
    int64_t batch_rows = 0;  // Split: rows per (pass 1, pass 2) pair
    size_t smem = 0;         // Staged: dynamic shared memory per CTA
    bool vec = true;         // 16-byte units (true) or element units
    int u = 1;               // elements per unit
    int ept = kEpt;          // elements per thread per tile
    int ru = 0;              // Staged: 16-byte units a thread holds in registers
    bool forced = false;
};

// Launch one kernel of the given kind for a dtype combination.  `grid` is the
// number of CTAs; Cluster launches use a.cs as the cluster size.
template <Dt DI, Dt DO>
cudaError_t launch_softmax(Kind k, const RowArgs &a, int g, bool vec, int64_t grid,
                           cudaStream_t st);
template <Dt D, bool FUSED>
cudaError_t launch_rmsnorm(Kind k, const RowArgs &a, int g, bool vec, int64_t grid,
                           cudaStream_t st);

template <Dt D>
cudaError_t launch_layernorm(Kind k, const RowArgs &a, int g, bool vec, int64_t grid,
                             cudaStream_t st);
template <Dt D>
cudaError_t layernorm_cluster_occupancy(int g, bool vec, int cs, int *n);

// Resident clusters of cs CTAs the cluster kernel could have at once
// (cudaOccupancyMaxActiveClusters); 0 means the shape cannot be scheduled.
template <Dt DI, Dt DO>
cudaError_t softmax_cluster_occupancy(int g, bool vec, int cs, int *n);
template <Dt D, bool FUSED>
cudaError_t rmsnorm_cluster_occupancy(int g, bool vec, int cs, int *n);

// Per-row log-sum-exp and argmax (k_lse.cu): g threads per row (g <= 32:
// 128-thread CTAs of 128/g rows) or 256-thread CTAs; cluster: a.cs CTAs per
// row over pieces of a.chunk units.  Results go to a.row_sum / a.row_arg.
template <Dt DI>
cudaError_t launch_lse(const RowArgs &a, int g, bool cluster, bool vec, int64_t grid,
                       cudaStream_t st);
// Staged variant (16-byte rows): a.cs CTAs per row, each bulk-copying its
// piece of a.chunk units into `smem` bytes of shared memory (128 + piece).
template <Dt DI>
cudaError_t launch_lse_staged(const RowArgs &a, int64_t grid, size_t smem, cudaStream_t st);

}  // namespace osr
