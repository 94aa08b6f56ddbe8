// lse.h -- what the log-sum-exp planner needs to know of the kernels in
// k_lse.cu, apart from launch.h.
#pragma once

#include <cuda_runtime.h>

#include "device_common.cuh"
#include "row_common.cuh"

namespace osr {

// CTAs an SM the streaming cluster kernel is compiled to hold (its launch
// bound: registers are capped to fit), which the planner counts on
constexpr int lse_cluster_ctas_per_sm(Dt d) { return d == Dt::BF16 ? 5 : 4; }

// The streaming kernels on rows that are not 16-byte aligned or not a whole
// number of vectors long: each row's aligned body in vectors, its head and
// tail elements folded in one a lane (g >= the vector width; cluster: 256).
template <Dt DI>
cudaError_t launch_lse_peel(const RowArgs &a, int g, bool cluster, int64_t grid, cudaStream_t st);

}  // namespace osr
