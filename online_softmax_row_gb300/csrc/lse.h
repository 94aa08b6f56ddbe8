// lse.h -- what the log-sum-exp planner needs to know of the kernels in
// k_lse.cu, apart from launch.h.
#pragma once

#include "device_common.cuh"

namespace osr {

// CTAs an SM the streaming cluster kernel is compiled to hold (its launch
// bound: registers are capped to fit), which the planner counts on
constexpr int lse_cluster_ctas_per_sm(Dt d) { return d == Dt::BF16 ? 5 : 4; }

}  // namespace osr
