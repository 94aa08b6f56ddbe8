// RMSNorm kernels, storage BF16, fused residual-add: false.
#include "launch_rmsnorm.cuh"

namespace osr {
template cudaError_t launch_rmsnorm<Dt::BF16, false>(Kind, const RowArgs &, int, bool, int64_t,
                                                cudaStream_t);
template cudaError_t rmsnorm_cluster_occupancy<Dt::BF16, false>(int, bool, int, int *);
}  // namespace osr
