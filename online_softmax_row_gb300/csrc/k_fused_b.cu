// RMSNorm kernels, storage BF16, fused residual-add: true.
#include "launch_rmsnorm.cuh"

namespace osr {
template cudaError_t launch_rmsnorm<Dt::BF16, true>(Kind, const RowArgs &, int, bool, int64_t,
                                                cudaStream_t);
template cudaError_t rmsnorm_cluster_occupancy<Dt::BF16, true>(int, bool, int, int *);
}  // namespace osr
