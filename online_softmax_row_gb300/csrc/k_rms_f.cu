// RMSNorm kernels, storage F32, fused residual-add: false.
#include "launch_rmsnorm.cuh"

namespace osr {
template cudaError_t launch_rmsnorm<Dt::F32, false>(Kind, const RowArgs &, int, bool, int64_t,
                                                cudaStream_t);
template cudaError_t rmsnorm_cluster_occupancy<Dt::F32, false>(int, bool, int, int *);
}  // namespace osr
