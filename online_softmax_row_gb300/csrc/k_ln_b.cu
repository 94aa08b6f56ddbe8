// LayerNorm kernels, storage BF16.
#include "launch_layernorm.cuh"

namespace osr {
template cudaError_t launch_layernorm<Dt::BF16>(Kind, const RowArgs &, int, bool, int64_t,
                                              cudaStream_t);
template cudaError_t layernorm_cluster_occupancy<Dt::BF16>(int, bool, int, int *);
}  // namespace osr
