// LayerNorm kernels, storage F32.
#include "launch_layernorm.cuh"

namespace osr {
template cudaError_t launch_layernorm<Dt::F32>(Kind, const RowArgs &, int, bool, int64_t,
                                              cudaStream_t);
template cudaError_t layernorm_cluster_occupancy<Dt::F32>(int, bool, int, int *);
}  // namespace osr
