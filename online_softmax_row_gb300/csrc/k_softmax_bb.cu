// Softmax kernels, input BF16 / output BF16.
#include "launch_softmax.cuh"

namespace osr {
template cudaError_t launch_softmax<Dt::BF16, Dt::BF16>(Kind, const RowArgs &, int, bool, int64_t,
                                                    cudaStream_t);
template cudaError_t softmax_cluster_occupancy<Dt::BF16, Dt::BF16>(int, bool, int, int *);
}  // namespace osr
