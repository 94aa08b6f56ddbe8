// Softmax kernels, input F32 / output F32.
#include "launch_softmax.cuh"

namespace osr {
template cudaError_t launch_softmax<Dt::F32, Dt::F32>(Kind, const RowArgs &, int, bool, int64_t,
                                                    cudaStream_t);
template cudaError_t softmax_cluster_occupancy<Dt::F32, Dt::F32>(int, bool, int, int *);
}  // namespace osr
