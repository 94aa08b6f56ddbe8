// launch_common.cuh -- launch helpers shared by the per-operation launch
// headers (launch_softmax.cuh, launch_rmsnorm.cuh, launch_layernorm.cuh).
// Each k_*.cu translation unit includes one of those and explicitly
// instantiates one dtype combination, so the kernels compile in parallel and
// a translation unit holds only its own operation's kernels.
#pragma once

#include "launch.h"

namespace osr {

using KernelFn = void (*)(RowArgs);

inline cudaError_t launch_plain(KernelFn k, int64_t grid, int threads, const RowArgs &a,
                                cudaStream_t st) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(threads);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = use_pdl() ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, k, a);
}

inline cudaError_t launch_clustered(KernelFn k, int64_t grid, int threads, int cs,
                                    const RowArgs &a, cudaStream_t st) {
    if (cs > 8) {
        cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (e != cudaSuccess) return e;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)cs;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = use_pdl() ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, k, a);
}

// How many clusters of `cs` CTAs of kernel k can be resident at once
// (0: the cluster shape cannot be scheduled on this device).
inline cudaError_t cluster_occupancy(KernelFn k, int threads, int cs, int *n) {
    *n = 0;
    if (cs > 8) {
        cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (e != cudaSuccess) return e;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)cs * 64u);
    cfg.blockDim = dim3(threads);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)cs;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaOccupancyMaxActiveClusters(n, k, &cfg);
}

#define OSR_ROWS_G_CASES(MAKE) \
    MAKE(1) MAKE(2) MAKE(4) MAKE(8) MAKE(16) MAKE(32) MAKE(64) MAKE(128) MAKE(256) MAKE(512) MAKE(1024)
#define OSR_CLUSTER_G_CASES(MAKE) MAKE(256) MAKE(1024)

}  // namespace osr
