// launch_impl.cuh -- definitions of the launch templates declared in
// launch.h.  Each k_*.cu translation unit includes this file and explicitly
// instantiates one dtype combination, so the kernels compile in parallel.
#pragma once

#include "launch.h"
#include "split.cuh"

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

template <Dt DI, Dt DO, int U>
cudaError_t launch_softmax_u(Kind k, const RowArgs &a, int g, int64_t grid, cudaStream_t st) {
    KernelFn fn = nullptr;
    int threads = g;
    switch (k) {
    case Kind::Rows:
#define OSR_MAKE(G) \
    if (g == G) { fn = softmax_rows_kernel<DI, DO, G, softmax_ept<DI, U>(), U, false>; threads = RowsGeom<G>::kThreads; }
        OSR_ROWS_G_CASES(OSR_MAKE)
#undef OSR_MAKE
        return fn ? launch_plain(fn, grid, threads, a, st) : cudaErrorInvalidConfiguration;
    case Kind::Cluster:
#define OSR_MAKE(G) \
    if (g == G) fn = softmax_rows_kernel<DI, DO, G, softmax_ept<DI, U>(), U, true>;
        OSR_CLUSTER_G_CASES(OSR_MAKE)
#undef OSR_MAKE
        return fn ? launch_clustered(fn, grid, g, a.cs, a, st) : cudaErrorInvalidConfiguration;
    case Kind::SplitStats:
        return launch_plain(softmax_split_stats_kernel<DI, kSplitThreads, kEpt, U>, grid,
                            kSplitThreads, a, st);
    case Kind::SplitApply:
        return launch_plain(softmax_split_apply_kernel<DI, DO, kSplitThreads, kEpt, U>, grid,
                            kSplitThreads, a, st);
    }
    return cudaErrorInvalidConfiguration;
}

template <Dt DI, Dt DO>
cudaError_t launch_softmax(Kind k, const RowArgs &a, int g, bool vec, int64_t grid,
                           cudaStream_t st) {
    if (vec) return launch_softmax_u<DI, DO, Elem<DI>::kVec>(k, a, g, grid, st);
    return launch_softmax_u<DI, DO, 1>(k, a, g, grid, st);
}

template <Dt DI, Dt DO, int U>
cudaError_t softmax_cluster_occupancy_u(int g, int cs, int *n) {
    KernelFn fn = nullptr;
#define OSR_MAKE(G) \
    if (g == G) fn = softmax_rows_kernel<DI, DO, G, softmax_ept<DI, U>(), U, true>;
    OSR_CLUSTER_G_CASES(OSR_MAKE)
#undef OSR_MAKE
    return fn ? cluster_occupancy(fn, g, cs, n) : cudaErrorInvalidConfiguration;
}

template <Dt DI, Dt DO>
cudaError_t softmax_cluster_occupancy(int g, bool vec, int cs, int *n) {
    if (vec) return softmax_cluster_occupancy_u<DI, DO, Elem<DI>::kVec>(g, cs, n);
    return softmax_cluster_occupancy_u<DI, DO, 1>(g, cs, n);
}

template <Dt D, bool FUSED, int U>
cudaError_t launch_rmsnorm_u(Kind k, const RowArgs &a, int g, int64_t grid, cudaStream_t st) {
    KernelFn fn = nullptr;
    int threads = g;
    switch (k) {
    case Kind::Rows:
#define OSR_MAKE(G) \
    if (g == G) { fn = rmsnorm_rows_kernel<D, G, norm_ept<D, U, FUSED>(), U, false, FUSED>; threads = RowsGeom<G>::kThreads; }
        OSR_ROWS_G_CASES(OSR_MAKE)
#undef OSR_MAKE
        return fn ? launch_plain(fn, grid, threads, a, st) : cudaErrorInvalidConfiguration;
    case Kind::Cluster:
#define OSR_MAKE(G) \
    if (g == G) fn = rmsnorm_rows_kernel<D, G, norm_ept<D, U, FUSED>(), U, true, FUSED>;
        OSR_CLUSTER_G_CASES(OSR_MAKE)
#undef OSR_MAKE
        return fn ? launch_clustered(fn, grid, g, a.cs, a, st) : cudaErrorInvalidConfiguration;
    case Kind::SplitStats:
        return launch_plain(rmsnorm_split_stats_kernel<D, kSplitThreads, norm_ept<D, U, FUSED>(), U, FUSED>, grid,
                            kSplitThreads, a, st);
    case Kind::SplitApply:
        return launch_plain(rmsnorm_split_apply_kernel<D, kSplitThreads, norm_ept<D, U, FUSED>(), U, FUSED>, grid,
                            kSplitThreads, a, st);
    }
    return cudaErrorInvalidConfiguration;
}

template <Dt D, bool FUSED>
cudaError_t launch_rmsnorm(Kind k, const RowArgs &a, int g, bool vec, int64_t grid,
                           cudaStream_t st) {
    if (vec) return launch_rmsnorm_u<D, FUSED, Elem<D>::kVec>(k, a, g, grid, st);
    return launch_rmsnorm_u<D, FUSED, 1>(k, a, g, grid, st);
}

template <Dt D, bool FUSED, int U>
cudaError_t rmsnorm_cluster_occupancy_u(int g, int cs, int *n) {
    KernelFn fn = nullptr;
#define OSR_MAKE(G) \
    if (g == G) fn = rmsnorm_rows_kernel<D, G, norm_ept<D, U, FUSED>(), U, true, FUSED>;
    OSR_CLUSTER_G_CASES(OSR_MAKE)
#undef OSR_MAKE
    return fn ? cluster_occupancy(fn, g, cs, n) : cudaErrorInvalidConfiguration;
}

template <Dt D, bool FUSED>
cudaError_t rmsnorm_cluster_occupancy(int g, bool vec, int cs, int *n) {
    if (vec) return rmsnorm_cluster_occupancy_u<D, FUSED, Elem<D>::kVec>(g, cs, n);
    return rmsnorm_cluster_occupancy_u<D, FUSED, 1>(g, cs, n);
}

template <Dt D, int U>
cudaError_t launch_layernorm_u(Kind k, const RowArgs &a, int g, int64_t grid, cudaStream_t st) {
    KernelFn fn = nullptr;
    int threads = g;
    switch (k) {
    case Kind::Rows:
#define OSR_MAKE(G) \
    if (g == G) { fn = layernorm_rows_kernel<D, G, norm_ept<D, U>(), U, false>; threads = RowsGeom<G>::kThreads; }
        OSR_ROWS_G_CASES(OSR_MAKE)
#undef OSR_MAKE
        return fn ? launch_plain(fn, grid, threads, a, st) : cudaErrorInvalidConfiguration;
    case Kind::Cluster:
#define OSR_MAKE(G) \
    if (g == G) fn = layernorm_rows_kernel<D, G, norm_ept<D, U>(), U, true>;
        OSR_CLUSTER_G_CASES(OSR_MAKE)
#undef OSR_MAKE
        return fn ? launch_clustered(fn, grid, g, a.cs, a, st) : cudaErrorInvalidConfiguration;
    case Kind::SplitStats:
        return launch_plain(layernorm_split_stats_kernel<D, kSplitThreads, norm_ept<D, U>(), U>, grid,
                            kSplitThreads, a, st);
    case Kind::SplitApply:
        return launch_plain(layernorm_split_apply_kernel<D, kSplitThreads, norm_ept<D, U>(), U>, grid,
                            kSplitThreads, a, st);
    }
    return cudaErrorInvalidConfiguration;
}

template <Dt D>
cudaError_t launch_layernorm(Kind k, const RowArgs &a, int g, bool vec, int64_t grid,
                             cudaStream_t st) {
    if (vec) return launch_layernorm_u<D, Elem<D>::kVec>(k, a, g, grid, st);
    return launch_layernorm_u<D, 1>(k, a, g, grid, st);
}

template <Dt D, int U>
cudaError_t layernorm_cluster_occupancy_u(int g, int cs, int *n) {
    KernelFn fn = nullptr;
#define OSR_MAKE(G) \
    if (g == G) fn = layernorm_rows_kernel<D, G, norm_ept<D, U>(), U, true>;
    OSR_CLUSTER_G_CASES(OSR_MAKE)
#undef OSR_MAKE
    return fn ? cluster_occupancy(fn, g, cs, n) : cudaErrorInvalidConfiguration;
}

template <Dt D>
cudaError_t layernorm_cluster_occupancy(int g, bool vec, int cs, int *n) {
    if (vec) return layernorm_cluster_occupancy_u<D, Elem<D>::kVec>(g, cs, n);
    return layernorm_cluster_occupancy_u<D, 1>(g, cs, n);
}

}  // namespace osr
