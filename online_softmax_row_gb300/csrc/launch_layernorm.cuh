// launch_layernorm.cuh -- definitions of launch_layernorm and
// layernorm_cluster_occupancy (declared in launch.h).
#pragma once

#include "launch_common.cuh"
#include "layernorm_kernels.cuh"

namespace osr {

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
