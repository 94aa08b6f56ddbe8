// launch_rmsnorm.cuh -- definitions of launch_rmsnorm and rmsnorm_cluster_occupancy
// (declared in launch.h).
#pragma once

#include "launch_common.cuh"
#include "rmsnorm_kernels.cuh"

namespace osr {

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

}  // namespace osr
