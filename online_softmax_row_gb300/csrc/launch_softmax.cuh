// launch_softmax.cuh -- definitions of launch_softmax and softmax_cluster_occupancy
// (declared in launch.h).
#pragma once

#include "launch_common.cuh"
#include "softmax_kernels.cuh"

namespace osr {

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

}  // namespace osr
