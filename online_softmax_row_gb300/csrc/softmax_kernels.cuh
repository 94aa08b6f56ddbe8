// softmax_kernels.cuh -- softmax (and log-softmax) kernels: the register-cached
// row/cluster kernel and the two split-row passes.
#pragma once

#include "row_common.cuh"

namespace osr {

// ============================================================ softmax
// Per thread: chunk summary of its cached elements (max, then sum of
// exp(x - max), overwriting the cache with those exps) -- the chunk-summary
// form of "两个融合算子" §4·四 "S4" with the chunk = the thread's elements.
// The row's (m, d) follows by max-then-sum over the row's threads (and CTAs);
// each thread then rescales its cached exps by e^(m_t - m) / d, so every
// element costs one exp.
template <Dt DI, Dt DO, int G, int EPT, int U, bool CLUSTER>
__global__ void __launch_bounds__(RowsGeom<G>::kThreads)
softmax_rows_kernel(const RowArgs a) {
    constexpr int NU = EPT / U;
    const int64_t nunits = a.N / U;
    const Slice s = make_slice<G, CLUSTER>(a, nunits);
    const char *xrow = reinterpret_cast<const char *>(a.x) + s.row * a.N * Elem<DI>::kBytes;
    if constexpr (CLUSTER) cluster_push_init(cluster_push_area<0>(), nullptr, a.cs);
    pdl_wait();

    float v[NU][U];
#pragma unroll
    for (int j = 0; j < NU; ++j) {
        const int64_t ui = s.u0 + (int64_t)j * G + s.t;
        if (s.ok && ui < s.u1) {
            load_unit<DI, U>(xrow, ui * U, v[j]);
        } else {
#pragma unroll
            for (int k = 0; k < U; ++k) v[j][k] = -INFINITY;  // contributes e^-inf = 0
        }
    }

    float mt = -INFINITY;
#pragma unroll
    for (int j = 0; j < NU; ++j)
#pragma unroll
        for (int k = 0; k < U; ++k) mt = fmaxf(mt, v[j][k]);
    // log-softmax keeps the inputs; softmax replaces them by their exps
    const bool logm = (a.flags & kFlagLog) != 0;
    const float ms = md_shift(mt);
    float dt = 0.f;
#pragma unroll
    for (int j = 0; j < NU; ++j)
#pragma unroll
        for (int k = 0; k < U; ++k) {
            const float e = exp_shifted(v[j][k], ms);
            dt += e;
            v[j][k] = logm ? v[j][k] : e;
        }

    RowNorm rn;
    if constexpr (G <= 32) {
        rn = group_norm<G>(mt, dt);
    } else {
        __shared__ float red_m[32], red_d[32];
        rn = block_norm<RowsGeom<G>::kWarps>(mt, dt, red_m, red_d);
    }
    if constexpr (CLUSTER) rn = cluster_norm(mt, rn, a.cs, cluster_push_area<0>(), true);

    const float scale = rn.f / rn.d;
    const float logd = logf(rn.d);
    if (a.row_max != nullptr && s.ok && s.t == 0 && s.u0 == 0) {
        a.row_max[s.row] = rn.m;
        if (a.row_sum != nullptr) a.row_sum[s.row] = rn.d;
    }

    char *yrow = reinterpret_cast<char *>(a.y) + s.row * a.N * Elem<DO>::kBytes;
#pragma unroll
    for (int j = 0; j < NU; ++j) {
        const int64_t ui = s.u0 + (int64_t)j * G + s.t;
        if (s.ok && ui < s.u1) {
            float o[U];
#pragma unroll
            for (int k = 0; k < U; ++k) o[k] = logm ? (v[j][k] - rn.m) - logd : v[j][k] * scale;
            store_unit<DO, U>(yrow, ui * U, o);
        }
    }
    pdl_trigger();
}

// ------------------------------------------------------------ softmax pass 1
// Each tile of the piece is summarised (max, then sum of exp(x - max)) and
// merged into the thread's running (m, d), the chunk-summary update of
// "两个融合算子：RMSNorm 与 online softmax" §4·四 "S4".
template <Dt DI, int G, int EPT, int U>
__global__ void __launch_bounds__(G) softmax_split_stats_kernel(const RowArgs a) {
    constexpr int NU = EPT / U;
    const int64_t nunits = a.N / U;
    const Piece q = make_piece(a, nunits);
    const char *xrow = reinterpret_cast<const char *>(a.x) + q.row * a.N * Elem<DI>::kBytes;
    pdl_wait();
    MD st = md_identity();
    for (int64_t base = q.u0; base < q.u1; base += (int64_t)G * NU) {
        float v[NU][U];
#pragma unroll
        for (int j = 0; j < NU; ++j) {
            const int64_t ui = base + (int64_t)j * G + threadIdx.x;
            if (ui < q.u1) {
                load_unit<DI, U, Hint::Keep>(xrow, ui * U, v[j]);
            } else {
#pragma unroll
                for (int k = 0; k < U; ++k) v[j][k] = -INFINITY;
            }
        }
        float tm = -INFINITY;
#pragma unroll
        for (int j = 0; j < NU; ++j)
#pragma unroll
            for (int k = 0; k < U; ++k) tm = fmaxf(tm, v[j][k]);
        const float ts = md_shift(tm);
        float td = 0.f;
#pragma unroll
        for (int j = 0; j < NU; ++j)
#pragma unroll
            for (int k = 0; k < U; ++k) td += exp_shifted(v[j][k], ts);
        st = md_merge(st, MD{tm, td});
    }
    __shared__ float red_m[32], red_d[32];
    const RowNorm rn = block_norm<SplitGeom<G>::kWarps>(st.m, st.d, red_m, red_d);
    if (threadIdx.x == 0)
        reinterpret_cast<float2 *>(a.ws)[q.row * a.cs + q.p] = make_float2(rn.m, rn.d);
    pdl_trigger();
}

// ------------------------------------------------------------ softmax pass 2
template <Dt DI, Dt DO, int G, int EPT, int U>
__global__ void __launch_bounds__(G) softmax_split_apply_kernel(const RowArgs a) {
    constexpr int NU = EPT / U;
    const int64_t nunits = a.N / U;
    const Piece q = make_piece(a, nunits);
    pdl_wait();
    // merge the row's S partials: thread i holds partial i (S <= G), the
    // rest the identity; max-then-sum in a fixed tree
    MD st = md_identity();
    if (threadIdx.x < a.cs) {
        const float2 w = reinterpret_cast<const float2 *>(a.ws)[q.row * a.cs + threadIdx.x];
        st = MD{w.x, w.y};
    }
    __shared__ float red_m[32], red_d[32];
    const RowNorm rn = block_norm<SplitGeom<G>::kWarps>(st.m, st.d, red_m, red_d);
    st = MD{rn.m, rn.d};
    if (a.row_max != nullptr && q.p == 0 && threadIdx.x == 0) {
        a.row_max[q.row] = st.m;
        if (a.row_sum != nullptr) a.row_sum[q.row] = st.d;
    }
    const float inv_d = 1.0f / st.d, logd = logf(st.d);
    const bool logm = (a.flags & kFlagLog) != 0;
    const char *xrow = reinterpret_cast<const char *>(a.x) + q.row * a.N * Elem<DI>::kBytes;
    char *yrow = reinterpret_cast<char *>(a.y) + q.row * a.N * Elem<DO>::kBytes;
    for (int64_t base = q.u0; base < q.u1; base += (int64_t)G * NU) {
        float v[NU][U];
#pragma unroll
        for (int j = 0; j < NU; ++j) {
            const int64_t ui = base + (int64_t)j * G + threadIdx.x;
            if (ui < q.u1) load_unit<DI, U>(xrow, ui * U, v[j]);
        }
#pragma unroll
        for (int j = 0; j < NU; ++j) {
            const int64_t ui = base + (int64_t)j * G + threadIdx.x;
            if (ui < q.u1) {
                float o[U];
#pragma unroll
                for (int k = 0; k < U; ++k)
                    o[k] = logm ? (v[j][k] - st.m) - logd : exp_shifted(v[j][k], st.m) * inv_d;
                store_unit<DO, U>(yrow, ui * U, o);
            }
        }
    }
    pdl_trigger();
}

}  // namespace osr
