// split.cuh -- split-row tier for rows of any length: a row is cut into S
// pieces handled by S independent CTAs.
//   pass 1: each CTA streams its piece and writes one partial state to the
//           workspace ws[row][piece] -- (m, d) for softmax, the sum of
//           squares for the norms (the fused norm also writes the new
//           residual here);
//   pass 2: each CTA merges the S partials of its row in a fixed order (so
//           every piece of a row sees bit-identical statistics and repeated
//           runs are bit-identical), then streams its piece again and writes
//           the output.
// "Softmax 与归一化" (anrans.github.io), table "按行长度选择并行方式" (the
// "very long rows, few rows: several blocks per row, partial (m, d) then
// merge" row) and "第23讲：为什么Attention必须先算Max？" (lilinji.mintlify.site)
// §8.3 thought question 1 (rows beyond 65536).  The host keeps the second read
// in L2 by issuing the two passes over batches of rows whose pieces fit L2.
#pragma once

#include "rows.cuh"

namespace osr {

template <int G>
struct SplitGeom {
    static constexpr int kThreads = G;
    static constexpr int kWarps = G / 32;
};

// CTA (row, piece) of a split launch; rows are a.row0 + blockIdx.x / S.
struct Piece {
    int64_t row;
    int p;
    int64_t u0, u1;
};

__device__ __forceinline__ Piece make_piece(const RowArgs &a, int64_t nunits) {
    Piece q;
    q.row = a.row0 + blockIdx.x / a.cs;
    q.p = blockIdx.x % a.cs;
    q.u0 = (int64_t)q.p * a.chunk;
    q.u1 = q.u0 + a.chunk < nunits ? q.u0 + a.chunk : nunits;
    return q;
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
        float tm = -FLT_MAX;
#pragma unroll
        for (int j = 0; j < NU; ++j)
#pragma unroll
            for (int k = 0; k < U; ++k) tm = fmaxf(tm, v[j][k]);
        float td = 0.f;
#pragma unroll
        for (int j = 0; j < NU; ++j)
#pragma unroll
            for (int k = 0; k < U; ++k) td += exp_shifted(v[j][k], tm);
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

// ------------------------------------------------------------ RMSNorm pass 1
template <Dt D, int G, int EPT, int U, bool FUSED>
__global__ void __launch_bounds__(G) rmsnorm_split_stats_kernel(const RowArgs a) {
    constexpr int NU = EPT / U;
    const int64_t nunits = a.N / U;
    const Piece q = make_piece(a, nunits);
    const int64_t row_off = q.row * a.N * Elem<D>::kBytes;
    const char *xrow = reinterpret_cast<const char *>(a.x) + row_off;
    pdl_wait();
    float ss = 0.f;
    for (int64_t base = q.u0; base < q.u1; base += (int64_t)G * NU) {
        float v[NU][U];
#pragma unroll
        for (int j = 0; j < NU; ++j) {
            const int64_t ui = base + (int64_t)j * G + threadIdx.x;
            if (ui < q.u1) {
                if constexpr (FUSED) {
                    char *rrow = reinterpret_cast<char *>(a.res) + row_off;
                    float r[U];
                    load_unit<D, U>(xrow, ui * U, v[j]);
                    load_unit<D, U>(rrow, ui * U, r);
#pragma unroll
                    for (int k = 0; k < U; ++k) v[j][k] = round_to<D>(v[j][k] + r[k]);
                    store_unit<D, U>(rrow, ui * U, v[j]);
                } else {
                    load_unit<D, U, Hint::Keep>(xrow, ui * U, v[j]);
                }
            } else {
#pragma unroll
                for (int k = 0; k < U; ++k) v[j][k] = 0.f;
            }
        }
#pragma unroll
        for (int j = 0; j < NU; ++j)
#pragma unroll
            for (int k = 0; k < U; ++k) ss = fmaf(v[j][k], v[j][k], ss);
    }
    __shared__ float red[32];
    ss = block_sum<SplitGeom<G>::kWarps>(ss, red);
    if (threadIdx.x == 0) reinterpret_cast<float *>(a.ws)[q.row * a.cs + q.p] = ss;
    pdl_trigger();
}

// ------------------------------------------------------------ RMSNorm pass 2
// Reads x (or, fused, the new residual written by pass 1) again.
template <Dt D, int G, int EPT, int U, bool FUSED>
__global__ void __launch_bounds__(G) rmsnorm_split_apply_kernel(const RowArgs a) {
    constexpr int NU = EPT / U;
    const int64_t nunits = a.N / U;
    const Piece q = make_piece(a, nunits);
    pdl_wait();
    float ss = 0.f;
    if (threadIdx.x < a.cs) ss = reinterpret_cast<const float *>(a.ws)[q.row * a.cs + threadIdx.x];
    __shared__ float red[32];
    ss = block_sum<SplitGeom<G>::kWarps>(ss, red);
    const float r = rsqrtf(ss / (float)a.N + a.eps);
    const int64_t row_off = q.row * a.N * Elem<D>::kBytes;
    const char *src = reinterpret_cast<const char *>(FUSED ? a.res : a.x) + row_off;
    char *yrow = reinterpret_cast<char *>(a.y) + row_off;
    for (int64_t base = q.u0; base < q.u1; base += (int64_t)G * NU) {
        float v[NU][U], g[NU][U];
#pragma unroll
        for (int j = 0; j < NU; ++j) {
            const int64_t ui = base + (int64_t)j * G + threadIdx.x;
            if (ui < q.u1) {
                load_unit<D, U>(src, ui * U, v[j]);
                load_unit<D, U, Hint::ReadOnly>(a.gamma, ui * U, g[j]);
            }
        }
#pragma unroll
        for (int j = 0; j < NU; ++j) {
            const int64_t ui = base + (int64_t)j * G + threadIdx.x;
            if (ui < q.u1) {
                float o[U];
#pragma unroll
                for (int k = 0; k < U; ++k) o[k] = v[j][k] * r * g[j][k];
                store_unit<D, U>(yrow, ui * U, o);
            }
        }
    }
    pdl_trigger();
}

// ------------------------------------------------------------ LayerNorm, split
// Pass 1: each piece's (n, mean, M2) of the pivot-shifted values (the pivot,
// x[row][0], is stored with them, so pass 2 never reads x[row][0] after a
// piece has overwritten it in place): every tile
// is summarised by its own two passes in registers and folded into the
// thread's state with Chan's merge ("GPU Kernel 工程（04）" 八.2, Welford and
// Chan et al.), then the CTA's states are merged in a fixed tree.  Pass 2:
// every CTA of a row merges the row's S states in the same fixed tree (so all
// of them normalise with identical statistics) and streams its piece again.
struct Chan {
    float n, mean, m2;
};

__device__ __forceinline__ Chan chan_merge(Chan a, Chan b) {
    if (a.n == 0.f) return b;
    if (b.n == 0.f) return a;
    const float n = a.n + b.n, delta = b.mean - a.mean, fb = b.n / n;
    return {n, fmaf(delta, fb, a.mean), a.m2 + b.m2 + delta * delta * a.n * fb};
}

// Merge the CTA's per-thread states; the result is valid in thread 0.
template <int NW>
__device__ __forceinline__ Chan block_chan_to_thread0(Chan c, float4 *red) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        Chan o;
        o.n = __shfl_down_sync(0xffffffffu, c.n, off);
        o.mean = __shfl_down_sync(0xffffffffu, c.mean, off);
        o.m2 = __shfl_down_sync(0xffffffffu, c.m2, off);
        if (lane + off < 32) c = chan_merge(c, o);
    }
    if (lane == 0) red[warp] = make_float4(c.n, c.mean, c.m2, 0.f);
    __syncthreads();
    if (warp == 0) {
        c = Chan{0.f, 0.f, 0.f};
        if (lane < NW) {
            const float4 q = red[lane];
            c = Chan{q.x, q.y, q.z};
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            Chan o;
            o.n = __shfl_down_sync(0xffffffffu, c.n, off);
            o.mean = __shfl_down_sync(0xffffffffu, c.mean, off);
            o.m2 = __shfl_down_sync(0xffffffffu, c.m2, off);
            if (lane + off < 32) c = chan_merge(c, o);
        }
    }
    return c;
}

template <Dt D, int G, int EPT, int U>
__global__ void __launch_bounds__(G) layernorm_split_stats_kernel(const RowArgs a) {
    constexpr int NU = EPT / U;
    const int64_t nunits = a.N / U;
    const Piece q = make_piece(a, nunits);
    const char *xrow = reinterpret_cast<const char *>(a.x) + q.row * a.N * Elem<D>::kBytes;
    pdl_wait();
    float p;
    {
        float t[1];
        load_unit<D, 1, Hint::Keep>(xrow, 0, t);
        p = t[0];
    }
    Chan st{0.f, 0.f, 0.f};
    for (int64_t base = q.u0; base < q.u1; base += (int64_t)G * NU) {
        float v[NU][U];
        int cnt = 0;
        float s1 = 0.f;
#pragma unroll
        for (int j = 0; j < NU; ++j) {
            const int64_t ui = base + (int64_t)j * G + threadIdx.x;
            if (ui < q.u1) {
                load_unit<D, U, Hint::Keep>(xrow, ui * U, v[j]);
#pragma unroll
                for (int k = 0; k < U; ++k) {
                    v[j][k] -= p;
                    s1 += v[j][k];
                }
                cnt += U;
            }
        }
        if (cnt == 0) continue;
        const float tm = s1 / (float)cnt;
        float s2 = 0.f;
#pragma unroll
        for (int j = 0; j < NU; ++j) {
            const int64_t ui = base + (int64_t)j * G + threadIdx.x;
            if (ui < q.u1) {
#pragma unroll
                for (int k = 0; k < U; ++k) {
                    const float c = v[j][k] - tm;
                    s2 = fmaf(c, c, s2);
                }
            }
        }
        st = chan_merge(st, Chan{(float)cnt, tm, s2});
    }
    __shared__ float4 red[32];
    st = block_chan_to_thread0<G / 32>(st, red);
    if (threadIdx.x == 0)
        reinterpret_cast<float4 *>(a.ws)[q.row * a.cs + q.p] = make_float4(st.n, st.mean, st.m2, p);
    pdl_trigger();
}

template <Dt D, int G, int EPT, int U>
__global__ void __launch_bounds__(G) layernorm_split_apply_kernel(const RowArgs a) {
    constexpr int NU = EPT / U;
    const int64_t nunits = a.N / U;
    const Piece q = make_piece(a, nunits);
    const int64_t row_off = q.row * a.N * Elem<D>::kBytes;
    const char *xrow = reinterpret_cast<const char *>(a.x) + row_off;
    pdl_wait();
    Chan st{0.f, 0.f, 0.f};
    if (threadIdx.x < a.cs) {
        const float4 w = reinterpret_cast<const float4 *>(a.ws)[q.row * a.cs + threadIdx.x];
        st = Chan{w.x, w.y, w.z};
    }
    __shared__ float4 red[32];
    __shared__ float2 stats;
    st = block_chan_to_thread0<G / 32>(st, red);
    if (threadIdx.x == 0) stats = make_float2(st.mean, rsqrtf(st.m2 / (float)a.N + a.eps));
    const float p = reinterpret_cast<const float4 *>(a.ws)[q.row * a.cs].w;  // pass 1's pivot
    __syncthreads();
    const float mu = stats.x, r = stats.y;
    char *yrow = reinterpret_cast<char *>(a.y) + row_off;
    for (int64_t base = q.u0; base < q.u1; base += (int64_t)G * NU) {
        float v[NU][U], g[NU][U], b[NU][U];
#pragma unroll
        for (int j = 0; j < NU; ++j) {
            const int64_t ui = base + (int64_t)j * G + threadIdx.x;
            if (ui < q.u1) {
                load_unit<D, U>(xrow, ui * U, v[j]);
                load_unit<D, U, Hint::ReadOnly>(a.gamma, ui * U, g[j]);
                load_unit<D, U, Hint::ReadOnly>(a.beta, ui * U, b[j]);
            }
        }
#pragma unroll
        for (int j = 0; j < NU; ++j) {
            const int64_t ui = base + (int64_t)j * G + threadIdx.x;
            if (ui < q.u1) {
                float o[U];
#pragma unroll
                for (int k = 0; k < U; ++k) o[k] = fmaf(((v[j][k] - p) - mu) * r, g[j][k], b[j][k]);
                store_unit<D, U>(yrow, ui * U, o);
            }
        }
    }
    pdl_trigger();
}

}  // namespace osr
